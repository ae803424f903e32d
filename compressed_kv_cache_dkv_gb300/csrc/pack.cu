// Pack plain row-major factors into the packed cache layout (dkv_import_factors).
// One CTA per (block, unit); the extra CTA per unit (blockIdx.x == NB) packs the
// recency window.  Setup path, not timed: simple element-wise stores.
#include "dkv_internal.cuh"

namespace dkv {

namespace {

__device__ inline __half ld_h(const void* base, size_t idx) { return static_cast<const __half*>(base)[idx]; }

__global__ void __launch_bounds__(256) pack_kernel(Layout L, dkv_factors f, uint8_t* cache, uint32_t* err) {
  const int u = blockIdx.y;
  const int b = blockIdx.x;
  const int d = L.d, r = L.r, r8 = L.r8, R = L.R, R8 = L.R8;
  uint8_t* unit = cache + (uint64_t)u * L.unit_stride;
  const int tid = threadIdx.x, nt = blockDim.x;
  const __half zero = __float2half(0.f);

  if (b == L.NB) {  // window
    uint8_t* win = unit + L.off_window;
    for (int e = tid; e < L.W16 * d; e += nt) {
      int t = e / d, j = e % d;
      __half kv = zero, vv = zero;
      if (t < L.W) {
        size_t idx = ((size_t)u * L.W + t) * d + j;
        kv = ld_h(f.win_K, idx);
        vv = ld_h(f.win_V, idx);
      }
      *reinterpret_cast<__half*>(win + win_k_off(L, t, j)) = kv;
      *reinterpret_cast<__half*>(win + win_v_off(L, t, j)) = vv;
    }
    return;
  }

  const size_t base = (size_t)u * L.NB + b;
  uint8_t* blk = unit + L.off_blocks + (uint64_t)b * L.block_stride;
  uint8_t* router = unit + L.off_router + (uint64_t)b * router_row_bytes(L);
  for (int j = tid; j < d; j += nt) {
    reinterpret_cast<__half*>(blk)[j] = ld_h(f.a_k, base * d + j);
    reinterpret_cast<__half*>(blk)[d + j] = ld_h(f.a_v, base * d + j);
    if (L.rope) {  // un-rotated pool: fp32 box of the rotated keys
      reinterpret_cast<float*>(router)[j] = static_cast<const float*>(f.kmin)[base * d + j];
      reinterpret_cast<float*>(router)[d + j] = static_cast<const float*>(f.kmax)[base * d + j];
    } else {
      reinterpret_cast<__half*>(router)[j] = ld_h(f.kmin, base * d + j);
      reinterpret_cast<__half*>(router)[d + j] = ld_h(f.kmax, base * d + j);
    }
  }
  // residual mask + cold positions; positions must be strictly ascending in 1..255
  __shared__ uint32_t mask[8];
  __shared__ int bad;
  if (tid < 8) mask[tid] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int i = tid; i < R; i += nt) {
    int p = f.res_pos[base * R + i];
    int prev = i ? f.res_pos[base * R + i - 1] : 0;
    if (p < 1 || p > 255 || p <= prev) bad = 1;
  }
  __syncthreads();
  if (!bad) {
    for (int i = tid; i < R; i += nt) {
      int p = f.res_pos[base * R + i];
      atomicOr(&mask[p >> 5], 1u << (p & 31));
    }
  } else if (tid == 0) {
    raise_error(err, DKV_DEVERR_INDEX);
  }
  __syncthreads();
  if (tid < 8) reinterpret_cast<uint32_t*>(blk + L.off_mask)[tid] = mask[tid];
  uint16_t* cold = reinterpret_cast<uint16_t*>(unit + L.off_cold) + (size_t)b * R8;
  for (int i = tid; i < R8; i += nt) cold[i] = (i < R && !bad) ? (uint16_t)f.res_pos[base * R + i] : 0;
  // V_K [r8][d] in B^T layout
  for (int e = tid; e < r8 * d; e += nt) {
    int k = e / d, j = e % d;
    __half v = k < r ? ld_h(f.V_K, (base * r + k) * d + j) : zero;
    *reinterpret_cast<__half*>(blk + L.off_vk + bt_layout_off(r8, d, k, j)) = v;
  }
  // U [256][r8], row 0 (the anchor) all zero
  for (int e = tid; e < 256 * r8; e += nt) {
    int t = e / r8, k = e % r8;
    __half v = (t >= 1 && k < r) ? ld_h(f.U, (base * 255 + (t - 1)) * r + k) : zero;
    *reinterpret_cast<__half*>(blk + blk_u_off(L, t, k)) = v;
  }
  // residual K and V (group-quantised when the layout asks for it; every thread takes part)
  if (L.qbits) {
    write_quant_residuals(
        L, blk + L.off_res, R, [&](int i, int j) { return ld_h(f.K_res, (base * R + i) * d + j); },
        [&](int i, int j) { return ld_h(f.V_res, (base * R + i) * d + j); });
  } else {
    for (int e = tid; e < R8 * d; e += nt) {
      int i = e / d, j = e % d;
      __half kv = zero, vv = zero;
      if (i < R) {
        kv = ld_h(f.K_res, (base * R + i) * d + j);
        vv = ld_h(f.V_res, (base * R + i) * d + j);
      }
      *reinterpret_cast<__half*>(blk + blk_resk_off(L, i, j)) = kv;
      *reinterpret_cast<__half*>(blk + blk_resv_off(L, i, j)) = vv;
    }
  }
  // V_V [r8][d]
  for (int e = tid; e < r8 * d; e += nt) {
    int k = e / d, j = e % d;
    __half v = k < r ? ld_h(f.V_V, (base * r + k) * d + j) : zero;
    *reinterpret_cast<__half*>(blk + blk_vv_off(L, k, j)) = v;
  }
}

}  // namespace

cudaError_t launch_pack(const Layout& L, const dkv_factors& f, uint8_t* cache, uint32_t* err, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(cache, 0, L.total, s);
  if (e != cudaSuccess) return e;
  e = launch_rope_tables(L, cache, s);
  if (e != cudaSuccess) return e;
  dim3 grid(L.NB + 1, L.units);
  pack_kernel<<<grid, 256, 0, s>>>(L, f, cache, err);
  return cudaGetLastError();
}

}  // namespace dkv
