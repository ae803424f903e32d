// Block router and split-LSE combine of the DKV decode path.
//
// route: per unit, the group-mean query qbar = (1/G) sum_g c q_g
// (DKV_CB_GQA_ROUTE head averaging, Differential-KV README section "Key
// Environment Knobs") scores every block by the upper bound of qbar . k over
// the block's key box, sum_j max(qbar_j kmax_bj, qbar_j kmin_bj) (the per-block
// "Key Min/Max ... Decode router bounds" of the README's per-block memory
// table), and keeps the top K (DKV_TOPK_BLOCKS) by (score desc, index asc);
// indices are written in ascending order.
//
// combine: the flash-style log-sum-exp merge of every partial of a unit
// ("Flash-Style LSE Combine", README section "Core Architecture & Paper
// Overview"): m* = max m_j, l* = sum l_j 2^(m_j - m*),
// o = sum acc_j 2^(m_j - m*) / l*, all in fp32, in a fixed order (deterministic).
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kRouteBlocks = 64;  // blocks scored per route CTA (8 warps x 8 blocks)

// Scores the blocks [64*blockIdx.x, +64) of unit blockIdx.y into the workspace;
// the last CTA of the unit to finish (arrival counter, no waiting) ranks all of
// the unit's scores and writes the routed indices.
__global__ void __launch_bounds__(256) route_kernel(Layout L, int G, int Hq, int Hkv, int K_eff, float cq,
                                                    const __half* __restrict__ q, const uint8_t* __restrict__ cache,
                                                    float* __restrict__ bounds, uint32_t* __restrict__ counters,
                                                    int32_t* __restrict__ routed, int32_t* __restrict__ routed_out) {
  extern __shared__ float sm[];  // last CTA: scores [NB], selection flags [NB]
  __shared__ float qbar[128];
  __shared__ int s_last;
  const int d = L.d, NB = L.NB;
  const int u = blockIdx.y, split = blockIdx.x, nsplit = gridDim.x;
  const int b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  griddep_launch();  // the attention grid may start its window work now; its block work waits for this grid
  for (int j = tid; j < d; j += nt) {
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += __half2float(q[((size_t)b * Hq + (size_t)h * G + g) * d + j]);
    qbar[j] = s * cq;  // cq = c / G
  }
  __syncthreads();
  // A block's router record is [kmin | kmax], 4d bytes = d/4 pieces of 16 bytes.
  // The warp's 8 blocks are contiguous: 2d pieces, 2d/32 per lane, all loaded first.
  const uint8_t* router = cache + (uint64_t)u * L.unit_stride + L.off_router;
  const int blk0 = split * kRouteBlocks + warp * 8;
  const int per_blk = d / 4;                  // pieces per block (32 or 16)
  const int npl = (2 * d) / 32;               // pieces per lane (8 or 4)
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (i < npl) {
      const int piece = i * 32 + lane;
      const int blk = blk0 + piece / per_blk;
      if (blk < NB) v[i] = *reinterpret_cast<const uint4*>(router + (size_t)blk0 * 4 * d + (size_t)piece * 16);
    }
  }
  const int half_pcs = d / 8;                 // kmin pieces per block; kmax partner at +d/8
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i >= npl) break;
    const int piece = i * 32 + lane;
    const int q_in = piece % per_blk;
    uint4 partner;
    partner.x = __shfl_xor_sync(0xffffffffu, v[i].x, half_pcs);
    partner.y = __shfl_xor_sync(0xffffffffu, v[i].y, half_pcs);
    partner.z = __shfl_xor_sync(0xffffffffu, v[i].z, half_pcs);
    partner.w = __shfl_xor_sync(0xffffffffu, v[i].w, half_pcs);
    float acc = 0.f;
    if (q_in < half_pcs) {
      const __half* kmn = reinterpret_cast<const __half*>(&v[i]);
      const __half* kmx = reinterpret_cast<const __half*>(&partner);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float qj = qbar[8 * q_in + e];
        acc += fmaxf(qj * __half2float(kmx[e]), qj * __half2float(kmn[e]));
      }
    }
    // sum over the per_blk lanes of this block (kmax lanes hold 0)
    for (int o = per_blk >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int blk = blk0 + piece / per_blk;
    if (q_in == 0 && blk < NB && blk < (split + 1) * kRouteBlocks)
      bounds[(size_t)u * NB + blk] = isnan(acc) ? -INFINITY : acc;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&counters[u], 1u) == (unsigned)(nsplit - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* sc = sm;
  int* sel = reinterpret_cast<int*>(sm + NB);
  for (int i = tid; i < NB; i += nt) sc[i] = __ldcg(bounds + (size_t)u * NB + i);
  __syncthreads();
  for (int i = tid; i < NB; i += nt) {
    int s = 1;
    if (K_eff < NB) {
      const float bi = sc[i];
      int rank = 0;
      for (int j = 0; j < NB; ++j) {
        const float bj = sc[j];
        rank += (bj > bi) || (bj == bi && j < i);
      }
      s = rank < K_eff;
    }
    sel[i] = s;
  }
  __syncthreads();
  for (int i = tid; i < NB; i += nt) {
    if (!sel[i]) continue;
    int pos = 0;
    for (int j = 0; j < i; ++j) pos += sel[j];
    if (pos < K_eff) {
      routed[(size_t)u * K_eff + pos] = i;
      if (routed_out) routed_out[(size_t)u * K_eff + pos] = i;
    }
  }
  if (tid == 0) counters[u] = 0u;  // ready for the next call on this workspace
}

// One CTA per unit: its G queries.  Launched as a programmatic dependent of the
// attention grid, so its launch overlaps that grid's tail; griddepcontrol.wait
// makes the partials visible before they are read.
__global__ void __launch_bounds__(256) combine_kernel(int n_items, int G, int Hq, int Hkv, int d,
                                                      const float* __restrict__ partials, float* __restrict__ out,
                                                      float* __restrict__ lse) {
  griddep_wait();
  __shared__ float mstar[8], linv[8];
  const int u = blockIdx.x, b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x;
  const size_t rs = 16 + 8 * (size_t)d;
  const float* p = partials + (size_t)u * n_items * rs;
  const size_t qrow0 = (size_t)b * Hq + (size_t)h * G;
  if (tid < G) {
    float m = -INFINITY;
    for (int i = 0; i < n_items; ++i) m = fmaxf(m, __ldg(p + i * rs + tid));
    const float ms = m == -INFINITY ? 0.f : m;
    float l = 0.f;
    for (int i = 0; i < n_items; ++i) l += __ldg(p + i * rs + 8 + tid) * fast_exp2(__ldg(p + i * rs + tid) - ms);
    mstar[tid] = ms;
    linv[tid] = 1.f / l;
    if (lse) lse[qrow0 + tid] = (ms + log2f(l)) * 0.6931471805599453f;
  }
  __syncthreads();
  // float4 outputs, eight independent partial loads in flight per thread
  for (int e = tid; e < G * d / 4; e += blockDim.x) {
    const int g = (4 * e) / d, j = (4 * e) % d;
    const float ms = mstar[g];
    const float* src = p + 16 + g * d + j;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int i = 0;
    for (; i + 8 <= n_items; i += 8) {
      float4 v[8];
      float wv[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        v[x] = __ldg(reinterpret_cast<const float4*>(src + (i + x) * rs));
        wv[x] = __ldg(p + (i + x) * rs + g);
      }
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float wx = fast_exp2(wv[x] - ms);
        acc.x = fmaf(wx, v[x].x, acc.x); acc.y = fmaf(wx, v[x].y, acc.y);
        acc.z = fmaf(wx, v[x].z, acc.z); acc.w = fmaf(wx, v[x].w, acc.w);
      }
    }
    for (; i < n_items; ++i) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src + i * rs));
      const float wx = fast_exp2(__ldg(p + i * rs + g) - ms);
      acc.x = fmaf(wx, v.x, acc.x); acc.y = fmaf(wx, v.y, acc.y);
      acc.z = fmaf(wx, v.z, acc.z); acc.w = fmaf(wx, v.w, acc.w);
    }
    const float li = linv[g];
    acc.x *= li; acc.y *= li; acc.z *= li; acc.w *= li;
    *reinterpret_cast<float4*>(out + (qrow0 + g) * d + j) = acc;
  }
}

}  // namespace

cudaError_t launch_route(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                         const uint8_t* cache, uint8_t* ws, int32_t* routed_out, cudaStream_t s) {
  const int G = n_q_heads / n_kv_heads;
  const float cq = 1.f / (sqrtf((float)L.d) * (float)G);
  const size_t smem = (size_t)L.NB * 8;
  static size_t configured = 48 * 1024;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  dim3 grid(P.route_splits, L.units);
  route_kernel<<<grid, 256, smem, s>>>(L, G, n_q_heads, n_kv_heads, P.K_eff, cq, q, cache,
                                       reinterpret_cast<float*>(ws + P.off_bounds),
                                       reinterpret_cast<uint32_t*>(ws + P.off_counters),
                                       reinterpret_cast<int32_t*>(ws + P.off_routed), routed_out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Layout& L, const DecodePlan& P, int batch, int n_q_heads, int n_kv_heads,
                           const float* partials, float* out, float* lse, cudaStream_t s) {
  (void)batch;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.units);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, P.n_items, n_q_heads / n_kv_heads, n_q_heads, n_kv_heads, L.d,
                            partials, out, lse);
}

}  // namespace dkv
