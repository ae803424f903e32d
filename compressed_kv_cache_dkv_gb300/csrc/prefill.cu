// Block-sparse prefill attention ("Prefill uses training-free block-sparse
// attention", DKV Zenodo abstract; "Sub-Quadratic Prefill", Differential-KV
// README section "Core Architecture & Paper Overview": O(L^2) down to O(L K)).
//
// Every 256-token query block attends the keys of its own block causally and
// every key of the top-K earlier blocks, ranked by the decode router's key-box
// bound taken with the block's mean query:
//   qbar_i   = mean over the block's tokens and the GQA group's heads of c q
//   bound_ij = sum_d max(qbar_id kmax_jd, qbar_id kmin_jd),   j < i
//   routed_i = top-K of j < i by (bound desc, j asc); every j < i when K is 0 or >= i
// Three kernels:
//   stats:  per (unit, block) the channel min/max of its keys and its mean query (fp32)
//   route:  per (unit, query block) the bounds of the earlier blocks, ranked on
//           order-preserving integer keys; the selected blocks written ascending
//   attend: one CTA of four warps per (64-query tile, query head), 16 queries a
//           warp; the key tiles of the routed blocks, then those of its own block
//           up to the diagonal one (causal mask), stream through a three-stage
//           cp.async pipeline of swizzled 64-token K and V tiles.  S = Q K^T and
//           O += P V on mma.sync m16n8k16 (fp16 operands, fp32 accumulation); the
//           S accumulators are the P operand registers of the next product, p split
//           into fp16 hi + lo; online softmax in base 2.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kPfThreads = 128;  // four warps, 16 queries each
constexpr int kPfQTile = 64;     // queries of one CTA
constexpr int kPfKTile = 64;     // keys of one pipeline stage
constexpr int kPfStages = 3;
constexpr int kPfMaxRouted = 1024;  // routed blocks of a query block kept in shared memory

struct PfArgs {
  int Hq, Hkv, G, T, nb, K_eff;
  float scale_log2;  // log2(e) / sqrt(d)
  float cq;          // 1 / (sqrt(d) G n) is applied per block in the stats kernel
  const __half* q;   // [B][Hq][T][d]
  const __half* K;   // [B][Hkv][T][d]
  const __half* V;
  float* kbox;       // [units][nb][2][d]  kmin, kmax
  float* qbar;       // [units][nb][d]
  int32_t* routed;   // [units][nb][K_eff]  ascending, -1 past the block's count
  float* out;        // [B][Hq][T][d]
  float* lse;        // [B][Hq][T] or null
};

// ---------------------------------------------------------------- stats
template <int D>
__global__ void __launch_bounds__(256) prefill_stats_kernel(PfArgs a) {
  const int j = blockIdx.x, u = blockIdx.y, b = u / a.Hkv, h = u % a.Hkv;
  const int t0 = j * 256, n = min(256, a.T - t0);
  const int tid = threadIdx.x;
  if (tid < D) {  // the block's key box, channel tid
    const __half* k = a.K + ((size_t)u * a.T + t0) * D + tid;
    float lo = INFINITY, hi = -INFINITY;
    for (int t = 0; t < n; ++t) {
      const float x = __half2float(k[(size_t)t * D]);
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
    float* box = a.kbox + ((size_t)u * a.nb + j) * 2 * D;
    box[tid] = lo;
    box[D + tid] = hi;
  } else if (tid < 2 * D) {  // the block's mean query over the group, channel tid - D
    const int c = tid - D;
    float s = 0.f;
    for (int g = 0; g < a.G; ++g) {
      const __half* qp = a.q + (((size_t)b * a.Hq + (size_t)h * a.G + g) * a.T + t0) * D + c;
      for (int t = 0; t < n; ++t) s += __half2float(qp[(size_t)t * D]);
    }
    a.qbar[((size_t)u * a.nb + j) * D + c] = s * (a.scale_log2 / 1.4426950408889634f) / (float)(a.G * n);
  }
}

// Order-preserving integer image of a bound (NaN ranked as -inf, -0 as +0)
__device__ inline int pf_key(float v) {
  if (isnan(v)) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const int x = __float_as_int(v);
  return x >= 0 ? x : x ^ 0x7fffffff;
}

// ---------------------------------------------------------------- route
template <int D>
__global__ void __launch_bounds__(256) prefill_route_kernel(PfArgs a) {
  extern __shared__ int keys[];  // [i] bound keys of the earlier blocks
  __shared__ float qb[D];
  __shared__ unsigned char sel[kPfMaxRouted + 1024];
  const int i = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
  int32_t* out = a.routed + ((size_t)u * a.nb + i) * a.K_eff;
  const int k = min(i, a.K_eff);
  if (k == i) {  // every earlier block
    for (int x = tid; x < a.K_eff; x += blockDim.x) out[x] = x < i ? x : -1;
    return;
  }
  for (int c = tid; c < D; c += blockDim.x) qb[c] = a.qbar[((size_t)u * a.nb + i) * D + c];
  __syncthreads();
  for (int j = tid; j < i; j += blockDim.x) {
    const float* box = a.kbox + ((size_t)u * a.nb + j) * 2 * D;
    float s = 0.f;
    for (int c = 0; c < D; ++c) s += fmaxf(qb[c] * box[c], qb[c] * box[D + c]);
    keys[j] = pf_key(s);
  }
  __syncthreads();
  for (int j = tid; j < i; j += blockDim.x) {  // rank = blocks ahead by (bound desc, index asc)
    const int kj = keys[j];
    int rank = 0;
    for (int x = 0; x < i; ++x) rank += (keys[x] > kj) || (keys[x] == kj && x < j);
    sel[j] = rank < k;
  }
  __syncthreads();
  if (tid == 0) {  // ascending
    int pos = 0;
    for (int j = 0; j < i; ++j)
      if (sel[j]) out[pos++] = j;
    for (; pos < a.K_eff; ++pos) out[pos] = -1;
  }
}

// ---------------------------------------------------------------- attend
__device__ inline void pf_cp16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ inline void pf_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void pf_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ inline uint4 pf_ldsm(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ inline uint4 pf_ldsm_t(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
template <int D>
__device__ inline uint32_t pf_swz(int row, int chunk) {  // 16-byte chunk of a row, XOR-swizzled by row
  return (uint32_t)(row * D * 2 + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 2) prefill_attend_kernel(PfArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KT = D / 16, NT = kPfKTile / 8, CPR = D / 8;
  constexpr uint32_t TILE = kPfKTile * D * 2;
  int* rsm = reinterpret_cast<int*>(smem + kPfStages * 2 * TILE);  // [kPfMaxRouted]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3, gq = lane >> 2;
  const int mi = lane >> 3, mr = lane & 7;
  const int q0 = blockIdx.x * kPfQTile, hq = blockIdx.y, b = blockIdx.z;
  const int h = hq / a.G, u = b * a.Hkv + h, i = q0 / 256;
  const __half* Kb = a.K + (size_t)u * a.T * D;
  const __half* Vb = a.V + (size_t)u * a.T * D;
  const uint32_t sbase = smem_u32(smem);
  // the tile list: the routed blocks' four tiles each, then the own block's tiles up to the diagonal
  const int n_r = min(i, a.K_eff);
  for (int x = threadIdx.x; x < n_r; x += kPfThreads) rsm[x] = a.routed[((size_t)u * a.nb + i) * a.K_eff + x];
  __syncthreads();
  const int own_last = (q0 - i * 256) / kPfKTile;
  const int ntile = 4 * n_r + own_last + 1;
  auto tile_key0 = [&](int p) -> int {
    return p < 4 * n_r ? rsm[p >> 2] * 256 + (p & 3) * kPfKTile : i * 256 + (p - 4 * n_r) * kPfKTile;
  };
  auto issue = [&](int p) {
    const int k0 = tile_key0(p);
    const uint32_t kd = sbase + (uint32_t)(p % kPfStages) * 2u * TILE, vd = kd + TILE;
    for (int e = threadIdx.x; e < kPfKTile * CPR; e += kPfThreads) {
      const int r = e / CPR, ch = e % CPR;
      const int tok = k0 + r;
      const bool valid = tok < a.T;
      const size_t off = (size_t)(valid ? tok : 0) * D + ch * 8;  // rows past the sequence read zeros
      pf_cp16(kd + pf_swz<D>(r, ch), Kb + off, valid ? 16u : 0u);
      pf_cp16(vd + pf_swz<D>(r, ch), Vb + off, valid ? 16u : 0u);
    }
  };
#pragma unroll
  for (int s = 0; s < kPfStages - 1; ++s) {
    if (s < ntile) issue(s);
    pf_commit();
  }
  // this warp's 16 queries as A fragments (rows = queries, k = d)
  const int qr0 = q0 + 16 * warp + gq, qr1 = qr0 + 8;
  uint32_t qa[KT][4];
  {
    const __half* qp = a.q + ((size_t)b * a.Hq + hq) * a.T * D;
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(qp + (size_t)min(qr0, a.T - 1) * D);
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(qp + (size_t)min(qr1, a.T - 1) * D);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      qa[kt][0] = __ldg(r0 + 8 * kt + t);
      qa[kt][1] = __ldg(r1 + 8 * kt + t);
      qa[kt][2] = __ldg(r0 + 8 * kt + 4 + t);
      qa[kt][3] = __ldg(r1 + 8 * kt + 4 + t);
    }
  }
  const float slog2 = a.scale_log2;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq, gq + 8
  float o[D / 8][4];
#pragma unroll
  for (int x = 0; x < D / 8; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
  for (int p = 0; p < ntile; ++p) {
    if (p + kPfStages - 1 < ntile) issue(p + kPfStages - 1);
    pf_commit();
    pf_wait<kPfStages - 1>();
    __syncthreads();
    const uint32_t kb = sbase + (uint32_t)(p % kPfStages) * 2u * TILE, vb = kb + TILE;
    const int k0 = tile_key0(p);
    const bool diag = p == ntile - 1;
    // ---- S = Q K^T over the tile's 64 keys: 8 n-tiles of 8 keys
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int row = 16 * np + (mi >> 1) * 8 + mr;  // keys of n-tiles 2 np, 2 np + 1
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const uint4 kv = pf_ldsm(kb + pf_swz<D>(row, 2 * kt + (mi & 1)));
        mma16816(s[2 * np], qa[kt][0], qa[kt][1], qa[kt][2], qa[kt][3], kv.x, kv.y);
        mma16816(s[2 * np + 1], qa[kt][0], qa[kt][1], qa[kt][2], qa[kt][3], kv.z, kv.w);
      }
    }
    // ---- scale, masks (keys past the sequence; on the diagonal tile keys after the query)
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int kk = k0 + 8 * nt + 2 * t;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kk + e;
        const bool bad0 = key >= a.T || (diag && key > qr0);
        const bool bad1 = key >= a.T || (diag && key > qr1);
        s[nt][e] = bad0 ? -INFINITY : s[nt][e] * slog2;
        s[nt][2 + e] = bad1 ? -INFINITY : s[nt][2 + e] * slog2;
      }
      x0 = fmaxf(x0, fmaxf(s[nt][0], s[nt][1]));
      x1 = fmaxf(x1, fmaxf(s[nt][2], s[nt][3]));
    }
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    const float ms0 = n0 == -INFINITY ? 0.f : n0, ms1 = n1 == -INFINITY ? 0.f : n1;
    const float sc0 = fast_exp2(m0 - ms0), sc1 = fast_exp2(m1 - ms1);
    m0 = n0;
    m1 = n1;
    l0 *= sc0;
    l1 *= sc1;
#pragma unroll
    for (int x = 0; x < D / 8; ++x) { o[x][0] *= sc0; o[x][1] *= sc0; o[x][2] *= sc1; o[x][3] *= sc1; }
    // ---- O += P V: the S fragments of n-tiles 2 kk, 2 kk + 1 are the P fragment of key k-tile kk
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
      float p0[4], p1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p0[e] = fast_exp2(s[2 * kk][e] - (e < 2 ? ms0 : ms1));
        p1[e] = fast_exp2(s[2 * kk + 1][e] - (e < 2 ? ms0 : ms1));
      }
      l0 += (p0[0] + p0[1]) + (p1[0] + p1[1]);
      l1 += (p0[2] + p0[3]) + (p1[2] + p1[3]);
      uint32_t h0, lo0, h1, lo1, h2, lo2, h3, lo3;
      split_half2(p0[0], p0[1], h0, lo0);  // a0: row gq, keys 2t.. of the k-tile's first 8
      split_half2(p0[2], p0[3], h1, lo1);  // a1: row gq + 8
      split_half2(p1[0], p1[1], h2, lo2);  // a2: row gq, keys 8 + 2t..
      split_half2(p1[2], p1[3], h3, lo3);  // a3: row gq + 8
      const int row = 16 * kk + (mi & 1) * 8 + mr;  // V rows (keys) of the k-tile
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const uint4 vv = pf_ldsm_t(vb + pf_swz<D>(row, 2 * dp + (mi >> 1)));
        mma16816(o[2 * dp], h0, h1, h2, h3, vv.x, vv.y);
        mma16816(o[2 * dp], lo0, lo1, lo2, lo3, vv.x, vv.y);
        mma16816(o[2 * dp + 1], h0, h1, h2, h3, vv.z, vv.w);
        mma16816(o[2 * dp + 1], lo0, lo1, lo2, lo3, vv.z, vv.w);
      }
    }
    __syncthreads();  // the stage is refilled by a later issue
  }
  pf_wait<0>();
  // ---- normalise and write rows gq, gq + 8 (l summed over the four lanes of a row)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float i0 = 1.f / l0, i1 = 1.f / l1;
  float* ob = a.out + ((size_t)b * a.Hq + hq) * a.T * D;
#pragma unroll
  for (int x = 0; x < D / 8; ++x) {
    const int c = 8 * x + 2 * t;
    if (qr0 < a.T) *reinterpret_cast<float2*>(ob + (size_t)qr0 * D + c) = make_float2(o[x][0] * i0, o[x][1] * i0);
    if (qr1 < a.T) *reinterpret_cast<float2*>(ob + (size_t)qr1 * D + c) = make_float2(o[x][2] * i1, o[x][3] * i1);
  }
  if (a.lse && t == 0) {
    float* lb = a.lse + ((size_t)b * a.Hq + hq) * a.T;
    if (qr0 < a.T) lb[qr0] = (m0 + log2f(l0)) * 0.6931471805599453f;
    if (qr1 < a.T) lb[qr1] = (m1 + log2f(l1)) * 0.6931471805599453f;
  }
}

template <int D>
cudaError_t launch_prefill_d(const PfArgs& a, int batch, cudaStream_t s) {
  const int units = batch * a.Hkv;
  prefill_stats_kernel<D><<<dim3(a.nb, units), 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prefill_route_kernel<D><<<dim3(a.nb, units), 256, (size_t)a.nb * 4, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)kPfStages * 2 * kPfKTile * D * 2 + (size_t)kPfMaxRouted * 4;
  e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_attend_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  prefill_attend_kernel<D><<<dim3((a.T + kPfQTile - 1) / kPfQTile, a.Hq, batch), kPfThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

PrefillPlan plan_prefill(int batch, int n_kv_heads, int d, int T, int top_k) {
  PrefillPlan P;
  P.nb = (T + 255) / 256;
  P.K_eff = (top_k == 0 || top_k >= P.nb - 1) ? (P.nb > 1 ? P.nb - 1 : 1) : top_k;
  const size_t units = (size_t)batch * n_kv_heads;
  P.off_kbox = kWsHeader;
  P.off_qbar = round_up(P.off_kbox + units * P.nb * 2 * d * 4, 256);
  P.off_routed = round_up(P.off_qbar + units * P.nb * d * 4, 256);
  P.ws_bytes = P.off_routed + units * P.nb * P.K_eff * 4;
  return P;
}

cudaError_t launch_prefill(int batch, int n_q_heads, int n_kv_heads, int d, int T, int top_k, const __half* q,
                           const __half* K, const __half* V, float* out, float* lse, int32_t* routed_out, uint8_t* ws,
                           cudaStream_t s) {
  const PrefillPlan P = plan_prefill(batch, n_kv_heads, d, T, top_k);
  PfArgs a;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.G = n_q_heads / n_kv_heads;
  a.T = T;
  a.nb = P.nb;
  a.K_eff = P.K_eff;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  a.cq = 0.f;
  a.q = q;
  a.K = K;
  a.V = V;
  a.kbox = reinterpret_cast<float*>(ws + P.off_kbox);
  a.qbar = reinterpret_cast<float*>(ws + P.off_qbar);
  a.routed = routed_out ? routed_out : reinterpret_cast<int32_t*>(ws + P.off_routed);
  a.out = out;
  a.lse = lse;
  return d == 128 ? launch_prefill_d<128>(a, batch, s) : launch_prefill_d<64>(a, batch, s);
}

}  // namespace dkv
