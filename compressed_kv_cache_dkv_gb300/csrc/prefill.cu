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
//   attend: head_dim 128 on the tcgen05 tensor cores (prefill_attend_tc_kernel,
//           below); head_dim 64 on mma.sync: one CTA of four warps per (64-query
//           tile, query head), 16 queries a warp; the key tiles of the routed blocks, then those of its own block
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
  uint32_t* err;     // the workspace header's device error word
};

// ---------------------------------------------------------------- stats
template <int D>
__global__ void __launch_bounds__(256) prefill_stats_kernel(PfArgs a) {
  // 16-byte loads: D / 8 threads cover a row, 256 / (D / 8) rows at a time; the per-row-slot
  // partials meet in shared memory and are reduced in a fixed order
  constexpr int kTpr = D / 8, kRows = 256 / kTpr;
  __shared__ float red[2][kRows][D];
  const int j = blockIdx.x, u = blockIdx.y, b = u / a.Hkv, h = u % a.Hkv;
  const int t0 = j * 256, n = min(256, a.T - t0);
  const int tid = threadIdx.x, rs = tid / kTpr, c0 = (tid % kTpr) * 8;
  float lo[8], hi[8], sm[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    lo[e] = INFINITY;
    hi[e] = -INFINITY;
    sm[e] = 0.f;
  }
  const __half* kb = a.K + ((size_t)u * a.T + t0) * D + c0;
#pragma unroll 4
  for (int t = rs; t < n; t += kRows) {  // the block's key box
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(kb + (size_t)t * D));
    const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h2[e]);
      lo[2 * e] = fminf(lo[2 * e], f.x);
      hi[2 * e] = fmaxf(hi[2 * e], f.x);
      lo[2 * e + 1] = fminf(lo[2 * e + 1], f.y);
      hi[2 * e + 1] = fmaxf(hi[2 * e + 1], f.y);
    }
  }
  for (int g = 0; g < a.G; ++g) {  // the sum of the group's queries over the block
    const __half* qb = a.q + (((size_t)b * a.Hq + (size_t)h * a.G + g) * a.T + t0) * D + c0;
#pragma unroll 4
    for (int t = rs; t < n; t += kRows) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qb + (size_t)t * D));
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h2[e]);
        sm[2 * e] += f.x;
        sm[2 * e + 1] += f.y;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    red[0][rs][c0 + e] = lo[e];
    red[1][rs][c0 + e] = hi[e];
  }
  __syncthreads();
  if (tid < D) {
    float l = INFINITY, m = -INFINITY;
    for (int r = 0; r < kRows; ++r) {
      l = fminf(l, red[0][r][tid]);
      m = fmaxf(m, red[1][r][tid]);
    }
    float* box = a.kbox + ((size_t)u * a.nb + j) * 2 * D;
    box[tid] = l;
    box[D + tid] = m;
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 8; ++e) red[0][rs][c0 + e] = sm[e];
  __syncthreads();
  if (tid < D) {  // the block's mean query over the group
    float x = 0.f;
    for (int r = 0; r < kRows; ++r) x += red[0][r][tid];
    a.qbar[((size_t)u * a.nb + j) * D + tid] = x * (a.scale_log2 / 1.4426950408889634f) / (float)(a.G * n);
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
  {  // one warp per earlier block: lanes over the channels, then a butterfly sum
    const int warp = tid >> 5, lane = tid & 31;
    for (int j = warp; j < i; j += (int)(blockDim.x >> 5)) {
      const float* box = a.kbox + ((size_t)u * a.nb + j) * 2 * D;
      float s = 0.f;
#pragma unroll
      for (int x = 0; x < D / 32; ++x) {
        const int c = lane + 32 * x;
        s += fmaxf(qb[c] * __ldg(box + c), qb[c] * __ldg(box + D + c));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) keys[j] = pf_key(s);
    }
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

// ---------------------------------------------------------------- attend on tcgen05 (head_dim 128)
// One CTA per (256-token query block, query head), as two groups of 128 query rows
// (A: the block's first 128 queries, B: the rest) that share every K and V tile, so
// a tile crosses from L2 once for 256 rows.  Warps 0-3 own group A's rows and warps
// 4-7 group B's, one row per thread in tensor-memory lane 32 (w % 4) + lane; warp 9
// streams the 64-key K and V tiles with cp.async into a four-stage ring: a stage
// takes tile t once the products of tile t - 4 have read it, and each lane's copies
// arrive on the stage's "loaded" barrier by themselves when they land
// (cp.async.mbarrier.arrive), so no arrival waits on a later product.  Each
// tcgen05.mma holds its issuing thread for about 75 cycles, so four threads issue:
// lane 0 of warps 8 and 11 the S products of groups A and B, of warps 10 and 12 their
// O products:
//   S_gj = Q_g K_j^T   M = 128 queries, N = 64 keys, K = 128     (TMEM, two buffers per group)
//   O_g += P_gj V_j    M = 128, N = 128 channels, K = 64 keys    (P from TMEM, V from shared memory)
// Q and K_j sit in shared memory as 8x8 core matrices without swizzle, K-major (rows
// = queries / keys, 16-byte rows of 8 channels); V_j is the same bytes read MN-major.
// The rows write P_gj (fp16 hi in columns 0-31, lo in 32-63, two keys a column) over
// the S_gj they have just read, and the tensor cores take it from there as the A
// operand.  While one group's rows turn S into P, the tensor cores run the other
// group's products, and no issuing thread waits for another.  S_{g,j} overwrites
// P_{g,j-2}, so it is issued once O_{g,j-2} is done.  Online softmax in base 2 with a
// lazy rescale: the row maximum moves only when a score exceeds it by kPtSlack, and
// only then do the rows wait for O_{g,j-1} and rescale O in tensor memory.  Group A
// stops after the block's second own tile (keys past its last query).
constexpr int kPtThreads = 416;  // 8 softmax warps (two groups), the load warp, S- and O-issuing warps per group
constexpr int kPtM = 128, kPtN = 64, kPtStages = 4;
constexpr float kPtSlack = 8.f;
constexpr uint32_t kPtTile = kPtN * 128 * 2;                      // one K or V tile: 16 KB
constexpr uint32_t kPtQ = kPtM * 128 * 2;                         // one group's Q: 32 KB
constexpr uint32_t kPtOffQ = 0;                                   // Q_A | Q_B
constexpr uint32_t kPtOffKV = kPtOffQ + 2 * kPtQ;                 // [stage][K | V]
constexpr uint32_t kPtOffBar = kPtOffKV + kPtStages * 2 * kPtTile; // mbarriers, TMEM address
constexpr uint32_t kPtSmem = kPtOffBar + 256;
constexpr uint32_t kPtTmemCols = 512;  // per group g: S / P buffers at 256 g + {0, 64}, O at 256 g + 128
constexpr uint32_t kPtColO = 128;

__device__ inline uint64_t pt_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}
// D f32, A and B f16, M = 128, N = n; a_mn / b_mn: MN-major operand
__device__ inline uint32_t pt_idesc(bool a_mn, bool b_mn, uint32_t n) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
// A and B from shared-memory descriptors
__device__ inline void pt_mma(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(id), "r"(acc)
      : "memory");
}
// A from tensor memory (row = lane, two 16-bit elements of K a column), B from a descriptor
__device__ inline void pt_mma_ta(uint32_t dt, uint32_t at, uint64_t bd, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(dt),
      "r"(at), "l"(bd), "r"(id), "r"(acc)
      : "memory");
}
__device__ inline void pt_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ inline void pt_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void pt_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ inline void pt_fence_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 16 consecutive fp32 columns of this thread's lane; the caller waits (pt_ld_wait)
__device__ inline void pt_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ inline void pt_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ inline void pt_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ inline void pt_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// arrive on `bar` once every cp.async this thread issued so far has landed (no count increment)
__device__ inline void pt_cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ inline void pt_cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// byte offset of (row, 16-byte chunk cc) of a K-major [rows x 128] fp16 operand in core matrices
__device__ inline uint32_t pt_core(int row, int cc) {
  return (uint32_t)((row >> 3) * 2048 + cc * 128 + (row & 7) * 16);
}

__global__ void __launch_bounds__(kPtThreads, 1) prefill_attend_tc_kernel(PfArgs a, int nqb) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + kPtOffBar);  // [group][j % 2] S_gj ready (commit)
  uint64_t* bar_p = bar_s + 4;                                       // [group][j % 2] P_gj written by the group's rows
  uint64_t* bar_o = bar_s + 8;                                       // [group][j % 2] O_g += P_gj V_j done (commit)
  uint64_t* bar_end = bar_s + 12;                                    // [group] the group's last product done (commit)
  uint64_t* bar_kv = bar_s + 14;                                     // [stage] loaded (32 loader lanes)
  uint64_t* bar_fr = bar_kv + kPtStages;                             // [stage] free again (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_fr + kPtStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int i = nqb - 1 - (int)blockIdx.x;  // later query blocks (more keys without routing) first
  const int q0 = i * 256, hq = blockIdx.y, b = blockIdx.z;
  const int h = hq / a.G, u = b * a.Hkv + h;
  const int n_r = min(i, a.K_eff);
  // query rows of the groups and the own-block tiles each needs (up to its last query)
  const int rowsA = min(kPtM, a.T - q0), rowsB = max(0, min(kPtM, a.T - q0 - kPtM));
  const int ownA = (rowsA + kPtN - 1) / kPtN, ownB = rowsB > 0 ? (kPtM + rowsB + kPtN - 1) / kPtN : 0;
  const int ntA = 4 * n_r + ownA, ntB = rowsB > 0 ? 4 * n_r + ownB : 0;
  const int ntile = max(ntA, ntB);
  const int32_t* routed = a.routed + ((size_t)u * a.nb + i) * a.K_eff;
  const __half* Kb = a.K + (size_t)u * a.T * 128;
  const __half* Vb = a.V + (size_t)u * a.T * 128;
  if (tid == 0) {
    for (int x = 0; x < 4; ++x) {
      mbar_init(&bar_s[x], 1);
      mbar_init(&bar_p[x], 128);
      mbar_init(&bar_o[x], 1);
    }
    for (int x = 0; x < 2; ++x) mbar_init(&bar_end[x], 1);
    for (int x = 0; x < kPtStages; ++x) {
      mbar_init(&bar_kv[x], 32);
      mbar_init(&bar_fr[x], 4);  // one commit from each issuing thread
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(kPtTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  pt_fence_before();
  __syncthreads();
  pt_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 9) {
    // =========================== loads (Q with tile 0)
    auto load_kv = [&](int p) {
      const int k0 = p < 4 * n_r ? __ldg(routed + (p >> 2)) * 256 + (p & 3) * kPtN : q0 + (p - 4 * n_r) * kPtN;
      const uint32_t kd = sb + kPtOffKV + (uint32_t)(p % kPtStages) * 2u * kPtTile, vd = kd + kPtTile;
      // one instruction fills 8 rows x 4 chunks: 512 contiguous bytes of core matrices
#pragma unroll 4
      for (int it = 0; it < kPtN * 16 / 32; ++it) {
        const int r = 8 * (it >> 2) + (lane & 7), cc = 4 * (it & 3) + (lane >> 3), tok = k0 + r;
        const bool valid = tok < a.T;
        const size_t off = (size_t)(valid ? tok : 0) * 128 + cc * 8;  // rows past the prompt read zeros
        pf_cp16(kd + pt_core(r, cc), Kb + off, valid ? 16u : 0u);
        pf_cp16(vd + pt_core(r, cc), Vb + off, valid ? 16u : 0u);
      }
    };
    {
      const __half* qp = a.q + ((size_t)b * a.Hq + hq) * a.T * 128;
      for (int it = 0; it < 2 * kPtM * 16 / 32; ++it) {
        const int r = 8 * (it >> 2) + (lane & 7), cc = 4 * (it & 3) + (lane >> 3), tok = q0 + r;
        const bool valid = tok < a.T;
        pf_cp16(sb + kPtOffQ + (uint32_t)(r >> 7) * kPtQ + pt_core(r & 127, cc), qp + (size_t)(valid ? tok : 0) * 128 + cc * 8,
                valid ? 16u : 0u);
      }
    }
    for (int p = 0; p < ntile && ok; ++p) {
      // stage p % 4 held tile p - 4: wait until every product that reads it is done
      if (p >= kPtStages) ok = mbar_wait(&bar_fr[p % kPtStages], (uint32_t)(((p / kPtStages) - 1) & 1), a.err);
      if (!ok) break;
      load_kv(p);
      pt_cp_arrive(&bar_kv[p % kPtStages]);
    }
    pt_cp_wait_all();
  } else if (warp == 8 || warp >= 10) {
    // =========================== tensor-core issue, lane 0 of: warp 8 S_A, 10 O_A, 11 S_B, 12 O_B
    const int g = warp >= 11 ? 1 : 0, nt = g ? ntB : ntA, nt_other = g ? ntA : ntB;
    const bool o_side = warp == 10 || warp == 12;
    if (lane == 0) {
      const uint32_t tg = tmem + 256u * (uint32_t)g;
      // a stage is free once every product of its tile is done: each thread commits once per
      // tile its group takes, and twice where the other group has no such tile
      auto release = [&](int j) {
        pt_commit(&bar_fr[j % kPtStages]);
        if (j >= nt_other) pt_commit(&bar_fr[j % kPtStages]);
      };
      if (!o_side) {
        const uint32_t id_s = pt_idesc(false, false, kPtN);
        const uint64_t qdesc = pt_sdesc(sb + kPtOffQ + (uint32_t)g * kPtQ, 128u, 2048u);
        for (int j = 0; j < nt && ok; ++j) {  // S_gj = Q_g K_j^T into buffer j % 2
          ok = mbar_wait(&bar_kv[j % kPtStages], (uint32_t)((j / kPtStages) & 1), a.err);
          pt_fence_async();  // the landed cp.async bytes, seen through the barrier, for the tensor cores
          // the buffer holds P_{g,j-2}: O_{g,j-2} has to be done reading it
          if (j >= 2 && ok) ok = mbar_wait(&bar_o[2 * g + (j & 1)], (uint32_t)(((j - 2) >> 1) & 1), a.err);
          pt_fence_after();
          if (!ok) break;
          const uint64_t kdesc = pt_sdesc(sb + kPtOffKV + (uint32_t)(j % kPtStages) * 2u * kPtTile, 128u, 2048u);
          const uint32_t dt = tg + (uint32_t)(j & 1) * kPtN;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) pt_mma(dt, qdesc + (uint64_t)(ks * 16), kdesc + (uint64_t)(ks * 16), id_s, ks > 0);
          pt_commit(&bar_s[2 * g + (j & 1)]);
          release(j);
        }
      } else {
        const uint32_t id_o = pt_idesc(false, true, 128);
        for (int j = 0; j < nt && ok; ++j) {  // O_g += P_gj V_j, P from S_gj's buffer
          ok = mbar_wait(&bar_p[2 * g + (j & 1)], (uint32_t)((j >> 1) & 1), a.err);
          pt_fence_after();
          if (!ok) break;
          const uint64_t vdesc = pt_sdesc(sb + kPtOffKV + (uint32_t)(j % kPtStages) * 2u * kPtTile + kPtTile, 2048u, 128u);
          const uint32_t pt = tg + (uint32_t)(j & 1) * kPtN, dt = tg + kPtColO;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            pt_mma_ta(dt, pt + 8u * (uint32_t)ks, vdesc + (uint64_t)(ks * 256), id_o, (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) pt_mma_ta(dt, pt + 32u + 8u * (uint32_t)ks, vdesc + (uint64_t)(ks * 256), id_o, 1u);
          pt_commit(&bar_o[2 * g + (j & 1)]);
          if (j == nt - 1) pt_commit(&bar_end[g]);
          release(j);
        }
      }
    }
  } else {
    // =========================== softmax: group g = warp / 4, one query row per thread
    const int g = warp >> 2, rw = warp & 3, row = 32 * rw + lane, qrow = q0 + kPtM * g + row;
    const int nt = g ? ntB : ntA;
    const uint32_t tl = tmem + ((uint32_t)(rw * 32) << 16) + 256u * (uint32_t)g;
    const float slog2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) {
      if (ok) ok = mbar_wait(&bar_s[2 * g + (j & 1)], (uint32_t)((j >> 1) & 1), a.err);
      pt_fence_after();
      uint32_t r[4][16];
      const uint32_t sc = tl + (uint32_t)(j & 1) * kPtN;
#pragma unroll
      for (int c = 0; c < 4; ++c) pt_ld16(sc + 16 * c, r[c]);
      pt_ld_wait();
      if (j >= 4 * n_r) {  // the own block: keys k0 + c valid for c < nv (causal, before the prompt's end)
        const int k0 = q0 + (j - 4 * n_r) * kPtN, nv = min(a.T, qrow + 1) - k0;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= nv) r[c >> 4][c & 15] = 0xff800000u;  // -inf
      }
      float mxp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 64; ++c) mxp[c & 3] = fmaxf(mxp[c & 3], __uint_as_float(r[c >> 4][c & 15]));
      // scaling by slog2 > 0 keeps the order, so the scaled maximum is the maximum scaled
      const float mx = fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])) * slog2;
      const bool up = mx > m + kPtSlack;
      const bool resc = __any_sync(0xffffffffu, up) && j > 0;
      const float nm = up ? mx : m;
      const float al = nm == -INFINITY ? 1.f : fast_exp2(m - nm);  // the factor on l and O (1 where m stays)
      m = nm;
      const float ms = m == -INFINITY ? 0.f : m;
      // P_gj over S_gj: hi words in columns 0-31, lo words in 32-63 (keys 2w and 2w + 1 in word w)
      float lp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int k = 32 * c + 2 * e;
          const float p0 = fast_exp2(fmaf(__uint_as_float(r[k >> 4][k & 15]), slog2, -ms));
          const float p1 = fast_exp2(fmaf(__uint_as_float(r[k >> 4][(k & 15) + 1]), slog2, -ms));
          lp[e & 3] += p0 + p1;
          split_half2(p0, p1, hi[e], lo[e]);
        }
        pt_st16(sc + 16u * (uint32_t)c, hi);
        pt_st16(sc + 32u + 16u * (uint32_t)c, lo);
      }
      l = fmaf(l, al, (lp[0] + lp[1]) + (lp[2] + lp[3]));
      if (resc) {  // O_{g,j-1} done, then O *= al in tensor memory
        if (ok) ok = mbar_wait(&bar_o[2 * g + ((j - 1) & 1)], (uint32_t)(((j - 1) >> 1) & 1), a.err);
        pt_fence_after();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[16];
          pt_ld16(tl + kPtColO + 16u * (uint32_t)c, o);
          pt_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * al);
          pt_st16(tl + kPtColO + 16u * (uint32_t)c, o);
        }
      }
      pt_st_wait();
      pt_fence_before();
      mbar_arrive(&bar_p[2 * g + (j & 1)]);
    }
    // the group's last product: normalise and store this row
    if (nt > 0 && ok) ok = mbar_wait(&bar_end[g], 0u, a.err);
    pt_fence_after();
    const float il = 1.f / l;
    const bool live = (g ? rowsB : rowsA) > row;
    float* orow = a.out + (((size_t)b * a.Hq + hq) * a.T + (size_t)min(qrow, a.T - 1)) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t o[16];
      pt_ld16(tl + kPtColO + 16u * (uint32_t)c, o);
      pt_ld_wait();
      if (live && nt > 0) {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(orow + 16 * c + e) =
              make_float4(__uint_as_float(o[e]) * il, __uint_as_float(o[e + 1]) * il, __uint_as_float(o[e + 2]) * il,
                          __uint_as_float(o[e + 3]) * il);
      }
    }
    if (live && nt > 0 && a.lse) a.lse[((size_t)b * a.Hq + hq) * a.T + qrow] = (m + log2f(l)) * 0.6931471805599453f;
  }
  pt_fence_before();
  __syncthreads();
  pt_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kPtTmemCols) : "memory");
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
  if (D == 128) {  // tensor cores with TMEM accumulators
    e = ensure_smem_limit(reinterpret_cast<const void*>(prefill_attend_tc_kernel), kPtSmem);
    if (e != cudaSuccess) return e;
    prefill_attend_tc_kernel<<<dim3(a.nb, a.Hq, batch), kPtThreads, kPtSmem, s>>>(a, a.nb);
    return cudaGetLastError();
  }
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
  a.err = reinterpret_cast<uint32_t*>(ws);
  return d == 128 ? launch_prefill_d<128>(a, batch, s) : launch_prefill_d<64>(a, batch, s);
}

}  // namespace dkv
