// Dense fp16 decode attention over uncompressed K, V: the bytes/throughput
// reference of the compressed path (the dense full-KV baselines the DKV Zenodo
// abstract compares against; "Measured Paper Benchmarks" of the
// Differential-KV README).  Exact softmax attention of every query against all
// T tokens of its KV head, fp16 operands, fp32 accumulation, split over token
// chunks and merged by the same fp32 log-sum-exp combine as the compressed path.
//
// One CTA of four warps per (unit, token chunk).  64-token K and V tiles stream
// through a three-stage cp.async pipeline into row-major shared-memory tiles
// whose 16-byte chunks are XOR-swizzled by row (conflict-free ldmatrix); warp w
// owns tokens 16w..16w+15 of every tile:
//   S   = K q        ldmatrix.x4 K fragments, mma.sync m16n8k16, tokens in M
//   o  += V^T p      ldmatrix.x4.trans V^T fragments, p split into fp16 hi + lo
// with a per-warp online softmax (base-2 units).  The four warps merge into one
// partial record [m 8][l 8][o 8 x d] per chunk.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kDenseThreads = 128;
constexpr int kDenseTile = 64;     // tokens per pipeline stage (16 per warp)
constexpr int kDenseStages = 3;
constexpr int kDenseWaves = 4;  // work items aimed at: about four resident waves of two CTAs per SM

struct DenseArgs {
  int Hq, Hkv, G, T, chunk, nchunk;
  float scale_log2;  // log2(e) / sqrt(d)
  const __half* q;
  const __half* K;
  const __half* V;
  float* partials;
};

__device__ inline void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ inline uint4 ldsm_x4(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ inline uint4 ldsm_x4_trans(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

template <int D>
__device__ inline uint32_t swz(int row, int chunk) {  // byte offset of a 16-byte chunk in a swizzled tile
  return (uint32_t)(row * D * 2 + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kDenseThreads, 2) dense_kernel(DenseArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KT = D / 16;
  constexpr int CPR = D / 8;                        // 16-byte chunks per row
  constexpr uint32_t TILE = kDenseTile * D * 2;     // bytes of one K (or V) tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = lane & 3, gq = lane >> 2;
  const int u = blockIdx.x / a.nchunk, c = blockIdx.x % a.nchunk;
  const int b = u / a.Hkv, h = u % a.Hkv;
  const int t0 = c * a.chunk, t1 = min(a.T, t0 + a.chunk);
  const int ntile = (t1 - t0 + kDenseTile - 1) / kDenseTile;
  const __half* Kb = a.K + (size_t)u * a.T * D;
  const __half* Vb = a.V + (size_t)u * a.T * D;
  const uint32_t sbase = smem_u32(smem);

  auto issue = [&](int tile) {
    const int tok0 = t0 + tile * kDenseTile;
    const uint32_t kd = sbase + (uint32_t)(tile % kDenseStages) * 2u * TILE, vd = kd + TILE;
    for (int e = threadIdx.x; e < kDenseTile * CPR; e += kDenseThreads) {
      const int r = e / CPR, ch = e % CPR;
      const int tok = tok0 + r;
      const bool valid = tok < t1;
      const size_t off = (size_t)(valid ? tok : t0) * D + ch * 8;  // rows past the chunk read zeros
      cp_async16(kd + swz<D>(r, ch), Kb + off, valid ? 16u : 0u);
      cp_async16(vd + swz<D>(r, ch), Vb + off, valid ? 16u : 0u);
    }
  };
#pragma unroll
  for (int i = 0; i < kDenseStages - 1; ++i) {
    if (i < ntile) issue(i);
    cp_async_commit();
  }

  // q as B fragments (k = head dim, n = group): q[gq][16kt + 2t, +1] and [16kt + 8 + 2t, +1]
  uint32_t qb[KT][2];
  {
    const bool gv = gq < a.G;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(a.q + ((size_t)b * a.Hq + (size_t)h * a.G + (gv ? gq : 0)) * D);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      qb[kt][0] = gv ? __ldg(qrow + 8 * kt + t) : 0u;
      qb[kt][1] = gv ? __ldg(qrow + 8 * kt + 4 + t) : 0u;
    }
  }
  const bool gv0 = 2 * t < a.G, gv1 = 2 * t + 1 < a.G;
  const float slog2 = a.scale_log2;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[KT][4];
#pragma unroll
  for (int i = 0; i < KT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  // ldmatrix lane roles: matrix mi = lane / 8, row lane % 8
  const int mi = lane >> 3, mr = lane & 7;

  for (int tile = 0; tile < ntile; ++tile) {
    if (tile + kDenseStages - 1 < ntile) issue(tile + kDenseStages - 1);
    cp_async_commit();
    cp_async_wait<kDenseStages - 1>();
    __syncthreads();
    const uint32_t kb = sbase + (uint32_t)(tile % kDenseStages) * 2u * TILE, vb = kb + TILE;
    // ---- scores of this warp's 16 tokens
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int row = 16 * warp + (mi & 1) * 8 + mr;  // K fragment matrices: (rows 0-7 | 8-15) x (k lo | hi)
      uint4 kv[KT];
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) kv[kt] = ldsm_x4(kb + swz<D>(row, 2 * kt + (mi >> 1)));
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) mma16816(acc, kv[kt].x, kv[kt].y, kv[kt].z, kv[kt].w, qb[kt][0], qb[kt][1]);
    }
    const int tk0 = t0 + tile * kDenseTile + 16 * warp + gq, tk1 = tk0 + 8;
    const bool v0 = tk0 < t1, v1 = tk1 < t1;
    float s[4];
    s[0] = v0 ? acc[0] * slog2 : -INFINITY;
    s[1] = v0 ? acc[1] * slog2 : -INFINITY;
    s[2] = v1 ? acc[2] * slog2 : -INFINITY;
    s[3] = v1 ? acc[3] * slog2 : -INFINITY;
    // ---- online softmax over the warp's tokens (columns 2t, 2t+1)
    float x0 = fmaxf(s[0], s[2]), x1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
      x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
    }
    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
    const float ms0 = n0 == -INFINITY ? 0.f : n0, ms1 = n1 == -INFINITY ? 0.f : n1;
    const float sc0 = fast_exp2(m0 - ms0), sc1 = fast_exp2(m1 - ms1);
    m0 = n0; m1 = n1;
    l0 *= sc0; l1 *= sc1;
#pragma unroll
    for (int i = 0; i < KT; ++i) { o[i][0] *= sc0; o[i][1] *= sc1; o[i][2] *= sc0; o[i][3] *= sc1; }
    float p[4];
    p[0] = gv0 ? fast_exp2(s[0] - ms0) : 0.f;
    p[1] = gv1 ? fast_exp2(s[1] - ms1) : 0.f;
    p[2] = gv0 ? fast_exp2(s[2] - ms0) : 0.f;
    p[3] = gv1 ? fast_exp2(s[3] - ms1) : 0.f;
    l0 += p[0] + p[2];
    l1 += p[1] + p[3];
    // p (C fragment: rows = tokens) -> B fragments (k = tokens, n = group), hi + lo
    uint32_t h01, o01, h23, o23;
    split_half2(p[0], p[1], h01, o01);
    split_half2(p[2], p[3], h23, o23);
    const uint32_t bh0 = movtrans(h01), bl0 = movtrans(o01), bh1 = movtrans(h23), bl1 = movtrans(o23);
    // ---- o += V^T p: V^T fragment matrices are the transposed (tokens 0-7 | 8-15) x (d lo | hi) blocks
    {
      const int row = 16 * warp + (mi >> 1) * 8 + mr;
#pragma unroll
      for (int md = 0; md < KT; ++md) {
        const uint4 v = ldsm_x4_trans(vb + swz<D>(row, 2 * md + (mi & 1)));
        mma16816(o[md], v.x, v.y, v.z, v.w, bh0, bh1);
        mma16816(o[md], v.x, v.y, v.z, v.w, bl0, bl1);
      }
    }
    __syncthreads();  // the stage is refilled by a later issue
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- merge the four warps (pipeline buffers reused): stats [4][4][8], o [4][D][8]
  float* st = reinterpret_cast<float*>(smem);
  float* ow = st + 128;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
  if (lane < 4) {
    st[warp * 32 + 2 * t] = m0; st[warp * 32 + 2 * t + 1] = m1;
    st[warp * 32 + 8 + 2 * t] = l0; st[warp * 32 + 8 + 2 * t + 1] = l1;
  }
#pragma unroll
  for (int md = 0; md < KT; ++md) {
    float* o0 = ow + ((size_t)warp * D + md * 16 + gq) * 8 + 2 * t;
    o0[0] = o[md][0]; o0[1] = o[md][1]; o0[64] = o[md][2]; o0[65] = o[md][3];
  }
  __syncthreads();
  float* rec = a.partials + (size_t)blockIdx.x * (16 + 8 * D);
  for (int e = threadIdx.x; e < 8 * D + 8; e += kDenseThreads) {
    const int g = e < 8 * D ? e / D : e - 8 * D;
    float M = -INFINITY;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) M = fmaxf(M, st[wi * 32 + g]);
    const float Ms = M == -INFINITY ? 0.f : M;
    if (e < 8 * D) {
      const int dd = e % D;
      float v = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) v += fast_exp2(st[wi * 32 + g] - Ms) * ow[((size_t)wi * D + dd) * 8 + g];
      rec[16 + e] = v;
    } else {
      float L = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) L += fast_exp2(st[wi * 32 + g] - Ms) * st[wi * 32 + 8 + g];
      rec[g] = M;
      rec[8 + g] = L;
    }
  }
}

struct DensePlan {
  int chunk, nchunk;
  size_t off_partials, ws_bytes;
};

DensePlan plan_dense(int batch, int n_kv_heads, int d, int T) {
  DensePlan P;
  const int units = batch * n_kv_heads;
  const int max_chunks = (T + kDenseTile - 1) / kDenseTile;
  const int items = kDenseWaves * 2 * sm_count();
  int n = (items + units - 1) / units;
  n = n < 1 ? 1 : (n > max_chunks ? max_chunks : n);
  P.chunk = ((T + n - 1) / n + kDenseTile - 1) / kDenseTile * kDenseTile;
  P.nchunk = (T + P.chunk - 1) / P.chunk;
  P.off_partials = kWsHeader;
  P.ws_bytes = P.off_partials + (size_t)units * P.nchunk * (16 + 8 * d) * 4;
  return P;
}

template <int D>
cudaError_t launch_dense_d(const DenseArgs& a, int units, cudaStream_t s) {
  const size_t smem = (size_t)kDenseStages * 2 * kDenseTile * D * 2;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(dense_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  dense_kernel<D><<<units * a.nchunk, kDenseThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t dense_ws_bytes(int batch, int n_q_heads, int n_kv_heads, int d, int T) {
  (void)n_q_heads;
  return plan_dense(batch, n_kv_heads, d, T).ws_bytes;
}

cudaError_t launch_dense(int batch, int n_q_heads, int n_kv_heads, int d, int T, const __half* q, const __half* K,
                         const __half* V, float* out, float* lse, uint8_t* ws, uint32_t* err, cudaStream_t s) {
  (void)err;
  const DensePlan P = plan_dense(batch, n_kv_heads, d, T);
  DenseArgs a;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.G = n_q_heads / n_kv_heads;
  a.T = T;
  a.chunk = P.chunk;
  a.nchunk = P.nchunk;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  a.q = q;
  a.K = K;
  a.V = V;
  a.partials = reinterpret_cast<float*>(ws + P.off_partials);
  const int units = batch * n_kv_heads;
  cudaError_t e = d == 128 ? launch_dense_d<128>(a, units, s) : launch_dense_d<64>(a, units, s);
  if (e != cudaSuccess) return e;
  return launch_combine_records(units, P.nchunk, n_q_heads, n_kv_heads, d, a.partials, out, lse, s);
}

}  // namespace dkv
