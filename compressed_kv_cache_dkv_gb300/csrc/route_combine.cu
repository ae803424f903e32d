// Block router and split-LSE combine of the DKV decode path.
//
// route: per unit, the group-mean query qbar = (1/G) sum_g c q_g
// (DKV_CB_GQA_ROUTE head averaging, Differential-KV README section "Key
// Environment Knobs") scores every block by the upper bound of qbar . k over
// the block's key box, sum_j max(qbar_j kmax_bj, qbar_j kmin_bj) (the per-block
// "Key Min/Max ... Decode router bounds" of the README's per-block memory
// table), and keeps the top K (DKV_TOPK_BLOCKS) by (score desc, index asc).
// The selected indices are written in ascending order when the caller asks for
// them; otherwise slot k of the attention grid's list holds the block of rank k
// (the attention result does not depend on the order of its blocks).
//
// combine: the flash-style log-sum-exp merge of every partial of a unit
// ("Flash-Style LSE Combine", README section "Core Architecture & Paper
// Overview"): m* = max m_j, l* = sum l_j 2^(m_j - m*),
// o = sum acc_j 2^(m_j - m*) / l*, all in fp32, in a fixed order (deterministic).
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kRouteCluster = 8;    // CTAs per unit (one thread-block cluster)
constexpr int kRouteThreads = 256;
constexpr int kRouteInFlight = 2;   // router rows in flight per lane (kmin and kmax pieces each)
constexpr int kRouteRounds = 2;     // ranking rounds (one at up to 2048 blocks over 8 CTAs of 256 threads)

// Order-preserving integer image of a bound: a < b as floats iff key(a) < key(b)
// as int32, equal floats give equal keys (-0 is taken as +0; NaN is ranked as
// -inf).  key - 1 never overflows (key(-inf) is far above INT_MIN).
__device__ inline int bound_key(float v) {
  if (isnan(v)) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const int u = __float_as_int(v);
  return u >= 0 ? u : u ^ 0x7fffffff;
}

// One cluster of kRouteCluster CTAs per unit; CTA c of the cluster owns blocks
// [c*per, (c+1)*per).  Each CTA loads its blocks' router rows ([kmin | kmax],
// 4d bytes per block), bounds them, and stores every bound into all CTAs of the
// cluster (distributed shared memory).  After a cluster barrier each CTA ranks
// its own blocks against all NB bounds (score desc, index asc), and the
// selected counts are exchanged once more so each CTA knows where its blocks
// go in the ascending output.  Without a caller's copy the rank itself is the
// slot: no second exchange, and every CTA is done after its own ranking.
//
// max(q kmax, q kmin) equals q kmax for q >= 0 and q kmin for q < 0 (rounding
// is monotone), so every channel costs one select and one FMA.
// F32: an un-rotated pool's fp32 router rows (8d bytes a block), 4 channels a piece.
template <bool F32>
__global__ void __cluster_dims__(kRouteCluster, 1, 1) __launch_bounds__(kRouteThreads)
    route_kernel(Layout L, int G, int Hq, int Hkv, int K_eff, float cq, const __half* __restrict__ q,
                 const uint8_t* __restrict__ cache, int32_t* __restrict__ routed, int32_t* __restrict__ routed_out) {
  extern __shared__ int4 key4[];  // bound keys of all NB blocks of the unit, padded to 4 with key(-inf)
  __shared__ float qbar[128];
  __shared__ int cnt[kRouteCluster];
  __shared__ int wsum[kRouteRounds * (kRouteThreads / 32)];
  const int d = L.d, NB = L.NB;
  const uint32_t crank = cluster_ctarank();
  const int u = blockIdx.x / kRouteCluster;
  const int b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nw = kRouteThreads / 32;
  cluster_arrive_relaxed();  // this CTA has started (matched by the wait before the first peer store)
  griddep_launch();          // the attention grid may start its window work now; its block work waits for this grid
  const uint8_t* router = cache + (uint64_t)u * L.unit_stride + L.off_router;
  const int per = (NB + kRouteCluster - 1) / kRouteCluster;
  const int b0 = min(NB, (int)crank * per), b1 = min(NB, b0 + per);
  constexpr int cpp = F32 ? 4 : 8;       // channels per 16-byte piece
  const int rb = (F32 ? 8 : 4) * d;      // router row bytes
  const int hp = d / cpp;                // 16-byte pieces per half row (kmin or kmax)
  const int bpw = 32 / hp;               // blocks per warp and pass
  const int bpp = bpw * nw;              // blocks per pass
  const int piece = lane % hp;
  const int lb = warp * bpw + lane / hp;
  const int n_pass = (b1 - b0 + bpp - 1) / bpp;
  uint4 mn[kRouteInFlight], mx[kRouteInFlight];
#pragma unroll
  for (int i = 0; i < kRouteInFlight; ++i) {
    const int blk = b0 + i * bpp + lb;
    mn[i] = mx[i] = make_uint4(0u, 0u, 0u, 0u);
    if (blk < b1) {
      const uint8_t* row = router + (size_t)blk * rb + (size_t)piece * 16;
      mn[i] = *reinterpret_cast<const uint4*>(row);
      mx[i] = *reinterpret_cast<const uint4*>(row + rb / 2);
    }
  }
  for (int j = tid; j < d; j += kRouteThreads) {
    float x[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)  // independent loads, summed in a fixed order below
      x[g] = g < G ? __half2float(q[((size_t)b * Hq + (size_t)h * G + g) * d + j]) : 0.f;
    float t = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) t += x[g];
    qbar[j] = t * cq;  // cq = c / G
  }
  int* key = reinterpret_cast<int*>(key4);
  const int NB4 = (NB + 3) / 4;
  if (tid < 4 * NB4 - NB) key[NB + tid] = bound_key(-INFINITY);  // padding never outranks a block
  __syncthreads();
  float qv[8];
  uint32_t selm[4];  // per half: all ones where q_j >= 0 (take kmax), zero where q_j < 0 (take kmin)
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = e < cpp ? qbar[cpp * piece + e] : 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) selm[w] = (qv[2 * w] >= 0.f ? 0x0000ffffu : 0u) | (qv[2 * w + 1] >= 0.f ? 0xffff0000u : 0u);
  cluster_wait();  // every CTA of the cluster has started: peer shared memory may be written
  for (int p0 = 0; p0 < n_pass; p0 += kRouteInFlight) {
    if (p0 > 0) {
#pragma unroll
      for (int i = 0; i < kRouteInFlight; ++i) {
        const int blk = b0 + (p0 + i) * bpp + lb;
        mn[i] = mx[i] = make_uint4(0u, 0u, 0u, 0u);
        if (blk < b1) {
          const uint8_t* row = router + (size_t)blk * rb + (size_t)piece * 16;
          mn[i] = *reinterpret_cast<const uint4*>(row);
          mx[i] = *reinterpret_cast<const uint4*>(row + rb / 2);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRouteInFlight; ++i) {
      const int blk = b0 + (p0 + i) * bpp + lb;
      const uint32_t wn[4] = {mn[i].x, mn[i].y, mn[i].z, mn[i].w};
      const uint32_t wx[4] = {mx[i].x, mx[i].y, mx[i].z, mx[i].w};
      float acc = 0.f;
      if constexpr (F32) {
#pragma unroll
        for (int w = 0; w < 4; ++w) acc = fmaf(qv[w], __uint_as_float(qv[w] >= 0.f ? wx[w] : wn[w]), acc);
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t v = (wx[w] & selm[w]) | (wn[w] & ~selm[w]);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
          acc = fmaf(qv[2 * w], f.x, acc);
          acc = fmaf(qv[2 * w + 1], f.y, acc);
        }
      }
      for (int o = hp >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (blk < b1 && piece < kRouteCluster) st_cluster_s32(key + blk, (uint32_t)piece, bound_key(acc));
    }
  }
  cluster_sync();  // all NB bounds are in every CTA
  // rank own blocks: tpb threads share one block's comparisons (tpb = 1 at the
  // 2048-block limit: 256 blocks per CTA); a CTA with more blocks than threads
  // would rank them in rounds, which the block limit never needs
  const int n_own = b1 - b0;
  int tpb = 32;
  while (tpb > 1 && tpb * n_own > kRouteThreads) tpb >>= 1;
  const int per_round = kRouteThreads / tpb;
  const int rounds = (n_own + per_round - 1) / per_round;  // at most kRouteRounds (NB <= 2048)
  const int sub = tid % tpb;
  bool sel[kRouteRounds];
  int rk[kRouteRounds];
  unsigned bal[kRouteRounds];
#pragma unroll
  for (int r = 0; r < kRouteRounds; ++r) {
    sel[r] = false;
    rk[r] = 0;
    bal[r] = 0u;
    if (r < rounds) {  // uniform over the CTA
      const int own = r * per_round + tid / tpb;
      const int i = b0 + own;
      const bool mine = own < n_own;
      int rank = 0;
      if (mine && K_eff < NB) {
        // rank of i = #{j < i: key_j >= key_i} + #{j > i: key_j > key_i}: one threshold per
        // group of four (key_i - 1 below i's group, key_i from it on), and the ties
        // inside i's own group below i added once
        const int ki = key[i], i4 = i >> 2;
        int ra = 0, rb = 0;
#pragma unroll 2
        for (int j4 = sub; j4 < NB4; j4 += tpb) {
          const int4 kj = key4[j4];
          const int th = j4 < i4 ? ki - 1 : ki;
          ra += (kj.x > th) + (kj.y > th);
          rb += (kj.z > th) + (kj.w > th);
        }
        rank = ra + rb;
        if (sub == 0)
          for (int e = i & ~3; e < i; ++e) rank += key[e] == ki;
      }
      for (int o = tpb >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
      rk[r] = K_eff < NB ? rank : i;  // every block routed: block i in slot i
      sel[r] = mine && sub == 0 && rank < K_eff;
      bal[r] = __ballot_sync(0xffffffffu, sel[r]);
    }
    if (lane == 0) wsum[r * nw + warp] = __popc(bal[r]);
  }
  if (routed_out == nullptr) {  // slot = rank; no peer access follows the first cluster barrier
#pragma unroll
    for (int r = 0; r < kRouteRounds; ++r)
      if (sel[r]) routed[(size_t)u * K_eff + rk[r]] = b0 + r * per_round + tid / tpb;
    return;
  }
  __syncthreads();
  int total = 0;  // selected blocks of this CTA
#pragma unroll
  for (int w = 0; w < kRouteRounds * nw; ++w) total += wsum[w];
  if (tid < kRouteCluster) st_cluster_s32(&cnt[crank], (uint32_t)tid, total);
  cluster_sync();  // every CTA's count is everywhere; no peer access follows
  int offset = 0;
  for (int c = 0; c < (int)crank; ++c) offset += cnt[c];
#pragma unroll
  for (int r = 0; r < kRouteRounds; ++r) {
    if (sel[r]) {
      int before = 0;  // selected blocks of this CTA below this one: earlier rounds, lower warps
      for (int w = 0; w < r * nw + warp; ++w) before += wsum[w];
      const int i = b0 + r * per_round + tid / tpb;
      const int pos = offset + before + __popc(bal[r] & ((1u << lane) - 1u));
      routed[(size_t)u * K_eff + pos] = i;
      if (routed_out) routed_out[(size_t)u * K_eff + pos] = i;
    }
  }
}

constexpr int kCombineThreads = 256;
constexpr int kCombinePrefetch = 8;  // records a thread loads before the reduction: 64 per pass at d = 128

// One CTA per (unit, query head).  Partial records of all items are merged with
// weights exp2(m_i - m*) / l* (m*, l* the merged maximum and normaliser);
// the first kCombinePrefetch records of every thread are loaded before the
// statistics are reduced, so both round trips to memory overlap.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(int n_items, int G, int Hq, int Hkv, int d,
                                                                  const float* __restrict__ partials,
                                                                  float* __restrict__ out, float* __restrict__ lse) {
  griddep_wait();
  extern __shared__ float csm[];  // [n_items] maxima, [n_items] normalisers
  __shared__ float4 red[kCombineThreads];
  __shared__ float wred[kCombineThreads / 32];
  const int u = blockIdx.x, g = blockIdx.y, b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t rs = 16 + 8 * (size_t)d;
  const float* p = partials + (size_t)u * n_items * rs;
  const size_t qrow = (size_t)b * Hq + (size_t)h * G + g;
  const int n4 = d / 4, n_sub = kCombineThreads / n4;
  const int e = tid % n4, sub = tid / n4;
  const float* src = p + 16 + (size_t)g * d + 4 * e;
  float4 pre[kCombinePrefetch];
#pragma unroll
  for (int x = 0; x < kCombinePrefetch; ++x) {
    const int i = sub + x * n_sub;
    pre[x] = i < n_items ? __ldg(reinterpret_cast<const float4*>(src + i * rs)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float* mi = csm;
  float* li = csm + n_items;
  float m = -INFINITY;
  for (int i = tid; i < n_items; i += kCombineThreads) {
    const float mv = __ldg(p + i * rs + g);
    mi[i] = mv;
    li[i] = __ldg(p + i * rs + 8 + g);
    m = fmaxf(m, mv);
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wred[warp] = m;
  __syncthreads();
  m = wred[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) m = fmaxf(m, wred[w]);
  const float ms = m == -INFINITY ? 0.f : m;
  float l = 0.f;
  for (int i = tid; i < n_items; i += kCombineThreads) l += li[i] * fast_exp2(mi[i] - ms);
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  __syncthreads();  // every thread has read wred
  if (lane == 0) wred[warp] = l;
  __syncthreads();
  l = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) l += wred[w];
  const float linv = 1.f / l;
  if (lse && tid == 0) lse[qrow] = (ms + log2f(l)) * 0.6931471805599453f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int x = 0; x < kCombinePrefetch; ++x) {
    const int i = sub + x * n_sub;
    if (i < n_items) {
      const float wx = fast_exp2(mi[i] - ms) * linv;
      acc.x = fmaf(wx, pre[x].x, acc.x); acc.y = fmaf(wx, pre[x].y, acc.y);
      acc.z = fmaf(wx, pre[x].z, acc.z); acc.w = fmaf(wx, pre[x].w, acc.w);
    }
  }
  for (int i0 = sub + kCombinePrefetch * n_sub; i0 < n_items; i0 += kCombinePrefetch * n_sub) {
#pragma unroll
    for (int x = 0; x < kCombinePrefetch; ++x) {
      const int i = i0 + x * n_sub;
      pre[x] = i < n_items ? __ldg(reinterpret_cast<const float4*>(src + i * rs)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int x = 0; x < kCombinePrefetch; ++x) {
      const int i = i0 + x * n_sub;
      if (i < n_items) {
        const float wx = fast_exp2(mi[i] - ms) * linv;
        acc.x = fmaf(wx, pre[x].x, acc.x); acc.y = fmaf(wx, pre[x].y, acc.y);
        acc.z = fmaf(wx, pre[x].z, acc.z); acc.w = fmaf(wx, pre[x].w, acc.w);
      }
    }
  }
  red[tid] = acc;
  __syncthreads();
  if (tid < n4) {
    float4 t = red[tid];
    for (int s2 = 1; s2 < n_sub; ++s2) {
      const float4 v = red[s2 * n4 + tid];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    *reinterpret_cast<float4*>(out + qrow * d + 4 * tid) = t;
  }
}

}  // namespace

cudaError_t launch_route(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                         const uint8_t* cache, uint8_t* ws, int32_t* routed_out, cudaStream_t s) {
  const int G = n_q_heads / n_kv_heads;
  const float cq = 1.f / (sqrtf((float)L.d) * (float)G);
  const size_t smem = ((size_t)L.NB + 3) / 4 * 16;  // at most 2048 blocks: 8 KB
  // an SM running a router CTA keeps room for attention CTAs of 108 KB
  const auto kern = L.rope ? route_kernel<true> : route_kernel<false>;
  const cudaError_t e = ensure_max_carveout(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  kern<<<L.units * kRouteCluster, kRouteThreads, smem, s>>>(L, G, n_q_heads, n_kv_heads, P.K_eff, cq, q, cache,
                                                            reinterpret_cast<int32_t*>(ws + P.off_routed), routed_out);
  return cudaGetLastError();
}

cudaError_t launch_combine_records(int units, int n_items, int n_q_heads, int n_kv_heads, int d,
                                   const float* partials, float* out, float* lse, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  const size_t smem = (size_t)n_items * 8;  // at most (2048 + 256) items: 18 KB
  cfg.gridDim = dim3(units, n_q_heads / n_kv_heads);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, n_items, n_q_heads / n_kv_heads, n_q_heads, n_kv_heads, d,
                            partials, out, lse);
}

cudaError_t launch_combine(const Layout& L, const DecodePlan& P, int batch, int n_q_heads, int n_kv_heads,
                           const float* partials, float* out, float* lse, cudaStream_t s) {
  (void)batch;
  return launch_combine_records(L.units, P.n_items, n_q_heads, n_kv_heads, L.d, partials, out, lse, s);
}

}  // namespace dkv
