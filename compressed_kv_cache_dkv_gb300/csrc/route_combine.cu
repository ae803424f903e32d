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

constexpr int kRouteThreads = 1024;
constexpr int kRouteInFlight = 6;  // router loads in flight per thread

// One CTA per unit.  The unit's router rows ([NB][kmin | kmax], 4d bytes per
// block) are requested before the group-mean query is formed, so the two
// memory round trips overlap; each block's bound is reduced over the lanes
// that hold its row, and the top K are ranked in shared memory by several
// threads per block.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(Layout L, int G, int Hq, int Hkv, int K_eff, float cq,
                                                               const __half* __restrict__ q,
                                                               const uint8_t* __restrict__ cache,
                                                               int32_t* __restrict__ routed,
                                                               int32_t* __restrict__ routed_out) {
  extern __shared__ float4 sc4[];  // bounds [NB rounded up to 4]
  __shared__ float qbar[128];
  __shared__ int wsum[kRouteThreads / 32 + 1];
  const int d = L.d, NB = L.NB;
  const int u = blockIdx.x;
  const int b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, nw = kRouteThreads / 32;
  griddep_launch();  // the attention grid may start its window work now; its block work waits for this grid
  const uint8_t* router = cache + (uint64_t)u * L.unit_stride + L.off_router;
  const int per_blk = d / 4;                  // 16-byte pieces per block (32 or 16): one warp covers 1 or 2 blocks
  const int blk_per_pass = (32 / per_blk) * nw;
  const int half_pcs = d / 8;                 // kmin pieces; the kmax partner is half_pcs lanes up
  const int q_in = lane % per_blk;
  const int blk_lane = warp * (32 / per_blk) + lane / per_blk;
  const int n_pass = (NB + blk_per_pass - 1) / blk_per_pass;
  uint4 v[kRouteInFlight];
#pragma unroll
  for (int i = 0; i < kRouteInFlight; ++i) {
    const int blk = i * blk_per_pass + blk_lane;
    v[i] = blk < NB ? *reinterpret_cast<const uint4*>(router + (size_t)blk * 4 * d + (size_t)q_in * 16)
                    : make_uint4(0u, 0u, 0u, 0u);
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
  float* sc = reinterpret_cast<float*>(sc4);
  const int NB4 = (NB + 3) / 4;
  if (tid >= NB && tid < 4 * NB4) sc[tid] = -INFINITY;  // padding never outranks a block
  __syncthreads();
  for (int p0 = 0; p0 < n_pass; p0 += kRouteInFlight) {
    if (p0 > 0) {
#pragma unroll
      for (int i = 0; i < kRouteInFlight; ++i) {
        const int blk = (p0 + i) * blk_per_pass + blk_lane;
        v[i] = blk < NB ? *reinterpret_cast<const uint4*>(router + (size_t)blk * 4 * d + (size_t)q_in * 16)
                        : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < kRouteInFlight; ++i) {
      const int blk = (p0 + i) * blk_per_pass + blk_lane;
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
      for (int o = per_blk >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (q_in == 0 && blk < NB) sc[blk] = isnan(acc) ? -INFINITY : acc;
    }
  }
  __syncthreads();
  // rank of block i = number of blocks ahead of it (score desc, index asc);
  // tpb threads share one block's comparisons
  int tpb = 32;
  while (tpb > 1 && tpb * NB > kRouteThreads) tpb >>= 1;
  const int per_round = kRouteThreads / tpb;
  const int sub = tid % tpb;
  for (int base = 0; base < NB; base += per_round) {
    const int i = base + tid / tpb;
    int rank = 0;
    if (i < NB && K_eff < NB) {
      const float bi = sc[i];
      for (int j4 = sub; j4 < NB4; j4 += tpb) {
        const float4 bj = sc4[j4];
        const int j = 4 * j4;
        rank += (bj.x > bi) || (bj.x == bi && j < i);
        rank += (bj.y > bi) || (bj.y == bi && j + 1 < i);
        rank += (bj.z > bi) || (bj.z == bi && j + 2 < i);
        rank += (bj.w > bi) || (bj.w == bi && j + 3 < i);
      }
    }
    for (int o = tpb >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    const bool sel = sub == 0 && i < NB && rank < K_eff;
    // ascending output position = number of routed blocks with a lower index
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
      const int c = lane < nw ? wsum[lane] : 0;
      int incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int run = base == 0 ? 0 : wsum[nw];
      __syncwarp();
      if (lane < nw) wsum[lane] = run + incl - c;
      if (lane == 31) wsum[nw] = run + incl;
    }
    __syncthreads();
    if (sel) {
      const int pos = wsum[warp] + __popc(bal & ((1u << lane) - 1u));
      routed[(size_t)u * K_eff + pos] = i;
      if (routed_out) routed_out[(size_t)u * K_eff + pos] = i;
    }
    __syncthreads();
  }
}

constexpr int kCombineThreads = 256;
constexpr int kCombinePrefetch = 4;

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
  route_kernel<<<L.units, kRouteThreads, smem, s>>>(L, G, n_q_heads, n_kv_heads, P.K_eff, cq, q, cache,
                                                    reinterpret_cast<int32_t*>(ws + P.off_routed), routed_out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Layout& L, const DecodePlan& P, int batch, int n_q_heads, int n_kv_heads,
                           const float* partials, float* out, float* lse, cudaStream_t s) {
  (void)batch;
  cudaLaunchConfig_t cfg = {};
  const size_t smem = (size_t)P.n_items * 8;  // at most (2048 + 256) items: 18 KB
  cfg.gridDim = dim3(L.units, n_q_heads / n_kv_heads);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = smem;
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
