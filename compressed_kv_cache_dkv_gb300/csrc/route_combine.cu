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
// o = sum acc_j 2^(m_j - m*) / l*, all in fp32.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

__global__ void __launch_bounds__(256) route_kernel(Layout L, int G, int Hq, int Hkv, int K_eff, float cq,
                                                    const __half* __restrict__ q, const uint8_t* __restrict__ cache,
                                                    int32_t* __restrict__ routed, int32_t* __restrict__ routed_out) {
  extern __shared__ float sm[];
  const int d = L.d, NB = L.NB;
  float* qbar = sm;               // [d]
  float* bounds = sm + d;         // [NB]
  int* sel = reinterpret_cast<int*>(bounds + NB);  // [NB]
  const int u = blockIdx.x;
  const int b = u / Hkv, h = u % Hkv;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
  for (int j = tid; j < d; j += nt) {
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += __half2float(q[((size_t)b * Hq + (size_t)h * G + g) * d + j]);
    qbar[j] = s * cq;  // cq = c / G
  }
  __syncthreads();
  const __half* router = reinterpret_cast<const __half*>(cache + (uint64_t)u * L.unit_stride + L.off_router);
  for (int blk = warp; blk < NB; blk += nw) {
    const __half* kmn = router + (size_t)blk * 2 * d;
    const __half* kmx = kmn + d;
    float acc = 0.f;
    for (int j = lane; j < d; j += 32) {
      float qj = qbar[j];
      acc += fmaxf(qj * __half2float(kmx[j]), qj * __half2float(kmn[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) bounds[blk] = isnan(acc) ? -INFINITY : acc;
  }
  __syncthreads();
  for (int i = tid; i < NB; i += nt) {
    int s = 1;
    if (K_eff < NB) {
      const float bi = bounds[i];
      int rank = 0;
      for (int j = 0; j < NB; ++j) {
        const float bj = bounds[j];
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
}

__global__ void __launch_bounds__(128) combine_kernel(int n_items, int G, int Hq, int Hkv, int d,
                                                      const float* __restrict__ partials, float* __restrict__ out,
                                                      float* __restrict__ lse) {
  const int jq = blockIdx.x, b = blockIdx.y;
  const int u = b * Hkv + jq / G, g = jq % G;
  const size_t rec = 16 + 8 * (size_t)d;
  const float* p = partials + (size_t)u * n_items * rec;
  float mstar = -INFINITY;
  for (int i = 0; i < n_items; ++i) mstar = fmaxf(mstar, p[i * rec + g]);
  const float ms = mstar == -INFINITY ? 0.f : mstar;
  float lstar = 0.f;
  for (int i = 0; i < n_items; ++i) lstar += p[i * rec + 8 + g] * exp2f(p[i * rec + g] - ms);
  const float inv = 1.f / lstar;
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < n_items; ++i) acc += p[i * rec + 16 + g * d + j] * exp2f(p[i * rec + g] - ms);
    out[((size_t)b * Hq + jq) * d + j] = acc * inv;
  }
  if (lse && threadIdx.x == 0) lse[(size_t)b * Hq + jq] = (ms + log2f(lstar)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t launch_route(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                         const uint8_t* cache, int32_t* routed, int32_t* routed_out, cudaStream_t s) {
  const int G = n_q_heads / n_kv_heads;
  const float cq = 1.f / (sqrtf((float)L.d) * (float)G);
  const size_t smem = (size_t)L.d * 4 + (size_t)L.NB * 8;
  static size_t configured = 48 * 1024;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  route_kernel<<<L.units, 256, smem, s>>>(L, G, n_q_heads, n_kv_heads, P.K_eff, cq, q, cache, routed, routed_out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Layout& L, const DecodePlan& P, int batch, int n_q_heads, int n_kv_heads,
                           const float* partials, float* out, float* lse, cudaStream_t s) {
  dim3 grid(n_q_heads, batch);
  combine_kernel<<<grid, 128, 0, s>>>(P.n_items, n_q_heads / n_kv_heads, n_q_heads, n_kv_heads, L.d, partials, out,
                                      lse);
  return cudaGetLastError();
}

}  // namespace dkv
