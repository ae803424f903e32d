// Streaming append of the DKV cache ([DKV-Z]; Differential-KV README, "Core
// Architecture & Paper Overview", items 1-4, applied as tokens arrive).
//
// New tokens go into the exact recency window.  When the window has no free
// slot, its oldest 256 tokens are compressed into the next block with the
// same compressor as a whole-layer compression (anchor, joint K|V truncated
// SVD, residual rows, router min / max), and the window slides down by 256
// tokens.  The window stays contiguous from token 0, so the decode kernels
// read it unchanged.  Default (fragment) layout only: its window is made of
// 16-token groups whose byte image does not depend on the window's length,
// so sliding by 256 tokens (16 groups) is a plain move of whole groups.
#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kMoveThreads = 1024;
constexpr int kMoveVec = 8;  // 16-byte vectors per thread and round

// window tokens [0, 256) of every unit -> plain K, V [units][256][d]
__global__ void extract_kernel(Layout L, const uint8_t* __restrict__ cache, __half* __restrict__ K,
                               __half* __restrict__ V) {
  const int u = blockIdx.x;
  const uint8_t* win = cache + (uint64_t)u * L.unit_stride + L.off_window;
  __half* Ku = K + (size_t)u * 256 * L.d;
  __half* Vu = V + (size_t)u * 256 * L.d;
  for (int e = threadIdx.x; e < 256 * L.d; e += blockDim.x) {
    const int t = e / L.d, j = e % L.d;
    Ku[e] = *reinterpret_cast<const __half*>(win + win_k_off(L, t, j));
    Vu[e] = *reinterpret_cast<const __half*>(win + win_v_off(L, t, j));
  }
}

// Slide every unit's window down by 256 tokens (16 groups of 64 d bytes):
// groups [16, n_groups) move to [0, n_groups - 16), the freed top 16 groups
// are zeroed.  Rounds of 16 groups run in increasing order, so a round only
// overwrites groups the previous round has already read.
__global__ void __launch_bounds__(kMoveThreads) slide_kernel(Layout L, uint8_t* __restrict__ cache, int n_groups) {
  const int u = blockIdx.x;
  uint4* win = reinterpret_cast<uint4*>(cache + (uint64_t)u * L.unit_stride + L.off_window);
  const int gvec = 4 * L.d;              // 16-byte vectors per 16-token group (64 d bytes)
  const int shift = 16 * gvec;           // 256 tokens
  const int total = n_groups * gvec;     // vectors of the old window
  for (int base = shift; base < total; base += shift) {
    uint4 v[kMoveVec];
#pragma unroll
    for (int i = 0; i < kMoveVec; ++i) {
      const int e = base + i * kMoveThreads + threadIdx.x;
      if (i * kMoveThreads < shift && e < total && e < base + shift) v[i] = win[e];
    }
#pragma unroll
    for (int i = 0; i < kMoveVec; ++i) {
      const int e = base + i * kMoveThreads + threadIdx.x;
      if (i * kMoveThreads < shift && e < total && e < base + shift) win[e - shift] = v[i];
    }
    __syncthreads();
  }
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int e = total - shift + (int)threadIdx.x; e < total; e += kMoveThreads) win[e] = z;
}

// new tokens [i0, i0 + take) of K_new, V_new [units][n_new][d] -> window slots [w0, w0 + take)
__global__ void write_kernel(Layout L, const __half* __restrict__ Kn, const __half* __restrict__ Vn, int n_new,
                             int i0, int take, int w0, uint8_t* __restrict__ cache) {
  const int u = blockIdx.y;
  uint8_t* win = cache + (uint64_t)u * L.unit_stride + L.off_window;
  const __half* Ku = Kn + ((size_t)u * n_new + i0) * L.d;
  const __half* Vu = Vn + ((size_t)u * n_new + i0) * L.d;
  const int n = take * L.d;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
    const int t = e / L.d, j = e % L.d;
    *reinterpret_cast<__half*>(win + win_k_off(L, w0 + t, j)) = Ku[e];
    *reinterpret_cast<__half*>(win + win_v_off(L, w0 + t, j)) = Vu[e];
  }
}

}  // namespace

size_t append_ws_bytes(const Layout& L) { return kWsHeader + 2ull * L.units * 256 * L.d * sizeof(__half); }

cudaError_t launch_append_compress(const Layout& L, uint8_t* cache, uint8_t* ws, uint32_t* err, cudaStream_t s) {
  // L describes the window before the slide: L.NB is the block the oldest 256 tokens become
  __half* K = reinterpret_cast<__half*>(ws + kWsHeader);
  __half* V = K + (size_t)L.units * 256 * L.d;
  extract_kernel<<<L.units, 256, 0, s>>>(L, cache, K, V);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_compress_blocks(L, K, V, 256, L.NB, 1, cache, err, s);
  if (e != cudaSuccess) return e;
  slide_kernel<<<L.units, kMoveThreads, 0, s>>>(L, cache, L.W16 / 16);
  return cudaGetLastError();
}

cudaError_t launch_append_write(const Layout& L, const __half* Kn, const __half* Vn, int n_new, int i0, int take,
                                int w0, uint8_t* cache, cudaStream_t s) {
  // L.W16 must cover w0 + take (every group the tokens land in holds 16 slots)
  const int n = take * L.d;
  dim3 grid((unsigned)((n + 255) / 256 < 64 ? (n + 255) / 256 : 64), (unsigned)L.units);
  write_kernel<<<grid, 256, 0, s>>>(L, Kn, Vn, n_new, i0, take, w0, cache);
  return cudaGetLastError();
}

}  // namespace dkv
