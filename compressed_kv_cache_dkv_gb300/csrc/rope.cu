// RoPE tables of an un-rotated pool ([README Knobs] DKV_ROTATED_POOL=0 of the
// Differential-KV README: keys are stored before RoPE and rotated to their
// absolute positions at read).
//
// With h = rope / 2 and theta_j = base^(-2j / rope) the cache ends with
//   page table   [pages][h]  (cos, sin)(256 p theta_j)
//   in-page table [256][h]   (cos, sin)(i theta_j)
// as fp32 pairs, each entry from one fp64 product and fp64 cos / sin, so that
// the fp32 composition of a page entry and an in-page entry (rope_cs) carries
// the angle of any position up to the capacities with an error of a few fp32
// roundings, whatever the position.  Setup path, not timed.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(Layout L, uint8_t* cache) {
  const int h = L.rope / 2, rows = L.rope_pages + 256;
  float2* tab = reinterpret_cast<float2*>(cache + L.off_rope);
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < rows * h; e += gridDim.x * blockDim.x) {
    const int row = e / h, j = e % h;
    const double theta = pow((double)L.rope_base, -2.0 * (double)j / (double)L.rope);
    const double pos = row < L.rope_pages ? 256.0 * (double)row : (double)(row - L.rope_pages);
    double sn, cs;
    sincos(pos * theta, &sn, &cs);
    tab[e] = make_float2((float)cs, (float)sn);
  }
}

}  // namespace

cudaError_t launch_rope_tables(const Layout& L, uint8_t* cache, cudaStream_t s) {
  if (!L.rope) return cudaSuccess;
  const int n = (L.rope_pages + 256) * (L.rope / 2);
  const int grid = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  rope_table_kernel<<<grid, 256, 0, s>>>(L, cache);
  return cudaGetLastError();
}

}  // namespace dkv
