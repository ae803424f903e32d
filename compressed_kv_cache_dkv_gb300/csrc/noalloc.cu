// dkv_decode_attend_noalloc: the decode call for callers that cannot
// allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocating
// routine) at decode time: runtimes that reserve a fixed memory pool at
// start-up and refuse further allocations, plugins or custom operators that
// run inside another framework and do not own its allocator, and serving
// loops where the device-wide synchronisation of cudaMalloc would stall
// other streams.  Such a caller can still pass its inputs and outputs; the
// scratch memory the decode needs (routed block indices and per-item
// partial results) comes from a fixed area compiled into this library.
//
// The area is a file-scope __device__ array of kNoAllocScratchBytes bytes.
// Every GPU that loads the library holds one copy of it until the process
// exits.  In host code the array's name is only a host-side stand-in, so its
// device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) on the first call made on that device, and that
// address is what the kernels receive.
#include <mutex>

#include "dkv_internal.cuh"

namespace dkv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch area on the current device (set-up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dkv

extern "C" int dkv_decode_attend_noalloc(const dkv_desc* d, const void* q, const void* cache, int32_t top_k,
                                         float* out, float* lse, int32_t* routed, void* stream) {
  if (!d) return DKV_ERR_ARG;
  if (top_k < 0) return DKV_ERR_ARG;
  dkv_desc c = *d;
  int st = dkv_layout(&c);
  if (st != DKV_OK) return st;
  const size_t need = dkv_decode_workspace_bytes(d, top_k);
  if (need == 0) return DKV_ERR_SHAPE;  // descriptor edited after dkv_layout()
  if (need > dkv::kNoAllocScratchBytes) return DKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (dkv::scratch_address(&scratch) != cudaSuccess) return DKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the header (device error word) and the tensor-core kernel's work-queue counters
  // right after it start every call at zero: a call that gave up on a bounded wait
  // can leave the counters set, and no caller can reach this area to clear them
  dkv::Layout L;
  dkv::make_layout(&c, &L);
  const size_t clear = dkv::plan_decode(L, c.n_q_heads, c.n_kv_heads, top_k).off_routed;
  if (cudaMemsetAsync(scratch, 0, clear, s) != cudaSuccess) return DKV_ERR_CUDA;
  return dkv_decode_attend(d, q, cache, top_k, out, lse, routed, scratch, dkv::kNoAllocScratchBytes, stream);
}
