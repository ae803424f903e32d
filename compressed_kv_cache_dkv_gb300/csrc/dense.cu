// Dense fp16 decode attention (the uncompressed reference) -- placeholder until the kernel lands.
#include "dkv_internal.cuh"

namespace dkv {
size_t dense_ws_bytes(int batch, int n_q_heads, int n_kv_heads, int d, int T) {
  (void)batch; (void)n_q_heads; (void)n_kv_heads; (void)d; (void)T; return kWsHeader;
}
cudaError_t launch_dense(int batch, int n_q_heads, int n_kv_heads, int d, int T, const __half* q, const __half* K,
                         const __half* V, float* out, float* lse, uint8_t* ws, uint32_t* err, cudaStream_t s) {
  (void)batch; (void)n_q_heads; (void)n_kv_heads; (void)d; (void)T; (void)q; (void)K; (void)V; (void)out;
  (void)lse; (void)ws; (void)err; (void)s;
  return cudaErrorNotSupported;
}
}  // namespace dkv
