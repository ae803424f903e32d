// Host side of libdkv: descriptor validation, layout, argument checks and the
// extern "C" entry points declared in include/dkv.h.  No kernel code here.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "dkv_internal.cuh"

namespace dkv {

// Kernel attributes are per device: one record per (kernel, device) of what was
// set on it, behind one lock (attribute calls happen at launch time only).
namespace {
std::mutex g_attr_mutex;
std::map<std::pair<const void*, int>, size_t> g_smem_limit;
std::map<std::pair<const void*, int>, bool> g_carveout;
}  // namespace

cudaError_t ensure_smem_limit(const void* func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  size_t& have = g_smem_limit[{func, dev}];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

cudaError_t ensure_max_carveout(const void* func) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  bool& done = g_carveout[{func, dev}];
  if (done) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done = true;
  return e;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 256-token pages of absolute positions an un-rotated pool can hold: every block
// and window slot of the capacities (block b's tokens on page b, the window after
// them)
static int rope_pages(const dkv_desc* d) {
  const int cap_b = d->block_capacity ? d->block_capacity : d->n_blocks;
  const int cap_w = d->window_capacity ? d->window_capacity : d->window;
  const int n = (cap_b * 256 + cap_w + 255) / 256;
  return n > 0 ? n : 1;
}

bool make_layout(const dkv_desc* d, Layout* L) {
  if (!d || !L || d->total_bytes == 0) return false;
  L->d = d->head_dim;
  L->r = d->rank;
  L->r8 = d->rank_pad;
  L->R = d->n_residual;
  L->R8 = d->res_pad;
  L->W = d->window;
  L->W16 = d->window_pad;
  L->NB = d->n_blocks;
  L->units = d->n_units;
  L->tc = d->layout == DKV_LAYOUT_TC ? 1 : 0;
  L->qbits = d->residual_bits;
  L->qgb = d->residual_bits ? (int)qgroup_bytes(d->head_dim, d->residual_bits) : 0;
  L->rope = d->rope_dims;
  L->rope_base = d->rope_base;
  L->rope_pages = d->rope_dims ? rope_pages(d) : 0;
  L->off_rope = d->off_rope;
  L->off_mask = d->blk_off_mask;
  L->off_vk = d->blk_off_vk;
  L->off_u = d->blk_off_u;
  L->off_res = d->blk_off_res;
  L->off_vv = d->blk_off_vv;
  L->block_bytes = d->block_bytes;
  L->off_router = d->off_router;
  L->off_blocks = d->off_blocks;
  L->off_cold = d->off_cold;
  L->off_window = d->off_window;
  L->block_stride = d->block_stride;
  L->unit_stride = d->unit_stride;
  L->total = d->total_bytes;
  return true;
}

// Recompute the layout from the caller-set fields and check that the filled
// fields agree (a descriptor edited after dkv_layout() is rejected).
static int check_desc(const dkv_desc* d, Layout* L) {
  if (!d) return DKV_ERR_ARG;
  dkv_desc c;
  std::memcpy(&c, d, sizeof(c));
  int st = dkv_layout(&c);
  if (st != DKV_OK) return st;
  if (std::memcmp(&c, d, sizeof(c)) != 0) return DKV_ERR_SHAPE;
  make_layout(&c, L);
  return DKV_OK;
}

}  // namespace dkv

using namespace dkv;

extern "C" {

int dkv_version(void) { return DKV_VERSION; }

const char* dkv_status_string(int status) {
  switch (status) {
    case DKV_OK: return "ok";
    case DKV_ERR_ARG: return "invalid argument";
    case DKV_ERR_SHAPE: return "inconsistent shape";
    case DKV_ERR_ALIGN: return "pointer not 16-byte aligned";
    case DKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case DKV_ERR_CUDA: return "CUDA runtime error";
    case DKV_ERR_TIMEOUT: return "device wait timed out";
    case DKV_ERR_WORKSPACE: return "workspace missing or too small";
    case DKV_ERR_DEVICE: return "device error word set";
    default: return "unknown status";
  }
}

int dkv_layout(dkv_desc* d) {
  if (!d) return DKV_ERR_ARG;
  if (d->batch < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 || d->head_dim < 1 || d->n_blocks < 0 ||
      d->window < 0 || d->rank < 0 || d->n_residual < 0 || d->block_size < 1 || d->block_capacity < 0 ||
      d->window_capacity < 0)
    return DKV_ERR_ARG;
  if (d->layout != DKV_LAYOUT_FRAGMENT && d->layout != DKV_LAYOUT_TC) return DKV_ERR_ARG;
  if (d->residual_bits != 0 && d->residual_bits != 8 && d->residual_bits != 4) return DKV_ERR_ARG;
  if (d->rope_dims < 0 || d->rope_dims > d->head_dim || (d->rope_dims && !(d->rope_base > 1.f && d->rope_base < INFINITY)))
    return DKV_ERR_ARG;
  if (d->n_q_heads % d->n_kv_heads != 0) return DKV_ERR_SHAPE;
  const int cap_b = d->block_capacity ? d->block_capacity : d->n_blocks;
  const int cap_w = d->window_capacity ? d->window_capacity : d->window;
  if (d->n_blocks > cap_b || d->window > cap_w) return DKV_ERR_SHAPE;
  // nothing to attend, and no room for tokens to come
  if (d->n_blocks == 0 && d->window == 0 && cap_w == 0) return DKV_ERR_SHAPE;
  if (d->block_size != DKV_BLOCK_SIZE) return DKV_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return DKV_ERR_UNSUPPORTED;
  if (d->n_q_heads / d->n_kv_heads > 8) return DKV_ERR_UNSUPPORTED;
  if (d->rank > 128 || d->n_residual > 255) return DKV_ERR_UNSUPPORTED;
  // the router and the combine keep per-block / per-item values in shared memory
  if (cap_b > 2048 || cap_w > 65536) return DKV_ERR_UNSUPPORTED;
  const uint64_t dd = (uint64_t)d->head_dim;
  const int r8 = (d->rank + 7) / 8 * 8;
  const int rq = d->residual_bits;
  if (rq && d->layout == DKV_LAYOUT_TC) return DKV_ERR_UNSUPPORTED;
  // the un-rotated pool: RoPE pairs (j, j + rope_dims / 2) sit in k tiles 16 channels apart
  if (d->rope_dims && (d->rope_dims % 32 != 0 || d->layout != DKV_LAYOUT_FRAGMENT || rq || r8 > 64))
    return DKV_ERR_UNSUPPORTED;
  const int R8 = rq ? (d->n_residual + 15) / 16 * 16 : (d->n_residual + 7) / 8 * 8;
  const uint64_t res_bytes = rq ? (uint64_t)(R8 / 16) * qgroup_bytes(d->head_dim, rq) : 4ull * R8 * dd;
  const int W16 = (d->window + 15) / 16 * 16;
  d->rank_pad = r8;
  d->res_pad = R8;
  d->window_pad = W16;
  d->n_units = d->batch * d->n_kv_heads;
  if (d->layout == DKV_LAYOUT_TC) {
    if (!tc_layout(d->head_dim, r8, d->n_residual)) return DKV_ERR_UNSUPPORTED;
    // tensor-core layout: [a_k a_v][mask][V_K][U][V_V][K_res V_res] (same bytes, other order)
    d->blk_off_mask = 4 * dd;
    d->blk_off_vk = 4 * dd + 32;
    d->blk_off_u = d->blk_off_vk + 2ull * r8 * dd;
    d->blk_off_vv = d->blk_off_u + 2ull * 256 * r8;
    d->blk_off_res = d->blk_off_vv + 2ull * r8 * dd;
    d->block_bytes = d->blk_off_res + 4ull * R8 * dd;
  } else {
    d->blk_off_mask = 4 * dd;
    d->blk_off_vk = 4 * dd + 32;
    d->blk_off_u = d->blk_off_vk + 2ull * r8 * dd;
    d->blk_off_res = d->blk_off_u + 2ull * 256 * r8;
    d->blk_off_vv = d->blk_off_res + res_bytes;
    d->block_bytes = d->blk_off_vv + 2ull * r8 * dd;
  }
  d->block_stride = round_up(d->block_bytes, 128);
  // offsets follow the capacities, so they stay put while the live counts change
  const uint64_t nb = (uint64_t)cap_b;
  const uint64_t W16cap = (uint64_t)(cap_w + 15) / 16 * 16;
  d->off_router = 0;
  d->off_blocks = round_up(nb * (d->rope_dims ? 8 : 4) * dd, 128);  // fp32 boxes in an un-rotated pool
  d->off_cold = d->off_blocks + nb * d->block_stride;
  d->off_window = d->off_cold + round_up(nb * (uint64_t)R8 * 2, 128);
  d->unit_stride = round_up(d->off_window + W16cap * 4 * dd, 128);
  d->total_bytes = d->unit_stride * (uint64_t)d->n_units;
  d->off_rope = 0;
  if (d->rope_dims) {  // [pages][h] then [256][h] (cos, sin) fp32 pairs
    d->off_rope = d->total_bytes;
    d->total_bytes += (uint64_t)(rope_pages(d) + 256) * (uint64_t)(d->rope_dims / 2) * 8;
  }
  return DKV_OK;
}

size_t dkv_layout_bytes(dkv_desc* d) { return dkv_layout(d) == DKV_OK ? (size_t)d->total_bytes : 0; }

size_t dkv_compress_workspace_bytes(const dkv_desc* d) {
  Layout L;
  if (check_desc(d, &L) != DKV_OK) return 0;
  return compress_ws_bytes(L);
}

int dkv_compress_layout(const dkv_desc* d, const void* K, const void* V, void* cache, void* workspace,
                        size_t ws_bytes, void* stream) {
  Layout L;
  int st = check_desc(d, &L);
  if (st != DKV_OK) return st;
  if (!K || !V || !cache || !workspace) return DKV_ERR_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(cache) || !aligned16(workspace)) return DKV_ERR_ALIGN;
  if (ws_bytes < compress_ws_bytes(L)) return DKV_ERR_WORKSPACE;
  const int p_cap = L.d == 128 ? 64 : 128;
  if (L.r > p_cap) return DKV_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_compress(L, static_cast<const __half*>(K), static_cast<const __half*>(V),
                                  static_cast<uint8_t*>(cache), ws, reinterpret_cast<uint32_t*>(ws),
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_import_factors(const dkv_desc* d, const dkv_factors* f, void* cache, void* workspace, void* stream) {
  Layout L;
  int st = check_desc(d, &L);
  if (st != DKV_OK) return st;
  if (!f || !cache || !workspace) return DKV_ERR_ARG;
  if (!aligned16(cache) || !aligned16(workspace)) return DKV_ERR_ALIGN;
  if (L.NB > 0) {
    if (!f->a_k || !f->a_v || !f->kmin || !f->kmax) return DKV_ERR_ARG;
    if (L.r > 0 && (!f->U || !f->V_K || !f->V_V)) return DKV_ERR_ARG;
    if (L.R > 0 && (!f->res_pos || !f->K_res || !f->V_res)) return DKV_ERR_ARG;
  }
  if (L.W > 0 && (!f->win_K || !f->win_V)) return DKV_ERR_ARG;
  cudaError_t e = launch_pack(L, *f, static_cast<uint8_t*>(cache), static_cast<uint32_t*>(workspace),
                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

size_t dkv_append_workspace_bytes(const dkv_desc* d) {
  Layout L;
  if (check_desc(d, &L) != DKV_OK) return 0;
  return append_ws_bytes(L);
}

int dkv_append(dkv_desc* d, const void* K_new, const void* V_new, int32_t n_new, void* cache, void* workspace,
               size_t ws_bytes, void* stream) {
  Layout L;
  int st = check_desc(d, &L);
  if (st != DKV_OK) return st;
  if (n_new < 0) return DKV_ERR_ARG;
  if (n_new == 0) return DKV_OK;
  if (!K_new || !V_new || !cache || !workspace) return DKV_ERR_ARG;
  if (!aligned16(K_new) || !aligned16(V_new) || !aligned16(cache) || !aligned16(workspace)) return DKV_ERR_ALIGN;
  if (L.tc) return DKV_ERR_UNSUPPORTED;  // the tensor-core window's byte image depends on its length
  if (ws_bytes < append_ws_bytes(L)) return DKV_ERR_WORKSPACE;
  const int p_cap = L.d == 128 ? 64 : 128;  // the GPU compressor's rank limit
  const int cap_b = d->block_capacity ? d->block_capacity : d->n_blocks;
  const int cap_w = d->window_capacity ? d->window_capacity : d->window;
  // plan every step on the host first: nothing is launched unless the whole append fits
  {
    int nb = d->n_blocks, w = d->window, rem = n_new;
    while (rem > 0) {
      if (w == cap_w) {
        if (w < 256 || nb == cap_b || L.r > p_cap) return DKV_ERR_UNSUPPORTED;
        ++nb;
        w -= 256;
      }
      const int take = rem < cap_w - w ? rem : cap_w - w;
      w += take;
      rem -= take;
    }
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* cb = static_cast<uint8_t*>(cache);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int nb = d->n_blocks, w = d->window, i0 = 0;
  // an un-rotated pool that holds no token yet gets its RoPE tables with its first tokens
  cudaError_t e = (L.rope && nb == 0 && w == 0) ? launch_rope_tables(L, cb, s) : cudaSuccess;
  while (i0 < n_new && e == cudaSuccess) {
    Layout S = L;  // the live state this step starts from
    S.NB = nb;
    S.W = w;
    S.W16 = (w + 15) / 16 * 16;
    if (w == cap_w) {
      e = launch_append_compress(S, cb, ws, err, s);
      ++nb;
      w -= 256;
      continue;
    }
    const int take = n_new - i0 < cap_w - w ? n_new - i0 : cap_w - w;
    S.W16 = (w + take + 15) / 16 * 16;
    e = launch_append_write(S, static_cast<const __half*>(K_new), static_cast<const __half*>(V_new), n_new, i0,
                            take, w, cb, s);
    w += take;
    i0 += take;
  }
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  d->n_blocks = nb;
  d->window = w;
  return dkv_layout(d);
}

int dkv_decode_launches(const dkv_desc* d, int32_t top_k) {
  Layout L;
  if (top_k < 0 || check_desc(d, &L) != DKV_OK) return 0;
  return decode_launches(L, plan_decode(L, d->n_q_heads, d->n_kv_heads, top_k), d->n_q_heads, d->n_kv_heads);
}

size_t dkv_decode_workspace_bytes(const dkv_desc* d, int32_t top_k) {
  Layout L;
  if (top_k < 0 || check_desc(d, &L) != DKV_OK) return 0;
  return plan_decode(L, d->n_q_heads, d->n_kv_heads, top_k).ws_bytes;
}

// shared argument checks of the decode calls; fills the plan and workspace views
struct DecodeCall {
  Layout L;
  DecodePlan P;
  cudaStream_t s;
  uint8_t* ws;
  float* parts;
};

static int prep_decode(const dkv_desc* d, int32_t top_k, void* workspace, size_t ws_bytes, void* stream,
                       DecodeCall* c) {
  int st = check_desc(d, &c->L);
  if (st != DKV_OK) return st;
  if (top_k < 0) return DKV_ERR_ARG;
  if (c->L.NB == 0 && c->L.W == 0) return DKV_ERR_SHAPE;  // an empty stream: nothing to attend yet
  if (!workspace) return DKV_ERR_ARG;
  if (!aligned16(workspace)) return DKV_ERR_ALIGN;
  c->P = plan_decode(c->L, d->n_q_heads, d->n_kv_heads, top_k);
  if (ws_bytes < c->P.ws_bytes) return DKV_ERR_WORKSPACE;
  c->ws = static_cast<uint8_t*>(workspace);
  c->s = static_cast<cudaStream_t>(stream);
  c->parts = reinterpret_cast<float*>(c->ws + c->P.off_partials);
  return DKV_OK;
}

int dkv_decode_route(const dkv_desc* d, const void* q, const void* cache, int32_t top_k, int32_t* routed,
                     void* workspace, size_t ws_bytes, void* stream) {
  DecodeCall c;
  int st = prep_decode(d, top_k, workspace, ws_bytes, stream, &c);
  if (st != DKV_OK) return st;
  if (!q || !cache) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(cache) || (routed && !aligned16(routed))) return DKV_ERR_ALIGN;
  if (c.P.K_eff == 0) return DKV_OK;
  cudaError_t e = launch_route(c.L, c.P, d->n_q_heads, d->n_kv_heads, static_cast<const __half*>(q),
                               static_cast<const uint8_t*>(cache), c.ws, routed, c.s);
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_decode_blocks(const dkv_desc* d, const void* q, const void* cache, int32_t top_k, float* out, float* lse,
                      void* workspace, size_t ws_bytes, void* stream) {
  DecodeCall c;
  int st = prep_decode(d, top_k, workspace, ws_bytes, stream, &c);
  if (st != DKV_OK) return st;
  if (!q || !cache || (!out && lse)) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(cache) || (out && !aligned16(out)) || (lse && !aligned16(lse)))
    return DKV_ERR_ALIGN;
  cudaError_t e = launch_attend(c.L, c.P, d->n_q_heads, d->n_kv_heads, static_cast<const __half*>(q),
                                static_cast<const uint8_t*>(cache), c.ws, out, lse, c.s);
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_decode_combine(const dkv_desc* d, int32_t top_k, float* out, float* lse, void* workspace, size_t ws_bytes,
                       void* stream) {
  DecodeCall c;
  int st = prep_decode(d, top_k, workspace, ws_bytes, stream, &c);
  if (st != DKV_OK) return st;
  if (!out) return DKV_ERR_ARG;
  if (!aligned16(out) || (lse && !aligned16(lse))) return DKV_ERR_ALIGN;
  cudaError_t e = launch_combine(c.L, c.P, d->batch, d->n_q_heads, d->n_kv_heads, c.parts, out, lse, c.s);
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_decode_attend(const dkv_desc* d, const void* q, const void* cache, int32_t top_k, float* out, float* lse,
                      int32_t* routed, void* workspace, size_t ws_bytes, void* stream) {
  DecodeCall c;
  int st = prep_decode(d, top_k, workspace, ws_bytes, stream, &c);
  if (st != DKV_OK) return st;
  if (!q || !cache || !out) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (routed && !aligned16(routed)))
    return DKV_ERR_ALIGN;
  const cudaError_t e = launch_decode(c.L, c.P, d->n_q_heads, d->n_kv_heads, static_cast<const __half*>(q),
                                      static_cast<const uint8_t*>(cache), c.ws, out, lse, routed, c.s);
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

size_t dkv_dense_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || T < 1 || n_q_heads % n_kv_heads) return 0;
  if ((head_dim != 64 && head_dim != 128) || n_q_heads / n_kv_heads > 8) return 0;
  return dense_ws_bytes(batch, n_q_heads, n_kv_heads, head_dim, T);
}

int dkv_dense_decode(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                     const void* q, const void* K, const void* V, float* out, float* lse, void* workspace,
                     size_t ws_bytes, void* stream) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || T < 1) return DKV_ERR_ARG;
  if (n_q_heads % n_kv_heads) return DKV_ERR_SHAPE;
  if ((head_dim != 64 && head_dim != 128) || n_q_heads / n_kv_heads > 8) return DKV_ERR_UNSUPPORTED;
  if (!q || !K || !V || !out || !workspace) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) || !aligned16(workspace) ||
      (lse && !aligned16(lse)))
    return DKV_ERR_ALIGN;
  if (ws_bytes < dense_ws_bytes(batch, n_q_heads, n_kv_heads, head_dim, T)) return DKV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_dense(batch, n_q_heads, n_kv_heads, head_dim, T, static_cast<const __half*>(q),
                               static_cast<const __half*>(K), static_cast<const __half*>(V), out, lse, ws,
                               reinterpret_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

static int check_prefill(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                         int32_t top_k) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || T < 1 || top_k < 0) return DKV_ERR_ARG;
  if (n_q_heads % n_kv_heads) return DKV_ERR_SHAPE;
  if ((head_dim != 64 && head_dim != 128) || n_q_heads / n_kv_heads > 8) return DKV_ERR_UNSUPPORTED;
  if (T > 1025 * DKV_BLOCK_SIZE) return DKV_ERR_UNSUPPORTED;  // routed lists kept in shared memory
  return DKV_OK;
}

int32_t dkv_prefill_routed_slots(int32_t T, int32_t top_k) {
  if (T < 1 || top_k < 0) return 0;
  return plan_prefill(1, 1, 64, T, top_k).K_eff;
}

size_t dkv_prefill_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                                   int32_t top_k) {
  if (check_prefill(batch, n_q_heads, n_kv_heads, head_dim, T, top_k) != DKV_OK) return 0;
  return plan_prefill(batch, n_kv_heads, head_dim, T, top_k).ws_bytes;
}

int dkv_prefill_attend(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                       int32_t top_k, const void* q, const void* K, const void* V, float* out, float* lse,
                       int32_t* routed, void* workspace, size_t ws_bytes, void* stream) {
  const int st = check_prefill(batch, n_q_heads, n_kv_heads, head_dim, T, top_k);
  if (st != DKV_OK) return st;
  if (!q || !K || !V || !out || !workspace) return DKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) || !aligned16(workspace) ||
      (lse && !aligned16(lse)) || (routed && !aligned16(routed)))
    return DKV_ERR_ALIGN;
  if (ws_bytes < plan_prefill(batch, n_kv_heads, head_dim, T, top_k).ws_bytes) return DKV_ERR_WORKSPACE;
  const cudaError_t e = launch_prefill(batch, n_q_heads, n_kv_heads, head_dim, T, top_k,
                                       static_cast<const __half*>(q), static_cast<const __half*>(K),
                                       static_cast<const __half*>(V), out, lse, routed,
                                       static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA;
}

int dkv_debug_set_limits(int32_t stop_after_chunks, uint32_t wait_polls) {
  set_debug_limits(stop_after_chunks, wait_polls);
  return DKV_OK;
}

int dkv_debug_set_launch(int32_t programmatic) {
  set_programmatic_launch(programmatic != 0);
  return DKV_OK;
}

int dkv_get_error(void* workspace, void* stream, uint32_t* word) {
  if (!workspace || !word) return DKV_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DKV_ERR_CUDA;
  if (cudaMemcpy(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return DKV_ERR_CUDA;
  if (w && cudaMemset(workspace, 0, sizeof(uint32_t) * 2) != cudaSuccess) return DKV_ERR_CUDA;
  *word = w;
  if (w & DKV_DEVERR_TIMEOUT) return DKV_ERR_TIMEOUT;
  return w ? DKV_ERR_DEVICE : DKV_OK;
}

}  // extern "C"
