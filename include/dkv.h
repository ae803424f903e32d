/*
 * dkv.h -- C ABI of libdkv: DKV decode-time attention over an anchor +
 * low-rank differential KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * Method (cited by page title and section):
 *   [DKV-Z]  "DKV: Anchor + Low-Rank Differential KV-Cache Compression for
 *            Scalable Long-Context Inference" (Zenodo record), abstract.
 *   [README] "Differential-KV (DKV): Anchor + Low-Rank KV-Cache Compression"
 *            (project README): "Core Architecture & Paper Overview" (Core),
 *            "Key Environment Knobs" (Knobs), "Measured Paper Benchmarks"
 *            (Bench), "Core Innovations" (Innov).
 *
 * Each 256-token block of a (sequence, KV head) is stored as an exact anchor
 * token (a_k, a_v), a rank-r joint K|V truncated-SVD delta (U with the
 * singular values folded in, V_K, V_V) and R exact residual rows; a dense
 * recency window sits beside the blocks ([DKV-Z]; [README Core] items 1-4).
 * At decode time each query group routes to the top-K blocks, scores them in
 * low-rank space as q.a_k + U_i.(V_K q) without materialising K, forms the
 * value as (sum p) a_v + (sum p U_i) V_V, attends the residual rows and the
 * window exactly, and merges all partial results with an fp32 log-sum-exp
 * reduction over fp16 operands ([DKV-Z]; [README Core] "Low-Rank Space Query
 * Scoring", "Flash-Style LSE Combine").
 *
 * Conventions for every call:
 *   - Pointers named "device" point to CUDA device memory that the CALLER
 *     allocated and owns; the library allocates nothing and keeps no pointer
 *     after a call returns.  Buffers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Work is enqueued asynchronously on it; the call returns
 *     before the GPU finishes.
 *   - Return value: DKV_OK (0) or a negative DKV_ERR_* code.  When arguments
 *     fail validation nothing is launched and no memory is touched.  Nothing
 *     throws across the ABI.
 *   - Faults found on the device (a bounded wait that gave up, an index out of
 *     range) set bits in an error word kept in the workspace header; read and
 *     clear it with dkv_get_error().
 *   - Units: a unit is one (sequence b, KV head h), numbered u = b*n_kv_heads + h.
 *     Query head j belongs to KV head j / G with G = n_q_heads / n_kv_heads.
 */
#ifndef DKV_H
#define DKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DKV_VERSION 5

#if defined(__GNUC__)
#define DKV_API __attribute__((visibility("default")))
#else
#define DKV_API
#endif

/* status codes */
#define DKV_OK               0
#define DKV_ERR_ARG         -1  /* null pointer, negative count, bad value */
#define DKV_ERR_SHAPE       -2  /* sizes inconsistent with each other or with the descriptor */
#define DKV_ERR_ALIGN       -3  /* a pointer is not 16-byte aligned */
#define DKV_ERR_UNSUPPORTED -4  /* well-formed but outside what the kernels implement */
#define DKV_ERR_CUDA        -5  /* a CUDA runtime call failed */
#define DKV_ERR_TIMEOUT     -6  /* a bounded device wait gave up (see dkv_get_error) */
#define DKV_ERR_WORKSPACE   -7  /* workspace missing or smaller than required */
#define DKV_ERR_DEVICE      -8  /* the device error word is non-zero (see dkv_get_error) */

/* bits of the device error word */
#define DKV_DEVERR_TIMEOUT  0x1u  /* an mbarrier wait exceeded its iteration limit */
#define DKV_DEVERR_INDEX    0x2u  /* a routed block index or residual position was out of range */
#define DKV_DEVERR_RANGE    0x4u  /* a compressed factor did not fit fp16 (saturated) */

#define DKV_BLOCK_SIZE 256      /* [README Core]: fixed micro-blocks of B_s = 256 tokens */

/* byte order of the packed cache (dkv_desc.layout); both hold the same bytes */
#define DKV_LAYOUT_FRAGMENT 0   /* operand tiles in mma.sync fragment order (default) */
#define DKV_LAYOUT_TC       1   /* operand tiles as 8x8 core matrices read by tcgen05.mma:
                                   head_dim 128, 1 <= rank <= 48, 1 <= n_residual <= 128 */

/*
 * Descriptor of one layer's compressed cache.  The caller sets the first
 * thirteen fields; dkv_layout() validates them and fills the rest.  Plain old
 * data: pass it by pointer, copy it freely.
 *
 * Supported: head_dim 64 or 128; 1 <= n_q_heads/n_kv_heads <= 8; block_size
 * 256; 0 <= rank <= 128; 0 <= n_residual <= 255; 0 <= n_blocks <= 2048;
 * 0 <= window <= 65536; n_blocks + window > 0.  layout DKV_LAYOUT_TC narrows
 * this to head_dim 128, 1 <= rank <= 48 and 1 <= n_residual <= 128.  The layout
 * picks the decode kernel: DKV_LAYOUT_FRAGMENT the mma.sync kernel,
 * DKV_LAYOUT_TC the tcgen05 kernel (TMEM accumulators).  A cache is only
 * readable under the layout it was written with.
 *
 * n_blocks and window are the live counts; the byte layout follows
 * block_capacity and window_capacity, so a cache keeps its offsets while
 * dkv_append() grows n_blocks and moves the window (0 means "no spare room").
 * Capacities obey the same limits as the counts (2048 blocks, 65536 tokens).
 *
 * residual_bits picks how the R exact residual rows are stored ([README Innov]
 * "Physical 4-Bit Group-Quantized Residual Buffers"; [README Knobs]
 * DKV_RESIDUAL_QUANT, DKV_RESIDUAL_QUANT_GROUP_SIZE): 0 keeps them as fp16; 8
 * or 4 stores each key row and each value row group-quantised: per 64
 * channels an fp16 bias (the group's minimum) and an fp16 scale ((maximum -
 * minimum) / (2^bits - 1)), and per channel the code round((x - bias) /
 * scale) clamped to [0, 2^bits - 1] (taken in fp32, ties to even; a group of
 * equal values has scale 0 and codes 0).  The decode attends the dequantised
 * rows scale * code + bias, rounded to fp16 (the operand precision).  Only the
 * fragment layout, and head_dim 64 or 128, take quantised residuals; R is then
 * padded to a multiple of 16.
 *
 * rope_dims > 0 makes the cache an un-rotated pool ([README Knobs]
 * DKV_ROTATED_POOL=0: keys are stored before RoPE and rotated to their absolute
 * positions at read).  The keys given to dkv_compress_layout, dkv_append and
 * dkv_import_factors are then keys BEFORE RoPE, stored as given; the decode
 * rotates every key it attends to its absolute position (block b's token i
 * at 256 b + i, window token w at 256 n_blocks + w) with the rotate-half
 * RoPE: for j < h = rope_dims / 2 the channel pair (j, j + h) turns by the
 * angle pos * rope_base^(-2j / rope_dims); channels from rope_dims on are not
 * rotated.  q is the query as the model gives it, already rotated to its own
 * position; values are never rotated.  The router section then holds each
 * block's box over its exact keys AFTER rotation, in fp32 ([kmin | kmax], 8d
 * bytes per block), and the cache ends with RoPE tables (cos, sin as fp32
 * pairs of the angles 256 p theta_j for every 256-token page p the
 * capacities reach, and i theta_j for i < 256), at off_rope, written by
 * dkv_compress_layout, dkv_import_factors and the first dkv_append into an
 * empty cache.  Supported with the fragment layout and fp16 residual rows,
 * rope_dims a multiple of 32 up to head_dim, rope_base > 1 and finite.
 * rope_dims 0 (the default) stores and attends keys as given (a rotated pool).
 */
typedef struct dkv_desc {
  int32_t batch;        /* sequences B */
  int32_t n_q_heads;    /* query heads Hq */
  int32_t n_kv_heads;   /* KV heads Hkv (Hq % Hkv == 0) */
  int32_t head_dim;     /* d */
  int32_t block_size;   /* must be 256 */
  int32_t n_blocks;     /* compressed blocks NB per unit */
  int32_t window;       /* exact recency-window tokens W per unit */
  int32_t rank;         /* r: rank of the joint K|V delta ([README Core] item 2) */
  int32_t n_residual;   /* R: exact residual rows per block ([README Core] item 3) */
  int32_t layout;       /* DKV_LAYOUT_FRAGMENT (0) or DKV_LAYOUT_TC (1) */
  int32_t block_capacity;   /* blocks the cache has room for (0: n_blocks); >= n_blocks */
  int32_t window_capacity;  /* window token slots (0: window); >= window */
  int32_t residual_bits;    /* 0: fp16 residual rows; 8 or 4: group-quantised (see above) */
  int32_t rope_dims;        /* 0: rotated pool; > 0: un-rotated pool, RoPE over this many channels at read */
  float rope_base;          /* RoPE base (un-rotated pool only) */
  /* ---- filled by dkv_layout() ---- */
  int32_t rank_pad;     /* r rounded up to a multiple of 8 (zero-padded) */
  int32_t res_pad;      /* R rounded up to a multiple of 8 (16 when quantised; zero-padded) */
  int32_t window_pad;   /* W rounded up to a multiple of 16 (zero-padded) */
  int32_t n_units;      /* B * Hkv */
  /* byte offsets inside one block record */
  uint64_t blk_off_mask, blk_off_vk, blk_off_u, blk_off_res, blk_off_vv, block_bytes;
  /* byte offsets inside one unit record */
  uint64_t off_router, off_blocks, off_cold, off_window;
  uint64_t block_stride, unit_stride, total_bytes;
  uint64_t off_rope;    /* byte offset of the RoPE tables in the cache (un-rotated pool; else 0) */
} dkv_desc;

/*
 * Plain row-major factors of a whole layer, used by dkv_import_factors() to
 * fill the packed cache from factors produced elsewhere (for instance a host
 * reference implementation).  All device pointers; fp16 unless noted.
 * Shapes use U_ = n_units, NB, r, R, W, d from the descriptor.
 */
typedef struct dkv_factors {
  const void* a_k;        /* [U_][NB][d]      anchor keys (the block's first token) */
  const void* a_v;        /* [U_][NB][d]      anchor values */
  const void* U;          /* [U_][NB][255][r] low-rank coefficients of tokens 1..255, S folded in */
  const void* V_K;        /* [U_][NB][r][d]   key half of the joint right basis */
  const void* V_V;        /* [U_][NB][r][d]   value half */
  const int32_t* res_pos; /* [U_][NB][R]      residual token positions, 1..255, strictly ascending */
  const void* K_res;      /* [U_][NB][R][d]   exact residual keys */
  const void* V_res;      /* [U_][NB][R][d]   exact residual values */
  const void* kmin;       /* [U_][NB][d]      per-channel key minimum over the block (an un-rotated
                                              pool: fp32, over the keys rotated to their positions) */
  const void* kmax;       /* [U_][NB][d]      per-channel key maximum (likewise) */
  const void* win_K;      /* [U_][W][d]       recency-window keys */
  const void* win_V;      /* [U_][W][d]       recency-window values */
} dkv_factors;

/* Library version (DKV_VERSION). */
DKV_API int dkv_version(void);

/* Human-readable name of a status code; never NULL. */
DKV_API const char* dkv_status_string(int status);

/*
 * Validate the caller-set fields of *d and fill the layout fields.
 * Returns DKV_OK, DKV_ERR_ARG (null / negative / unknown layout), DKV_ERR_SHAPE
 * (Hq % Hkv != 0, nothing to attend) or DKV_ERR_UNSUPPORTED.  Host only; needs
 * no GPU.
 */
DKV_API int dkv_layout(dkv_desc* d);

/* dkv_layout() then the total cache size in bytes; 0 when validation fails. */
DKV_API size_t dkv_layout_bytes(dkv_desc* d);

/*
 * Compress a layer's exact K and V into the packed cache ([DKV-Z]; [README
 * Core] items 1-4): per block the anchor = first token, a rank-r truncated
 * SVD of the joint deltas [K_i - a_k | V_i - a_v] (i = 1..255) with the
 * singular values folded into U, the R rows with the largest key
 * reconstruction error ||k_i - k_hat_i||_2 kept exact (ties to the lower
 * row; [README Innov] "vanilla L2" criterion), per-channel key min/max for
 * the router; the last W tokens are copied as the exact window.
 *   d      descriptor filled by dkv_layout()
 *   K, V   device fp16 [B][Hkv][T][head_dim], T = n_blocks*256 + window
 *   cache  device buffer of d->total_bytes bytes, written entirely
 *   workspace / ws_bytes  device scratch of dkv_compress_workspace_bytes(d)
 * The GPU compressor supports rank <= 64 at head_dim 128 (<= 112 at 64).
 */
DKV_API size_t dkv_compress_workspace_bytes(const dkv_desc* d);
DKV_API int dkv_compress_layout(const dkv_desc* d, const void* K, const void* V, void* cache,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Fill the packed cache from plain factors (see dkv_factors).  Overwrites the
 * whole cache.  `workspace` is a device buffer of at least 256 bytes whose
 * header receives the device error word: residual positions must be strictly
 * ascending in 1..255, else DKV_DEVERR_INDEX is raised and the offending
 * block keeps no residual row (its mask is left empty).
 */
DKV_API int dkv_import_factors(const dkv_desc* d, const dkv_factors* f, void* cache, void* workspace, void* stream);

/*
 * Streaming append ([DKV-Z]; [README Core] items 1-4 applied as tokens
 * arrive): add n_new tokens per unit to the exact recency window.  Whenever
 * the window has no free slot left, its oldest 256 tokens are first
 * compressed into block n_blocks (anchor, joint K|V truncated SVD, residual
 * rows, router min/max: the same computation as dkv_compress_layout) and the
 * window slides down by 256 tokens.  After any sequence of appends the cache
 * holds exactly what dkv_compress_layout writes for the whole token sequence
 * with the final (n_blocks, window).
 *   d          descriptor filled by dkv_layout(); on DKV_OK its n_blocks and
 *              window are advanced and its layout fields refreshed (the byte
 *              offsets do not change)
 *   K_new, V_new  device fp16 [B][Hkv][n_new][head_dim]
 *   cache      device buffer written by dkv_compress_layout / dkv_import_factors
 *              / dkv_append with the same capacities
 *   workspace / ws_bytes  device scratch of dkv_append_workspace_bytes(d); its
 *              header receives the device error word
 * Returns DKV_ERR_UNSUPPORTED, with nothing launched, when the appends would
 * need a block beyond block_capacity, when a compression step finds fewer than
 * 256 window tokens (window_capacity < 256), or for the tensor-core layout.
 */
DKV_API size_t dkv_append_workspace_bytes(const dkv_desc* d);
DKV_API int dkv_append(dkv_desc* d, const void* K_new, const void* V_new, int32_t n_new, void* cache,
                       void* workspace, size_t ws_bytes, void* stream);

/*
 * Decode-time attention for one layer ([DKV-Z]; [README Core]; [README
 * Knobs] DKV_TOPK_BLOCKS, DKV_CB_GQA_ROUTE).
 *   q       device fp16 [B][Hq][head_dim], one decode query per (sequence, head)
 *   cache   device packed cache (dkv_compress_layout / dkv_import_factors)
 *   top_k   blocks routed per unit; 0 or >= n_blocks attends every block
 *           (the README's DKV_TOPK_BLOCKS=0 reading); negative is DKV_ERR_ARG
 *   out     device fp32 [B][Hq][head_dim]: softmax(c q K_hat^T) V_hat over the
 *           routed blocks and the window, c = 1/sqrt(head_dim)
 *   lse     optional device fp32 [B][Hq]: natural-log log-sum-exp of the scores
 *   routed  optional device int32 [B][Hkv][K_eff]: routed block indices,
 *           ascending, K_eff = top_k clipped to n_blocks.  Asking for them
 *           costs the router a second cluster exchange (about 0.7 us at 64k); without
 *           them the router writes each block to its rank's slot.
 *   workspace / ws_bytes  device scratch of dkv_decode_workspace_bytes(d, top_k)
 *           (its size depends on the current device's multiprocessor count);
 *           zero-fill it once before its first use: its 256-byte header holds
 *           the device error word (read by dkv_get_error), and the 8 bytes
 *           right after the header hold the work-queue counters of the
 *           tensor-core layout's kernel, which every call that completes
 *           leaves at zero again.  After DKV_ERR_TIMEOUT zero-fill the
 *           workspace again before reusing it: a kernel that gave up on a
 *           wait can leave those counters set
 * Routing: qbar = mean over the group of c*q; block score
 * sum_j max(qbar_j kmax_bj, qbar_j kmin_bj); top-K by (score desc, index asc).
 */
DKV_API size_t dkv_decode_workspace_bytes(const dkv_desc* d, int32_t top_k);
DKV_API int dkv_decode_attend(const dkv_desc* d, const void* q, const void* cache, int32_t top_k,
                      float* out, float* lse, int32_t* routed,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Kernel launches one dkv_decode_attend(d, ..., top_k, ...) makes: the router,
 * the block/window attention and the log-sum-exp combine, 3; 2 when there is
 * nothing to route (n_blocks == 0, or, for the fragment layout, every block
 * routed: top_k 0 or >= n_blocks).  Returns 0 for an invalid descriptor or
 * top_k.
 */
DKV_API int dkv_decode_launches(const dkv_desc* d, int32_t top_k);

/*
 * The stages of dkv_decode_attend as separate calls, for callers that
 * schedule or time them individually.  Run them in this order on one stream
 * with one workspace (it carries the routed indices and the partial results
 * from stage to stage); arguments mean the same as for dkv_decode_attend.
 *   route:   top-K block selection per unit (does nothing when n_blocks == 0).
 *            With `routed` given, the workspace list and the caller's copy
 *            hold the indices in ascending order; with routed == NULL the
 *            workspace list holds block of rank k (by score desc, index asc)
 *            in slot k.  The attention result is the same set of blocks
 *            either way; only the fp32 summation order differs.
 *   blocks:  partial results (m, l, acc): for the fragment layout one per
 *            unit, balanced slice of its work and consumer warp, for the
 *            tensor-core layout one per routed block and window chunk; when
 *            `out` is given the combine follows at once (what
 *            dkv_decode_attend does); with out == NULL (and lse == NULL) the
 *            partials stay in the workspace for dkv_decode_combine
 *   combine: fp32 log-sum-exp merge of the partials into out (and lse)
 */
DKV_API int dkv_decode_route(const dkv_desc* d, const void* q, const void* cache, int32_t top_k, int32_t* routed,
                             void* workspace, size_t ws_bytes, void* stream);
DKV_API int dkv_decode_blocks(const dkv_desc* d, const void* q, const void* cache, int32_t top_k,
                              float* out, float* lse, void* workspace, size_t ws_bytes, void* stream);
DKV_API int dkv_decode_combine(const dkv_desc* d, int32_t top_k, float* out, float* lse,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * dkv_decode_attend without a workspace argument, for callers that cannot
 * allocate device memory when they decode: runtimes that reserve a fixed
 * memory pool at start-up and refuse later allocations, plugins that run
 * inside another framework without access to its allocator, and serving
 * loops that must not pay the device-wide synchronisation of cudaMalloc.
 * The paper has no counterpart to this call; it only changes where the
 * scratch memory comes from.
 *
 * The scratch (routed indices and partial results) lives in a fixed 8 MiB
 * area compiled into the library; each GPU that loads the library keeps its
 * own copy until the process exits.  A call whose scratch need
 * (dkv_decode_workspace_bytes) is larger returns DKV_ERR_WORKSPACE and
 * launches nothing.  The call itself allocates nothing.
 *   - The first call on a device looks up that device's copy of the area;
 *     make that first call before any stream capture on the device.
 *   - Every call on a device shares the one area, which keeps the last
 *     call's contents: calls that overlap on the GPU (on different streams,
 *     or from different threads) race and corrupt each other's results.
 *     Serialise them, for instance on one stream.
 *   - Each call first clears the area's header (the error word) and the
 *     work-queue counters after it, so a call that gave up on a wait does
 *     not leave later calls with a stale work queue; the error word cannot
 *     be read back; use dkv_decode_attend with a workspace to diagnose.
 * Other arguments, layouts and results are those of dkv_decode_attend.
 */
DKV_API int dkv_decode_attend_noalloc(const dkv_desc* d, const void* q, const void* cache, int32_t top_k,
                                      float* out, float* lse, int32_t* routed, void* stream);

/*
 * Dense fp16 decode attention over uncompressed K, V: the bytes/throughput
 * reference the compressed path is compared with.
 *   K, V   device fp16 [B][Hkv][T][head_dim]; T >= 1
 *   q      device fp16 [B][Hq][head_dim];  out fp32 [B][Hq][head_dim];  lse optional fp32 [B][Hq]
 */
DKV_API size_t dkv_dense_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t T);
DKV_API int dkv_dense_decode(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                     const void* q, const void* K, const void* V, float* out, float* lse,
                     void* workspace, size_t ws_bytes, void* stream);

/*
 * Block-sparse prefill attention ([DKV-Z]: "Prefill uses training-free
 * block-sparse attention, so its cost grows sub-quadratically"; [README Core]
 * "Sub-Quadratic Prefill": O(L^2) down to O(L * K)).  Exact K and V are in hand
 * at prefill; each 256-token query block i attends the keys of its own block
 * causally (token t sees keys up to t) and every key of the top_k earlier
 * blocks j < i, ranked by the decode router's key-box bound taken with the
 * block's mean query: qbar_i = mean over the block's tokens and the GQA
 * group's heads of c*q, bound_ij = sum_d max(qbar_id kmax_jd, qbar_id kmin_jd)
 * over the channel extremes of block j's keys, top_k by (bound desc, j asc);
 * top_k 0 or >= i attends every earlier block (top_k 0 is dense causal
 * attention).  The last block may be partial (T need not be a multiple of 256).
 *   q       device fp16 [B][Hq][T][head_dim]
 *   K, V    device fp16 [B][Hkv][T][head_dim]
 *   out     device fp32 [B][Hq][T][head_dim]: softmax(c q k^T) v over each token's key set
 *   lse     optional device fp32 [B][Hq][T]: natural-log log-sum-exp of the scores
 *   routed  optional device int32 [B][Hkv][nb][slots] with nb = ceil(T / 256) and
 *           slots = dkv_prefill_routed_slots(T, top_k): each query block's routed
 *           blocks ascending, -1 in the unused slots
 *   workspace / ws_bytes  device scratch of dkv_prefill_workspace_bytes(...)
 * Supported: head_dim 64 or 128, n_q_heads / n_kv_heads <= 8, 1 <= T <= 262400.
 * The products run on the tensor cores with fp16 operands and fp32 accumulation:
 * tcgen05 with tensor-memory accumulators at head_dim 128, mma.sync at head_dim 64.
 */
DKV_API int32_t dkv_prefill_routed_slots(int32_t T, int32_t top_k);
DKV_API size_t dkv_prefill_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                           int32_t T, int32_t top_k);
DKV_API int dkv_prefill_attend(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t T,
                               int32_t top_k, const void* q, const void* K, const void* V, float* out, float* lse,
                               int32_t* routed, void* workspace, size_t ws_bytes, void* stream);

/*
 * Diagnostics for the failure path (no counterpart in the pages): from the
 * next launch on, the producer of every attention CTA of the fragment layout
 * issues at most `stop_after_chunks` chunks (negative: all of them) and every
 * bounded device wait of that kernel gives up after `wait_polls` polls of at
 * most about 20 us each (0: the default limit, about 1.3 s).  A stopped
 * producer leaves its consumer warps waiting for data that never comes: their
 * waits give up, DKV_DEVERR_TIMEOUT is raised in the error word and the
 * outputs of the call are meaningless; every copy that was issued has landed
 * before the kernel ends, so the context stays usable.  The setting is
 * process-wide; dkv_debug_set_limits(-1, 0) restores the defaults.  Returns
 * DKV_OK.
 */
DKV_API int dkv_debug_set_limits(int32_t stop_after_chunks, uint32_t wait_polls);

/*
 * Timing aid (no counterpart in the pages): with programmatic = 0 the decode
 * grids that are normally programmatic dependents of the grid before them (the
 * attention grid of both layouts, and the combine grid) are launched in plain
 * stream order from the next launch on: each starts once the previous grid on
 * the stream has finished, so that consecutive attention grids of a timing loop
 * cannot overlap.  Results are unchanged.  programmatic = 1 restores the
 * default.  The setting is process-wide and read when a grid is launched (or
 * captured into a CUDA graph).  Returns DKV_OK.
 */
DKV_API int dkv_debug_set_launch(int32_t programmatic);

/*
 * Synchronise `stream`, read the device error word kept in the header of
 * `workspace` (any workspace passed to the calls above), store it in *word
 * and clear it.  Returns DKV_OK, DKV_ERR_TIMEOUT when the timeout bit is set,
 * DKV_ERR_DEVICE for other bits, DKV_ERR_CUDA when the stream failed.
 */
DKV_API int dkv_get_error(void* workspace, void* stream, uint32_t* word);

#ifdef __cplusplus
}
#endif
#endif /* DKV_H */
