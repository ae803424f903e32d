// Internal header of libdkv: packed-layout address math, PTX wrappers and
// the launcher prototypes shared by the .cu files of the library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dkv.h"

namespace dkv {

// ---------------------------------------------------------------------------
// Packed layout of one block record (all sections 16-byte aligned):
//
//   [0, 4d)            a_k[d], a_v[d]                       fp16, plain
//   [4d, 4d+32)        residual mask, 256 bits (bit i = token i kept exact)
//   [off_vk, off_u)    V_K  [r8][d]   "B^T layout"  (B operand of z^T = q^T V_K^T)
//   [off_u, off_res)   U    [256][r8] as 8x8 core matrices (tc_u_off; row 0 = anchor, all zero)
//   [off_res, off_vv)  residual groups of 16 tokens (last group may hold 8):
//                      K_res tile in "A layout" then V_res^T tile in "A layout"
//   [off_vv, bytes)    V_V^T [d][r8]  "A layout"    (A operand of o = V_V^T w)
//
// The router section of a unit is [NB][2][d] fp16 (kmin row, kmax row); the
// cold section is [NB][R8] uint16 residual positions; the window is W16
// tokens in 16-token groups laid out like the residual groups.
//
// "A layout" of an M x K fp16 matrix (M, K multiples of 8): 16-row m-tiles,
// inside each m-tile 16-column k-tiles, inside each (m-tile, k-tile) the 8x8
// sub-blocks of an mma.m16n8k16 A fragment, interleaved per lane:
//   lane l holds, for each existing sub-block in the order a0 (rows 0-7,
//   cols 0-7), a1 (rows 8-15, cols 0-7), a2 (rows 0-7, cols 8-15), a3 (rows
//   8-15, cols 8-15), the two halves at (row l/4, cols 2(l%4), 2(l%4)+1).
// A lane therefore reads its whole fragment with one 16-byte (full tile),
// 8-byte (half tile) or 4-byte load.  "B^T layout" of an N x K matrix
// (the transpose of an mma B operand): 8-row n-tiles, 32-column k-pairs,
// lane l holds b0,b1 of k-tile 2p then b0,b1 of k-tile 2p+1 (16 bytes).
// ---------------------------------------------------------------------------

struct Layout {
  int d, r, r8, R, R8, W, W16, NB, units;
  int tc;              // 1: tensor-core (core-matrix) layout, 0: mma.sync fragment layout
  int qbits;           // residual rows: 0 fp16, 8 or 4 group-quantised (fragment layout)
  int qgb;             // bytes of one 16-token group of quantised residual rows (0 for fp16)
  int rope;            // 0: rotated pool; > 0: un-rotated pool, RoPE over the first `rope` channels at read
  float rope_base;
  int rope_pages;      // 256-token pages the RoPE page table covers
  uint64_t off_rope;   // RoPE tables (after the units): [pages][rope/2] then [256][rope/2] float2 (cos, sin)
  uint64_t off_mask, off_vk, off_u, off_res, off_vv, block_bytes;
  uint64_t off_router, off_blocks, off_cold, off_window, block_stride, unit_stride, total;
};

__host__ __device__ inline uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Group-quantised residual rows (Layout.qbits = 8 or 4; fragment layout).  The
// residual rows are stored in 16-token groups (R padded to 16); one group is
//   [K codes: 16 tokens x d][V^T codes: d x 16 tokens]
//   [K scale: G x 16][K bias: G x 16][V scale: G x 16][V bias: G x 16]   fp16, G = d / 64
// Each code section is in the A-fragment order of mma.sync m16n8k16 per 16-wide
// k tile (K: rows = tokens, k = channels; V^T: rows = channels, k = tokens): per
// 512-byte chunk and lane 16 bytes, a chunk holding two k tiles (int8) or four
// (int4).  For the fragment registers a0..a3 of one k tile (two halves x, y each):
//   int8: two words, (a0.x, a1.x, a0.y, a1.y) and (a2.x, a3.x, a2.y, a3.y) as bytes
//   int4: one word, bits 4i..4i+3 = a_i.x and bits 16+4i..16+4i+3 = a_i.y
// so ((word >> s) & 0x00FF00FF) | 0x64006400 (int8; 0x000F000F for int4) is the
// half2 (1024 + code x, 1024 + code y) of one register, exactly.
// ---------------------------------------------------------------------------
constexpr int kQuantGroup = 64;  // channels per scale and bias
__host__ __device__ inline uint32_t qcode_bytes(int d, int bits) { return 16u * (uint32_t)d * (uint32_t)bits / 8u; }
__host__ __device__ inline uint32_t qgroup_bytes(int d, int bits) {
  return 2u * qcode_bytes(d, bits) + 128u * (uint32_t)(d / kQuantGroup);
}

// Write residual rows 0 .. n-1 of one block into its quantised residual store
// `res` (the rows n .. R8-1 of the padding get scale and bias 0 and code 0).
// src_k(i, j) / src_v(i, j) return channel j of residual row i as fp16.  Called by
// every thread of the CTA (it synchronises the CTA once): first the scale and bias
// of every (row, key or value, channel group), then every 32-bit code word, each
// written by one thread.
template <class FK, class FV>
__device__ void write_quant_residuals(const Layout& L, uint8_t* res, int n, FK src_k, FV src_v) {
  const int d = L.d, bits = L.qbits, G = d / kQuantGroup, levels = (1 << bits) - 1;
  const uint32_t cb = qcode_bytes(d, bits), gb = (uint32_t)L.qgb;
  for (int e = threadIdx.x; e < L.R8 * 2 * G; e += blockDim.x) {
    const int i = e / (2 * G), kv = (e / G) & 1, g = e % G;
    __half sh = __float2half(0.f), bh = __float2half(0.f);
    if (i < n) {
      float lo = INFINITY, hi = -INFINITY;
      for (int c = 0; c < kQuantGroup; ++c) {
        const float x = __half2float(kv ? src_v(i, g * kQuantGroup + c) : src_k(i, g * kQuantGroup + c));
        lo = fminf(lo, x);
        hi = fmaxf(hi, x);
      }
      sh = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), (float)levels));
      bh = __float2half_rn(lo);  // exact: the minimum is one of the fp16 values
    }
    __half* sc = reinterpret_cast<__half*>(res + (uint64_t)(i / 16) * gb + 2 * cb + (uint32_t)kv * 64u * G);
    sc[g * 16 + (i & 15)] = sh;
    sc[16 * G + g * 16 + (i & 15)] = bh;
  }
  __syncthreads();
  const uint32_t words = cb / 4, ngrp = (uint32_t)L.R8 / 16;
  for (uint32_t e = threadIdx.x; e < ngrp * 2 * words; e += blockDim.x) {
    const uint32_t grp = e / (2 * words), kv = (e / words) & 1u, w = e % words;
    const int chunk = (int)(w / 128), lane = (int)((w % 128) / 4), wi = (int)(w % 4);
    const int gq = lane >> 2, t = lane & 3;
    const __half* sc = reinterpret_cast<const __half*>(res + (uint64_t)grp * gb + 2 * cb + kv * 64u * G);
    uint32_t word = 0;
    const int ne = bits == 8 ? 4 : 8;
    for (int x = 0; x < ne; ++x) {
      int tile, ai, ex, shift;
      if (bits == 8) { tile = 2 * chunk + (wi >> 1); ai = 2 * (wi & 1) + (x & 1); ex = x >> 1; shift = 8 * x; }
      else { tile = 4 * chunk + wi; ai = x & 3; ex = x >> 2; shift = 4 * x; }
      const int r = gq + 8 * (ai & 1), c = 2 * t + ex + 8 * (ai >> 1);  // row and column inside the tile
      const int tok = 16 * (int)grp + (kv ? c : r), ch = 16 * tile + (kv ? r : c);
      uint32_t code = 0;
      if (tok < n) {
        const int g = ch / kQuantGroup;
        const float s = __half2float(sc[g * 16 + (tok & 15)]), b = __half2float(sc[16 * G + g * 16 + (tok & 15)]);
        if (s != 0.f) {
          const float xv = __half2float(kv ? src_v(tok, ch) : src_k(tok, ch));
          const float qv = rintf(__fdiv_rn(__fsub_rn(xv, b), s));
          code = (uint32_t)fminf(fmaxf(qv, 0.f), (float)levels);
        }
      }
      word |= code << shift;
    }
    *reinterpret_cast<uint32_t*>(res + (uint64_t)grp * gb + kv * cb + w * 4) = word;
  }
}

// ---------------------------------------------------------------------------
// Tensor-core layout (head_dim 128, 8 <= r8 <= 48, 1 <= R <= 128).  Operand
// matrices are stored as 8 x 8 "core matrices" (8 rows of 16 bytes, 128 B
// contiguous), the no-swizzle form tcgen05.mma reads through shared-memory
// descriptors in either K-major or MN-major role.  Block record (the same
// sections as the fragment layout; only V_V and the residual rows swap places):
//   [a_k | a_v]            fp16 d each
//   [mask 32 B]            residual rows
//   [V_K: r8 x d]          mma.sync B^T fragment layout (z is computed with mma.sync)
//   [U: 256 tokens x r8]   two 128-token tiles; inside a tile, per 8-token group
//                          the r8/8 core matrices side by side (r8 * 16 B a group)
//   [V_V: r8 x d]          plane per 8 r-rows (2048 B: 16 d groups)
//   [K_res: R8 x d][V_res: R8 x d]  plane per 8 token rows (2048 B: 16 d groups)
// Window: groups of 128 tokens, each [K: n x d][V: n x d] in the same planes.
// ---------------------------------------------------------------------------
__host__ __device__ inline bool tc_layout(int d, int r8, int R) {
  return d == 128 && r8 >= 8 && r8 <= 48 && R >= 1 && R <= 128;
}
// U element (token t, r-column k)
__host__ __device__ inline uint32_t tc_u_off(int r8, int t, int k) {
  return (uint32_t)(t >> 7) * 256u * (uint32_t)r8 + (uint32_t)((t & 127) >> 3) * 16u * (uint32_t)r8 +
         (uint32_t)(k >> 3) * 128u + (uint32_t)(t & 7) * 16u + (uint32_t)(k & 7) * 2u;
}
// element (row, j) of a [rows][d] matrix with d contiguous per row
__host__ __device__ inline uint32_t tc_rd_off(int d, int row, int j) {
  return (uint32_t)(row >> 3) * (uint32_t)(d >> 3) * 128u + (uint32_t)(j >> 3) * 128u + (uint32_t)(row & 7) * 16u +
         (uint32_t)(j & 7) * 2u;
}

// Section element offsets inside a block record (both layouts)
__host__ __device__ inline uint64_t blk_u_off(const Layout& L, int t, int k);
__host__ __device__ inline uint64_t blk_vv_off(const Layout& L, int k, int j);
__host__ __device__ inline uint64_t blk_resk_off(const Layout& L, int i, int j);
__host__ __device__ inline uint64_t blk_resv_off(const Layout& L, int i, int j);
__host__ __device__ inline uint64_t win_k_off(const Layout& L, int t, int j);
__host__ __device__ inline uint64_t win_v_off(const Layout& L, int t, int j);

// byte offset of element (row, col) inside an "A layout" matrix of rows x cols
__host__ __device__ inline uint32_t a_layout_off(int rows, int cols, int row, int col) {
  int mt = row >> 4, kt = col >> 4;
  int rows_in = rows - (mt << 4); rows_in = rows_in > 16 ? 16 : rows_in;
  int cols_in = cols - (kt << 4); cols_in = cols_in > 16 ? 16 : cols_in;
  int nr = rows_in >> 3, nc = cols_in >> 3;
  int nsb = nr * nc;
  int rr = (row & 15) >> 3, cc = (col & 15) >> 3;
  int sbi = cc * nr + rr;
  int lane = ((row & 7) << 2) | ((col & 7) >> 1);
  uint32_t base = (uint32_t)mt * 16u * (uint32_t)cols * 2u + (uint32_t)kt * 16u * (uint32_t)rows_in * 2u;
  return base + (uint32_t)lane * (uint32_t)nsb * 4u + (uint32_t)sbi * 4u + (uint32_t)(col & 1) * 2u;
}

// byte offset of element (row=n, col=k) inside a "B^T layout" matrix of rows x cols (cols % 32 == 0)
__host__ __device__ inline uint32_t bt_layout_off(int rows, int cols, int row, int col) {
  (void)rows;
  int nt = row >> 3, kp = col >> 5;
  int lane = ((row & 7) << 2) | ((col & 7) >> 1);
  int sb = (col & 31) >> 3;
  return (uint32_t)nt * 8u * (uint32_t)cols * 2u + (uint32_t)kp * 512u + (uint32_t)lane * 16u +
         (uint32_t)sb * 4u + (uint32_t)(col & 1) * 2u;
}

// offset of token t's K element / V element inside a run of 16-token exact groups
// (residual store or window); n_tok = number of stored tokens (multiple of 8)
__host__ __device__ inline uint32_t exact_k_off(int n_tok, int d, int t, int j) {
  int g = t >> 4;
  int in_g = n_tok - (g << 4); in_g = in_g > 16 ? 16 : in_g;
  uint32_t gbase = (uint32_t)g * 64u * (uint32_t)d;
  return gbase + a_layout_off(in_g, d, t & 15, j);
}
__host__ __device__ inline uint32_t exact_v_off(int n_tok, int d, int t, int j) {
  int g = t >> 4;
  int in_g = n_tok - (g << 4); in_g = in_g > 16 ? 16 : in_g;
  uint32_t gbase = (uint32_t)g * 64u * (uint32_t)d + (uint32_t)in_g * (uint32_t)d * 2u;
  return gbase + a_layout_off(d, in_g, j, t & 15);
}

__host__ __device__ inline uint64_t blk_u_off(const Layout& L, int t, int k) {
  return L.off_u + tc_u_off(L.r8, t, k);  // both layouts: 8 x 8 core matrices
}
__host__ __device__ inline uint64_t blk_vv_off(const Layout& L, int k, int j) {
  return L.off_vv + (L.tc ? tc_rd_off(L.d, k, j) : a_layout_off(L.d, L.r8, j, k));
}
__host__ __device__ inline uint64_t blk_resk_off(const Layout& L, int i, int j) {
  return L.off_res + (L.tc ? tc_rd_off(L.d, i, j) : exact_k_off(L.R8, L.d, i, j));
}
__host__ __device__ inline uint64_t blk_resv_off(const Layout& L, int i, int j) {
  return L.off_res + (L.tc ? (uint64_t)L.R8 * 2 * L.d + tc_rd_off(L.d, i, j) : exact_v_off(L.R8, L.d, i, j));
}
// window token t of W16 (relative to the unit's window section)
__host__ __device__ inline uint64_t win_k_off(const Layout& L, int t, int j) {
  if (!L.tc) return exact_k_off(L.W16, L.d, t, j);
  return (uint64_t)(t >> 7) * 128 * 4 * L.d + tc_rd_off(L.d, t & 127, j);
}
__host__ __device__ inline uint64_t win_v_off(const Layout& L, int t, int j) {
  if (!L.tc) return exact_v_off(L.W16, L.d, t, j);
  const int g = t >> 7, n = L.W16 - 128 * g < 128 ? L.W16 - 128 * g : 128;
  return (uint64_t)g * 128 * 4 * L.d + (uint64_t)n * 2 * L.d + tc_rd_off(L.d, t & 127, j);
}

bool make_layout(const dkv_desc* d, Layout* L);  // from a desc filled by dkv_layout()

// ---------------------------------------------------------------------------
// Un-rotated pool (Layout.rope > 0): bytes of one block's router row ([kmin |
// kmax] fp16, or fp32 over the rotated keys) and the RoPE tables at off_rope.
// rope_cs gives (cos, sin) of the angle P theta_j as the page entry of P >> 8
// turned by the in-page entry of P & 255 (one complex product in fp32).
// ---------------------------------------------------------------------------
__host__ __device__ inline uint64_t router_row_bytes(const Layout& L) { return (uint64_t)(L.rope ? 8 : 4) * L.d; }
__device__ inline float2 rope_cs(const float2* __restrict__ tab, int pages, int h, int P, int j) {
  const float2 a = __ldg(tab + (size_t)(P >> 8) * h + j);
  const float2 b = __ldg(tab + (size_t)(pages + (P & 255)) * h + j);
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
cudaError_t launch_rope_tables(const Layout& L, uint8_t* cache, cudaStream_t s);

// ---------------------------------------------------------------------------
// Workspace header (first 256 bytes of every workspace)
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t error_word;
  uint32_t error_detail;
  uint32_t reserved[62];
};
constexpr size_t kWsHeader = 256;

__device__ inline void raise_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// PTX wrappers (sm_90+ forms, used on sm_103a)
// ---------------------------------------------------------------------------
__device__ inline uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ inline void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ inline void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ inline void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ inline void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One bounded wait step: the thread may sleep in hardware until the phase
// completes, for at most kWaitHintNs (suspend-time hint), instead of spinning.
constexpr uint32_t kWaitHintNs = 20000;
__device__ inline bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kWaitHintNs)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after kWaitLimit steps (at most ~1.3 s), raises
// DKV_DEVERR_TIMEOUT and returns false.
constexpr uint32_t kWaitLimit = 1u << 16;
__device__ inline bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  raise_error(err, DKV_DEVERR_TIMEOUT);
  return false;
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`
__device__ inline void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ inline uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2^x with the hardware approximation (2 ulp; ex2(-inf) = 0)
__device__ inline float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ inline void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// thread-block clusters: rank inside the cluster, split barrier, stores into a
// peer CTA's shared memory (distributed shared memory)
__device__ inline uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ inline void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ inline void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ inline void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ inline void cluster_sync() { cluster_arrive(); cluster_wait(); }
__device__ inline void st_cluster_f32(const void* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ inline void st_cluster_s32(const void* local, uint32_t rank, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__device__ inline void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulate
__device__ inline void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D += A(16x8, row) * B(8x8, col)
__device__ inline void mma1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
// transpose an 8x8 b16 matrix held one 32-bit pair per lane
__device__ inline uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ inline uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// split (x, y) into fp16 hi + fp16 lo pairs so that hi + lo carries ~22 bits
__device__ inline void split_half2(float x, float y, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(x, y);
  float2 hf = __half22float2(h);
  __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ inline uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ inline uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ inline uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// launchers (host functions defined in the kernel .cu files)
// ---------------------------------------------------------------------------
cudaError_t launch_pack(const Layout& L, const dkv_factors& f, uint8_t* cache, uint32_t* err, cudaStream_t s);
cudaError_t launch_compress(const Layout& L, const __half* K, const __half* V, uint8_t* cache, uint8_t* ws,
                            uint32_t* err, cudaStream_t s);
size_t compress_ws_bytes(const Layout& L);
// compress source tokens [256 i, 256 i + 256) of K, V [units][T][d] into block blk0 + i, i < nblk
// (block record, router row, residual positions; nothing else of the cache is touched)
cudaError_t launch_compress_blocks(const Layout& L, const __half* K, const __half* V, int T, int blk0, int nblk,
                                   uint8_t* cache, uint32_t* err, cudaStream_t s);
// streaming append: the window's oldest 256 tokens -> block L.NB, then the window slides down by
// 256 tokens (L: the state before); new tokens into window slots [w0, w0 + take)
size_t append_ws_bytes(const Layout& L);
cudaError_t launch_append_compress(const Layout& L, uint8_t* cache, uint8_t* ws, uint32_t* err, cudaStream_t s);
cudaError_t launch_append_write(const Layout& L, const __half* Kn, const __half* Vn, int n_new, int i0, int take,
                                int w0, uint8_t* cache, cudaStream_t s);

// Decode workspace: [header 256 B][scheduler: 2 x u32][routed: i32 per unit and slot]
// [partials: per unit and item, m[8] l[8] o[8][d] in f32]
struct DecodePlan {
  int K_eff, n_wchunks, wchunk_tokens, n_items;
  size_t off_sched, off_routed, off_partials, ws_bytes;
};
DecodePlan plan_decode(const Layout& L, int n_q_heads, int n_kv_heads, int top_k);
cudaError_t launch_route(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                         const uint8_t* cache, uint8_t* ws, int32_t* routed_out, cudaStream_t s);
// out == nullptr: partials only (merge with launch_combine); otherwise the
// combine grid is launched right after (programmatic dependent launch)
cudaError_t launch_attend(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s);
// kernel launches launch_decode makes for this plan
int decode_launches(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads);
// the whole decode call: the router grid (not for the fragment layout when every
// block is routed), the attention grid and the combine grid
cudaError_t launch_decode(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, int32_t* routed_out,
                          cudaStream_t s);
// tcgen05 attention kernel (tensor-core cache layout)
bool tc_eligible(const Layout& L, int n_q_heads, int n_kv_heads);
int tc_window_tokens();
cudaError_t launch_attend_tc(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                             const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s);
// merge n_items partial records [m 8][l 8][o 8 x d] per unit into out (and lse)
cudaError_t launch_combine_records(int units, int n_items, int n_q_heads, int n_kv_heads, int d,
                                   const float* partials, float* out, float* lse, cudaStream_t s);
int sm_count();  // multiprocessors of the current device
// Diagnostic limits of the fragment-layout attention kernel (dkv_debug_set_limits):
// chunks a CTA's producer issues at most (negative: all) and polls of a bounded wait.
void debug_limits(int* stop_after, uint32_t* wait_polls);
void set_debug_limits(int stop_after, uint32_t wait_polls);
// whether the decode grids (attention, combine) are launched as programmatic dependents
bool programmatic_launch();
void set_programmatic_launch(bool on);
// Raise `func`'s dynamic shared-memory limit to at least `bytes` on the current
// device: once per (kernel, device), again only when a larger size is asked for.
// Thread-safe.
cudaError_t ensure_smem_limit(const void* func, size_t bytes);
// Ask for the largest shared-memory carveout for `func` on the current device,
// once per (kernel, device).  Thread-safe.
cudaError_t ensure_max_carveout(const void* func);
cudaError_t launch_combine(const Layout& L, const DecodePlan& P, int batch, int n_q_heads, int n_kv_heads,
                           const float* partials, float* out, float* lse, cudaStream_t s);

size_t dense_ws_bytes(int batch, int n_q_heads, int n_kv_heads, int d, int T);

// Block-sparse prefill: workspace [header][kbox: units x nb x 2d f32][qbar: units x nb x d f32]
// [routed: units x nb x K_eff i32]
struct PrefillPlan {
  int nb, K_eff;
  size_t off_kbox, off_qbar, off_routed, ws_bytes;
};
PrefillPlan plan_prefill(int batch, int n_kv_heads, int d, int T, int top_k);
cudaError_t launch_prefill(int batch, int n_q_heads, int n_kv_heads, int d, int T, int top_k, const __half* q,
                           const __half* K, const __half* V, float* out, float* lse, int32_t* routed_out, uint8_t* ws,
                           cudaStream_t s);
cudaError_t launch_dense(int batch, int n_q_heads, int n_kv_heads, int d, int T, const __half* q, const __half* K,
                         const __half* V, float* out, float* lse, uint8_t* ws, uint32_t* err, cudaStream_t s);

}  // namespace dkv
