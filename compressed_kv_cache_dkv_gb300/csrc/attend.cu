// Block + window attention of the DKV decode path (persistent kernel).
//
// Work items of one call: every (unit, routed block) and every (unit, chunk of
// the exact recency window).  A fixed grid of about two CTAs per SM takes
// items one after the other (the first statically, the rest from an atomic
// counter).  Half of the window chunks come first (they need nothing from the
// router, so they overlap its grid), then the routed blocks, then the other
// half, which fills the tail left by the larger block items.  Warp 4 is the producer: its lane 0 decodes items and streams their
// packed bytes, chunk by chunk, into a ring of shared-memory slots with 1-D TMA
// bulk copies (cp.async.bulk + mbarrier complete_tx), running ahead into the
// next item while the consumers finish the current one.  Warps 0-3 are the
// consumers; every matrix product runs on the tensor cores through
// mma.sync m16n8k16 / m16n8k8 (fp16 operands, fp32 accumulate) with the tokens
// (or the head dimension) in M and the GQA group in N = 8.
//
// Per routed block ("Low-Rank Space Query Scoring" / "Flash-Style LSE
// Combine", Differential-KV README, section "Core Architecture & Paper
// Overview"; DKV Zenodo abstract):
//   z_g   = V_K (c q_g)                          (per block, r numbers per query)
//   s_0   = c q_g . a_k                          (the anchor: U row 0 is zero)
//   s_i   = c q_g . a_k + U_i . z_g,  i not in S (K is never materialised)
//   s_j   = c q_g . k_j,              j in S     (exact residual rows)
//   acc_g = (sum_lowrank p) a_v + (sum_lowrank p_i U_i) V_V + sum_S p_j v_j
// emitted as a partial (m, l, acc) in base-2 units; the combine kernel merges
// a unit's partials with an fp32 log-sum-exp reduction.  Scores are kept in fp32; the fp32 operands of a product (z, p,
// w) are split into an fp16 pair hi + lo so the tensor-core products carry
// about 22 bits.
#include <float.h>
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kConsumers = 4;          // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kUTok = 64;              // U rows per chunk
constexpr int kWindowChunk = 256;      // window tokens per work item
constexpr int kMaxSlots = 8;
constexpr int kIQ = 3;                 // item descriptors in flight between producer and consumers

struct AttendArgs {
  Layout L;
  int G, Hq, Hkv, K_eff, n_items, n_wchunks, n_wfront, total, nslot, slot_bytes, xtok;
  float scale_log2;  // log2(e) / sqrt(d)
  const __half* q;
  const uint8_t* cache;
  const int32_t* routed;
  float* partials;
  uint32_t* err;
  uint32_t* sched;     // [0] next dynamic item, [1] CTAs done fetching
};

// One work item, as decoded by the producer and handed to the consumers.
struct ItemDesc {
  int stop;              // no more items for this CTA
  int is_block;
  int ok;                // routed index in range
  int u, item;           // unit, item index inside the unit's partials
  int n_chunks, n_u, n_x;
  int tok0, ntok, nvalid;
  uint32_t k0;           // global ring index of the item's first chunk
  uint64_t base;         // block record or window offset (bytes from the cache base)
};

struct Chunk {
  uint64_t src;   // byte offset from the cache base
  uint32_t bytes;
  int kind;       // 0 head, 1 U, 2 exact, 3 V_V
  int tok0;       // first token (U row / residual row / window token)
  int ntok;       // stored tokens in the chunk (multiple of 8)
};

__device__ inline Chunk item_chunk(const AttendArgs& a, const ItemDesc& it, int k) {
  const Layout& L = a.L;
  Chunk c;
  if (it.is_block) {
    if (k == 0) {
      c.src = it.base; c.bytes = (uint32_t)L.off_u; c.kind = 0; c.tok0 = 0; c.ntok = 0;
    } else if (k <= it.n_u) {
      const int t0 = (k - 1) * kUTok;
      c.src = it.base + L.off_u + (uint64_t)t0 * 2 * L.r8;
      c.bytes = (uint32_t)(kUTok * 2 * L.r8); c.kind = 1; c.tok0 = t0; c.ntok = kUTok;
    } else if (k <= it.n_u + it.n_x) {
      const int t0 = (k - 1 - it.n_u) * a.xtok;
      const int n = min(a.xtok, L.R8 - t0);
      c.src = it.base + L.off_res + (uint64_t)t0 * 4 * L.d;
      c.bytes = (uint32_t)(n * 4 * L.d); c.kind = 2; c.tok0 = t0; c.ntok = n;
    } else {
      c.src = it.base + L.off_vv; c.bytes = (uint32_t)(2 * L.r8 * L.d); c.kind = 3; c.tok0 = 0; c.ntok = 0;
    }
  } else {
    const int t0 = it.tok0 + k * a.xtok;
    const int n = min(a.xtok, it.tok0 + it.ntok - t0);
    c.src = it.base + (uint64_t)t0 * 4 * L.d;
    c.bytes = (uint32_t)(n * 4 * L.d); c.kind = 2; c.tok0 = t0; c.ntok = n;
  }
  return c;
}

__device__ inline int chunk_owner(const ItemDesc& it, int k) {
  if (it.is_block) {
    if (k == 0 || k == it.n_chunks - 1) return -1;  // all consumer warps
    return (k - 1) % kConsumers;
  }
  return k % kConsumers;
}

// Global item index -> item: n_wfront window chunks of every unit, the routed
// blocks, then the remaining window chunks; consecutive indices belong to
// different units.
__device__ inline bool needs_route(const AttendArgs& a, int gi) {
  const int nfront = a.n_wfront * a.L.units;
  return gi >= nfront && gi < nfront + a.K_eff * a.L.units;
}
__device__ inline ItemDesc decode_item(const AttendArgs& a, int gi) {
  const Layout& L = a.L;
  ItemDesc it;
  it.stop = 0;
  it.ok = 1;
  const int nfront = a.n_wfront * L.units, nblk = a.K_eff * L.units;
  const uint64_t unit_stride = L.unit_stride;
  if (gi < nfront || gi >= nfront + nblk) {
    const int wc = gi < nfront ? gi / L.units : a.n_wfront + (gi - nfront - nblk) / L.units;
    it.u = gi % L.units;
    it.item = a.K_eff + wc;
    it.is_block = 0;
    it.n_u = 0;
    it.tok0 = wc * kWindowChunk;
    it.ntok = min(kWindowChunk, L.W16 - it.tok0);
    it.n_x = (it.ntok + a.xtok - 1) / a.xtok;
    it.n_chunks = it.n_x;
    it.base = (uint64_t)it.u * unit_stride + L.off_window;
    it.nvalid = L.W;
  } else {
    const int bi = gi - nfront;
    const int slot = bi / L.units;
    it.u = bi % L.units;
    it.item = slot;
    int blk = a.routed[it.u * a.K_eff + slot];
    if (blk < 0 || blk >= L.NB) {
      it.ok = 0;
      raise_error(a.err, DKV_DEVERR_INDEX);
      blk = 0;
    }
    it.is_block = 1;
    it.n_u = 256 / kUTok;
    it.n_x = (L.R8 + a.xtok - 1) / a.xtok;
    it.n_chunks = 1 + it.n_u + it.n_x + 1;
    it.base = (uint64_t)it.u * unit_stride + L.off_blocks + (uint64_t)blk * L.block_stride;
    it.tok0 = 0; it.ntok = 0; it.nvalid = L.R;
  }
  return it;
}

__device__ inline float warp_max_rows(float v) {  // max over lanes with the same lane%4
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ inline float warp_sum_rows(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// power-of-two factor that brings max |x| under 2^14 (keeps fp16 hi/lo splits finite)
__device__ inline float pow2_down(float mx) {
  if (!(mx > 16384.f)) return 1.f;
  int e;
  frexpf(mx, &e);
  return ldexpf(1.f, 14 - e);
}

// Operand registers of one 16x16 fp16 tile stored in fragment order: a full
// tile holds 16 bytes per lane (at lane * 16); a half tile (8 rows or 8 columns)
// 8 bytes per lane (at lane * 8).  Both are read with one aligned 16-byte load;
// for a half tile each lane keeps its own 8 bytes in .x, .y (.z, .w are not
// meaningful and the caller zeroes what it does not use).
__device__ inline uint4 ld_tile(uint32_t base, int lane, bool full) {
  const uint4 v = lds128(base + (uint32_t)(full ? lane * 16 : (lane >> 1) * 16));
  const bool odd = (lane & 1) != 0;
  return make_uint4(full ? v.x : (odd ? v.z : v.x), full ? v.y : (odd ? v.w : v.y), v.z, v.w);
}

// Position in the ring of chunk slots.  Every consumer warp and the producer
// walk the chunks of all items in the same order, so each keeps its own cursor.
struct Ring {
  int slot;
  uint32_t use;  // how many times the slot ring has wrapped (parity = use & 1)
  __device__ inline void next(int nslot) {
    if (++slot == nslot) { slot = 0; ++use; }
  }
};

// Online-softmax statistics of one consumer warp for the two C-fragment
// columns it owns (g = 2t, 2t+1): running max m (base 2) and normaliser l.
struct Stat {
  float m[2], l[2];
};

__device__ inline void tile_max(const float (&s)[4], float& mx0, float& mx1) {
  mx0 = fmaxf(mx0, fmaxf(s[0], s[2]));
  mx1 = fmaxf(mx1, fmaxf(s[1], s[3]));
}

// Move the running maximum to include (mx0, mx1); returns the factors that
// rescale everything accumulated so far, and the subtrahends for the new p.
__device__ inline void stat_update(Stat& st, float mx0, float mx1, float& sc0, float& sc1, float& ms0, float& ms1) {
  mx0 = warp_max_rows(mx0);
  mx1 = warp_max_rows(mx1);
  const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
  ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
  ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
  sc0 = fast_exp2(st.m[0] - ms0);  // 2^(-inf) = 0
  sc1 = fast_exp2(st.m[1] - ms1);
  st.m[0] = mn0;
  st.m[1] = mn1;
  st.l[0] *= sc0;
  st.l[1] *= sc1;
}

__device__ inline void probs(const float (&s)[4], float ms0, float ms1, bool gv0, bool gv1, float (&p)[4], Stat& st) {
  p[0] = gv0 ? fast_exp2(s[0] - ms0) : 0.f;
  p[1] = gv1 ? fast_exp2(s[1] - ms1) : 0.f;
  p[2] = gv0 ? fast_exp2(s[2] - ms0) : 0.f;
  p[3] = gv1 ? fast_exp2(s[3] - ms1) : 0.f;
  st.l[0] += p[0] + p[2];
  st.l[1] += p[1] + p[3];
}

// P (C-fragment layout, rows = tokens) -> B fragments (k = tokens, n = group) hi/lo
__device__ inline void p_to_b(const float (&p)[4], uint32_t& bh0, uint32_t& bl0, uint32_t& bh1, uint32_t& bl1) {
  uint32_t h01, l01, h23, l23;
  split_half2(p[0], p[1], h01, l01);
  split_half2(p[2], p[3], h23, l23);
  bh0 = movtrans(h01); bl0 = movtrans(l01);
  bh1 = movtrans(h23); bl1 = movtrans(l23);
}

// shared-memory carve-up (the host computes the same sizes in launch_attend)
struct Smem {
  uint8_t* slots;
  uint64_t *full, *empty, *iq_full, *iq_empty;
  ItemDesc* iqd;
  __half* qbuf;      // [kIQ][8][D + 8] the item's query rows (padded rows)
  float2* zbuf;      // [RT*2][32] z^T C fragments, one n-tile per warp in turn
  float* obw;        // [4][D][8]  per-warp exact-token accumulators, merged in place
  float* wbw;        // [4][RT*16][8] per-warp low-rank w, merged in place
  float* basebuf;    // [4][8]
  float* stat;       // [4 warps][4][8]
  float* fin;        // [12][8] merged statistics and per-warp scales
  uint32_t* maskbuf; // [8]
  int* flag;         // [4]
  __half* av;        // [D]
};

template <int D, int RT>
__device__ inline Smem carve(uint8_t* smem, const AttendArgs& a) {
  Smem s;
  s.slots = smem;
  uint8_t* p = smem + (size_t)a.nslot * a.slot_bytes;
  s.full = reinterpret_cast<uint64_t*>(p);
  s.empty = s.full + kMaxSlots;
  s.iq_full = s.empty + kMaxSlots;
  s.iq_empty = s.iq_full + kIQ;
  s.iqd = reinterpret_cast<ItemDesc*>(s.iq_empty + kIQ);
  s.qbuf = reinterpret_cast<__half*>((reinterpret_cast<uintptr_t>(s.iqd + kIQ) + 15) & ~uintptr_t(15));
  s.zbuf = reinterpret_cast<float2*>(s.qbuf + kIQ * 8 * (D + 8));
  s.obw = reinterpret_cast<float*>(s.zbuf + RT * 2 * 32);
  s.wbw = s.obw + kConsumers * D * 8;
  s.basebuf = s.wbw + kConsumers * RT * 16 * 8;
  s.stat = s.basebuf + 32;
  s.fin = s.stat + 128;
  s.maskbuf = reinterpret_cast<uint32_t*>(s.fin + 96);
  s.flag = reinterpret_cast<int*>(s.maskbuf + 8);
  s.av = reinterpret_cast<__half*>(s.flag + 4);
  return s;
}

template <int D, int RT>
__host__ __device__ inline size_t smem_extra() {
  return 4 * kMaxSlots * 8 + kIQ * sizeof(ItemDesc) + 16 + (size_t)kIQ * 8 * (D + 8) * 2 + (size_t)RT * 2 * 32 * 8 +
         (size_t)kConsumers * D * 8 * 4 +
         (size_t)kConsumers * RT * 16 * 8 * 4 + (32 + 128 + 96) * 4 + 32 + 16 + (size_t)D * 2 + 128;
}

// ---------------------------------------------------------------------------
// consumers: one item
// ---------------------------------------------------------------------------
template <int D>
__device__ inline void load_qb(uint32_t qrow, bool valid, int t, uint32_t (&qb)[D / 16][2]) {
#pragma unroll
  for (int kt = 0; kt < D / 16; ++kt) {
    qb[kt][0] = valid ? lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u) : 0u;
    qb[kt][1] = valid ? lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u) : 0u;
  }
}

// One work item, processed by the four consumer warps.  A routed block runs in
// two phases whose register state never coexists: the low-rank phase (head:
// base score and z; U chunks; merge of the four warps' low-rank state into
// shared memory) and the exact phase (residual rows, merged the same way),
// followed by the low-rank value product V_V^T w and the item's partial record.
// A window item has the exact phase only.  The item's query slot is released
// once every warp holds the query fragments of its exact phase.
template <int D, int RT>
__device__ __forceinline__ void consume_item(const AttendArgs& a, const Smem& sm, const ItemDesc& it, Ring& rc,
                                             int iq) {
  const Layout& L = a.L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = lane & 3, gq = lane >> 2;
  const int tid = threadIdx.x;
  const int r8 = L.r8;
  const int nkk = r8 >> 4;                 // full 16-wide k tiles of r
  const bool rtail = (r8 & 15) != 0;       // one 8-wide tail
  const int nrt = nkk + (rtail ? 1 : 0);   // r tiles
  constexpr int KT = D / 16;               // 16-wide k tiles of the head dimension
  const int G = a.G;
  const bool gv0 = (2 * t) < G, gv1 = (2 * t + 1) < G;
  const float slog2 = a.scale_log2;
  const uint32_t slot0 = smem_u32(sm.slots);
  const uint32_t qrow = smem_u32(sm.qbuf + ((size_t)iq * 8 + gq) * (D + 8));
  const bool qvalid = gq < G;
  float* obw = sm.obw;
  float* wbw = sm.wbw;
  float* stat = sm.stat;  // [4 warps][mL 8 | lL 8 | mX 8 | lX 8]
  float* fin = sm.fin;    // [ML 8 | LL 8 | MX 8 | LX 8]
  float* scl = fin + 32;  // [4 warps][8]: low-rank scale factors
  float* scx = fin + 64;  // [4 warps][8]: exact-token scale factors
  bool ok = it.ok != 0;
  int k = 0;              // chunk index inside the item

  if (it.is_block) {
    // ======================= low-rank phase
    float base0, base1;        // c q_g . a_k in base-2 units, columns 2t, 2t+1
    float us0, us1;            // power-of-two unscale of z, columns 2t, 2t+1
    uint32_t zh[RT][2], zl[RT][2];  // z as B fragments (k = r, n = group), hi and lo
    {
      // ---------------- head chunk: anchors, residual mask, V_K -> base and z
      uint32_t qb[KT][2];
      load_qb<D>(qrow, qvalid, t, qb);
      const int hs = rc.slot;
      ok = mbar_wait(&sm.full[hs], rc.use & 1u, a.err) && ok;
      rc.next(a.nslot);
      const uint8_t* head = sm.slots + (size_t)hs * a.slot_bytes;
      {
        // q . a_k: the warps split the head dimension, partial sums meet in shared memory
        const __half* ak = reinterpret_cast<const __half*>(head);
        constexpr int KPW = KT / kConsumers > 0 ? KT / kConsumers : 1;
        float part = 0.f;
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
          if (kt / KPW == warp) {  // compile-time index: q fragments stay in registers
            const float2 qf0 = __half22float2(*reinterpret_cast<const __half2*>(&qb[kt][0]));
            const float2 qf1 = __half22float2(*reinterpret_cast<const __half2*>(&qb[kt][1]));
            const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(ak + 16 * kt + 2 * t));
            const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(ak + 16 * kt + 8 + 2 * t));
            part += qf0.x * a0.x + qf0.y * a0.y + qf1.x * a1.x + qf1.y * a1.y;
          }
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (t == 0) sm.basebuf[warp * 8 + gq] = part;
      }
      if (warp == 0) {
        for (int j = lane; j < D; j += 32) sm.av[j] = reinterpret_cast<const __half*>(head)[D + j];
        if (lane < 8) sm.maskbuf[lane] = reinterpret_cast<const uint32_t*>(head + L.off_mask)[lane];
      }
      // z^T = q^T V_K^T : n-tiles of 8 r-rows split across warps, shared through zbuf
      const uint32_t vk = smem_u32(head) + (uint32_t)L.off_vk;
      for (int nt = warp; nt < (r8 >> 3); nt += kConsumers) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        uint4 bv[D / 32];
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) bv[kp] = lds128(vk + (uint32_t)(nt * 8 * D * 2 + kp * 512 + lane * 16));
#pragma unroll
        for (int kp = 0; kp < D / 32; ++kp) {
          mma16816(c, qb[2 * kp][0], 0u, qb[2 * kp][1], 0u, bv[kp].x, bv[kp].y);
          mma16816(c, qb[2 * kp + 1][0], 0u, qb[2 * kp + 1][1], 0u, bv[kp].z, bv[kp].w);
        }
        sm.zbuf[nt * 32 + lane] = make_float2(c[0] * slog2, c[1] * slog2);
      }
      named_bar_sync(1, kConsumers * 32);  // basebuf, zbuf, av, mask are written; the head slot is read
      if (lane == 0) mbar_arrive(&sm.empty[hs]);
      float zf[RT][4];
#pragma unroll
      for (int kk = 0; kk < RT; ++kk) {
        float2 z0 = make_float2(0.f, 0.f), z1 = make_float2(0.f, 0.f);
        if (kk < nrt) {
          z0 = sm.zbuf[(2 * kk) * 32 + lane];
          if (2 * kk + 1 < (r8 >> 3)) z1 = sm.zbuf[(2 * kk + 1) * 32 + lane];
        }
        zf[kk][0] = z0.x; zf[kk][1] = z0.y; zf[kk][2] = z1.x; zf[kk][3] = z1.y;
      }
      const float* bb = sm.basebuf;
      base0 = (bb[2 * t] + bb[8 + 2 * t] + bb[16 + 2 * t] + bb[24 + 2 * t]) * slog2;
      base1 = (bb[2 * t + 1] + bb[9 + 2 * t] + bb[17 + 2 * t] + bb[25 + 2 * t]) * slog2;
      // z B fragments: b0 = z[16kk + 2t, +1][gq] (C fragment c0, c1 of n-tile 2kk), b1 from n-tile 2kk+1
      float zmax = 0.f;
#pragma unroll
      for (int kk = 0; kk < RT; ++kk)
        zmax = fmaxf(zmax, fmaxf(fmaxf(fabsf(zf[kk][0]), fabsf(zf[kk][1])), fmaxf(fabsf(zf[kk][2]), fabsf(zf[kk][3]))));
      zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, 1));
      zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, 2));
      const float zsc = pow2_down(zmax);  // for g = gq
#pragma unroll
      for (int kk = 0; kk < RT; ++kk) {
        split_half2(zf[kk][0] * zsc, zf[kk][1] * zsc, zh[kk][0], zl[kk][0]);
        split_half2(zf[kk][2] * zsc, zf[kk][3] * zsc, zh[kk][1], zl[kk][1]);
      }
      us0 = 1.f / __shfl_sync(0xffffffffu, zsc, 8 * t);
      us1 = 1.f / __shfl_sync(0xffffffffu, zsc, 8 * t + 4);
    }
    // ---------------- U chunks, round-robin over warps (every warp observes every chunk in order)
    Stat sL;  // its normaliser sums p over the low-rank tokens, anchor included
    sL.m[0] = sL.m[1] = -INFINITY;
    sL.l[0] = sL.l[1] = 0.f;
    float w[RT][4];
#pragma unroll
    for (int i = 0; i < RT; ++i) w[i][0] = w[i][1] = w[i][2] = w[i][3] = 0.f;
    for (k = 1; k <= it.n_u; ++k) {
      const int slot = rc.slot;
      const bool have = mbar_wait(&sm.full[slot], rc.use & 1u, a.err);
      rc.next(a.nslot);
      if (chunk_owner(it, k) == warp) {
        ok = ok && have;
        const int tok0 = (k - 1) * kUTok;
        const uint32_t sb = slot0 + (uint32_t)(slot * a.slot_bytes);
        if (have) {
          // ---- pass 1: every score of the chunk, then one rescale.  A half-width last
          // k tile (r8 % 16 == 8) has its missing half zeroed.
          constexpr int MT = kUTok / 16;
          const uint32_t mbase = smem_u32(sm.maskbuf) + (uint32_t)(tok0 >> 5) * 4u;
          const uint32_t mw0 = lds32(mbase), mw1 = lds32(mbase + 4u);  // residual rows among the chunk's 64
          float s[MT][4];
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t tb = sb + (uint32_t)(mt * 16 * r8 * 2);
            uint4 uv[RT];
#pragma unroll
            for (int kk = 0; kk < RT; ++kk) uv[kk] = ld_tile(tb + (uint32_t)(kk * 512), lane, kk < nkk);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < RT; ++kk) {
              if (kk < nrt) {
                const bool full = kk < nkk;
                // a half tile holds (x, y) = rows gq and gq + 8 of k 2t..2t+1 only
                const uint32_t a2 = full ? uv[kk].z : 0u, a3 = full ? uv[kk].w : 0u;
                mma16816(acc, uv[kk].x, uv[kk].y, a2, a3, zh[kk][0], zh[kk][1]);
                mma16816(acc, uv[kk].x, uv[kk].y, a2, a3, zl[kk][0], zl[kk][1]);
              }
            }
            const uint32_t wsel = mt < 2 ? mw0 : mw1;
            const bool m0 = (wsel >> ((mt & 1) * 16 + gq)) & 1u;
            const bool m1 = (wsel >> ((mt & 1) * 16 + gq + 8)) & 1u;
            s[mt][0] = m0 ? -INFINITY : fmaf(acc[0], us0, base0);
            s[mt][1] = m0 ? -INFINITY : fmaf(acc[1], us1, base1);
            s[mt][2] = m1 ? -INFINITY : fmaf(acc[2], us0, base0);
            s[mt][3] = m1 ? -INFINITY : fmaf(acc[3], us1, base1);
            tile_max(s[mt], mx0, mx1);
          }
          float sc0, sc1, ms0, ms1;
          stat_update(sL, mx0, mx1, sc0, sc1, ms0, ms1);
#pragma unroll
          for (int i = 0; i < RT; ++i) { w[i][0] *= sc0; w[i][1] *= sc1; w[i][2] *= sc0; w[i][3] *= sc1; }
          // ---- pass 2: p, and w += U^T p (U fragments reloaded, transposed in registers)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t tb = sb + (uint32_t)(mt * 16 * r8 * 2);
            uint4 uv[RT];
#pragma unroll
            for (int mr = 0; mr < RT; ++mr) uv[mr] = ld_tile(tb + (uint32_t)(mr * 512), lane, mr < nkk);
            float p[4];
            probs(s[mt], ms0, ms1, gv0, gv1, p, sL);
            uint32_t bh0, bl0, bh1, bl1;
            p_to_b(p, bh0, bl0, bh1, bl1);
#pragma unroll
            for (int mr = 0; mr < RT; ++mr) {
              if (mr < nrt) {
                const bool full = mr < nkk;
                // U^T tile (m = r, k = tokens): a half tile only has the first r half
                const uint32_t A0 = movtrans(uv[mr].x), A2 = movtrans(uv[mr].y);
                const uint32_t T2 = movtrans(uv[mr].z), T3 = movtrans(uv[mr].w);
                const uint32_t A1 = full ? T2 : 0u, A3 = full ? T3 : 0u;
                mma16816(w[mr], A0, A1, A2, A3, bh0, bh1);
                mma16816(w[mr], A0, A1, A2, A3, bl0, bl1);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    // ---------------- merge the low-rank state of the four warps (w and its statistics)
    sL.l[0] = warp_sum_rows(sL.l[0]);
    sL.l[1] = warp_sum_rows(sL.l[1]);
    if (lane < 4) {
      float* sw = stat + warp * 32;
      sw[2 * t] = sL.m[0]; sw[2 * t + 1] = sL.m[1];
      sw[8 + 2 * t] = sL.l[0]; sw[8 + 2 * t + 1] = sL.l[1];
    }
#pragma unroll
    for (int mr = 0; mr < RT; ++mr) {
      if (mr < nrt) {
        const int r0 = mr * 16 + gq;
        float* w0 = wbw + ((size_t)warp * RT * 16 + r0) * 8 + 2 * t;
        w0[0] = w[mr][0]; w0[1] = w[mr][1];
        if (r0 + 8 < r8) { w0[64] = w[mr][2]; w0[65] = w[mr][3]; }
      }
    }
    named_bar_sync(1, kConsumers * 32);
    if (tid < 8) {
      const int g = tid;
      float ML = -INFINITY;
      for (int wi = 0; wi < kConsumers; ++wi) ML = fmaxf(ML, stat[wi * 32 + g]);
      const float mls = ML == -INFINITY ? 0.f : ML;
      float LL = 0.f;
      for (int wi = 0; wi < kConsumers; ++wi) {
        const float fl = fast_exp2(stat[wi * 32 + g] - mls);
        scl[wi * 8 + g] = fl;
        LL += stat[wi * 32 + 8 + g] * fl;
      }
      fin[g] = ML; fin[8 + g] = LL;
    }
    named_bar_sync(1, kConsumers * 32);
    for (int e = tid; e < r8 * 8; e += kConsumers * 32) {  // in place, into warp 0's area
      const int r = e >> 3, g = e & 7;
      float v = 0.f;
#pragma unroll
      for (int wi = 0; wi < kConsumers; ++wi) v += scl[wi * 8 + g] * wbw[((size_t)wi * RT * 16 + r) * 8 + g];
      wbw[(size_t)r * 8 + g] = v;
    }
  }

  // ======================= exact phase (residual rows, or a window item)
  {
    uint32_t qb[KT][2];
    load_qb<D>(qrow, qvalid, t, qb);
    Stat sX;
    sX.m[0] = sX.m[1] = -INFINITY;
    sX.l[0] = sX.l[1] = 0.f;
    float o[KT][4];
#pragma unroll
    for (int i = 0; i < KT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const int k_last = it.is_block ? it.n_chunks - 2 : it.n_chunks - 1;
    for (; k <= k_last; ++k) {
      const int slot = rc.slot;
      const bool have = mbar_wait(&sm.full[slot], rc.use & 1u, a.err);
      rc.next(a.nslot);
      if (chunk_owner(it, k) == warp) {
        ok = ok && have;
        const Chunk c = item_chunk(a, it, k);
        const uint32_t sb = slot0 + (uint32_t)(slot * a.slot_bytes);
        if (have) {
          // ---- pass 1: scores of the chunk's 16-token groups.  A group holds 16, 8 (the
          // last residual group when R8 % 16 == 8) or 0 tokens; all three share one code
          // path (operands of missing rows are zeroed).
          constexpr int MG = 16384 / (64 * D);  // 16-token groups per chunk (2 at d = 128, 4 at d = 64)
          float s[MG][4];
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int gi = 0; gi < MG; ++gi) {
            const int in_g = max(0, min(16, c.ntok - gi * 16));
            const bool full = in_g == 16, any = in_g > 0;
            const uint32_t gb = sb + (uint32_t)(gi * 64 * D);
            const uint32_t kst = full ? 512u : 256u;
            uint4 kv[KT];
#pragma unroll
            for (int kt = 0; kt < KT; ++kt) kv[kt] = ld_tile(gb + (uint32_t)kt * kst, lane, full);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kt = 0; kt < KT; ++kt) {
              // K tile (m = tokens, k = d): a half group has only rows gq: (x, y) = k 2t.., 2t + 8..
              const uint4 v = kv[kt];
              const uint32_t a0 = any ? v.x : 0u, a1 = full ? v.y : 0u, a2 = full ? v.z : (any ? v.y : 0u),
                             a3 = full ? v.w : 0u;
              mma16816(acc, a0, a1, a2, a3, qb[kt][0], qb[kt][1]);
            }
            const int tk0 = c.tok0 + gi * 16 + gq, tk1 = tk0 + 8;
            const bool v0 = tk0 < it.nvalid && (gq < in_g);
            const bool v1 = tk1 < it.nvalid && (gq + 8 < in_g);
            s[gi][0] = v0 ? acc[0] * slog2 : -INFINITY;
            s[gi][1] = v0 ? acc[1] * slog2 : -INFINITY;
            s[gi][2] = v1 ? acc[2] * slog2 : -INFINITY;
            s[gi][3] = v1 ? acc[3] * slog2 : -INFINITY;
            tile_max(s[gi], mx0, mx1);
          }
          float sc0, sc1, ms0, ms1;
          stat_update(sX, mx0, mx1, sc0, sc1, ms0, ms1);
#pragma unroll
          for (int i = 0; i < KT; ++i) { o[i][0] *= sc0; o[i][1] *= sc1; o[i][2] *= sc0; o[i][3] *= sc1; }
          // ---- pass 2: p, and o += V^T p
#pragma unroll
          for (int gi = 0; gi < MG; ++gi) {
            const int in_g = max(0, min(16, c.ntok - gi * 16));
            const bool full = in_g == 16, any = in_g > 0;
            const uint32_t gb = sb + (uint32_t)(gi * 64 * D);
            const uint32_t kst = full ? 512u : 256u;
            const uint32_t vb = gb + (uint32_t)(in_g * D * 2);
            uint4 vv4[KT];
#pragma unroll
            for (int md = 0; md < KT; ++md) vv4[md] = ld_tile(vb + (uint32_t)md * kst, lane, full);
            float p[4];
            probs(s[gi], ms0, ms1, gv0, gv1, p, sX);
            uint32_t bh0, bl0, bh1, bl1;
            p_to_b(p, bh0, bl0, bh1, bl1);
#pragma unroll
            for (int md = 0; md < KT; ++md) {
              // V^T tile (m = d, k = tokens): a half group holds k 0..7 only
              const uint4 v = vv4[md];
              const uint32_t a0 = any ? v.x : 0u, a1 = any ? v.y : 0u, a2 = full ? v.z : 0u,
                             a3 = full ? v.w : 0u;
              mma16816(o[md], a0, a1, a2, a3, bh0, bh1);
              mma16816(o[md], a0, a1, a2, a3, bl0, bl1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    // ---------------- merge the exact state of the four warps
    sX.l[0] = warp_sum_rows(sX.l[0]);
    sX.l[1] = warp_sum_rows(sX.l[1]);
    if (lane < 4) {
      float* sw = stat + warp * 32;
      sw[16 + 2 * t] = sX.m[0]; sw[16 + 2 * t + 1] = sX.m[1];
      sw[24 + 2 * t] = sX.l[0]; sw[24 + 2 * t + 1] = sX.l[1];
    }
#pragma unroll
    for (int md = 0; md < KT; ++md) {
      float* o0 = obw + ((size_t)warp * D + md * 16 + gq) * 8 + 2 * t;
      o0[0] = o[md][0]; o0[1] = o[md][1]; o0[64] = o[md][2]; o0[65] = o[md][3];
    }
  }
  named_bar_sync(1, kConsumers * 32);
  // every warp holds its query fragments: the producer may reuse this item's query slot
  if (warp == 0 && lane == 0) mbar_arrive(&sm.iq_empty[iq]);
  if (tid < 8) {
    const int g = tid;
    float MX = -INFINITY;
    for (int wi = 0; wi < kConsumers; ++wi) MX = fmaxf(MX, stat[wi * 32 + 16 + g]);
    const float mxs = MX == -INFINITY ? 0.f : MX;
    float LX = 0.f;
    for (int wi = 0; wi < kConsumers; ++wi) {
      const float fx = fast_exp2(stat[wi * 32 + 16 + g] - mxs);
      scx[wi * 8 + g] = fx;
      LX += stat[wi * 32 + 24 + g] * fx;
    }
    fin[16 + g] = MX; fin[24 + g] = LX;
    if (!it.is_block) { fin[g] = -INFINITY; fin[8 + g] = 0.f; }  // no low-rank part
  }
  named_bar_sync(1, kConsumers * 32);
  // merge the warps' exact accumulators in place (into warp 0's area), one element per thread
  for (int e = tid; e < D * 8; e += kConsumers * 32) {
    const int d = e >> 3, g = e & 7;
    float v = 0.f;
#pragma unroll
    for (int wi = 0; wi < kConsumers; ++wi) v += scx[wi * 8 + g] * obw[((size_t)wi * D + d) * 8 + g];
    obw[(size_t)d * 8 + g] = v;
  }
  named_bar_sync(1, kConsumers * 32);

  float* rec = a.partials + ((size_t)it.u * a.n_items + it.item) * (16 + 8 * D);
  // final partial: M = max(M_L, M_X); o = 2^(M_L - M) (V_V^T w + L_L a_v) + 2^(M_X - M) o_X
  auto final_stats = [&](int g, float& aL, float& aX, float& M) {
    const float ML = fin[g], MX = fin[16 + g];
    M = fmaxf(ML, MX);
    const float ms = M == -INFINITY ? 0.f : M;
    aL = fast_exp2(ML - ms);
    aX = fast_exp2(MX - ms);
  };
  if (tid < 8) {
    float aL, aX, M;
    final_stats(tid, aL, aX, M);
    rec[tid] = ok ? M : -INFINITY;
    rec[8 + tid] = ok ? aL * fin[8 + tid] + aX * fin[24 + tid] : 0.f;
  }
  if (it.is_block) {
    // ---------------- low-rank value: V_V^T w (+ L_L a_v), combined with the exact part
    const int vs = rc.slot;
    ok = mbar_wait(&sm.full[vs], rc.use & 1u, a.err) && ok;
    rc.next(a.nslot);
    const uint32_t vv = slot0 + (uint32_t)(vs * a.slot_bytes);
    // merged w as B fragments: b0 = w[16kk + 2t, +1][gq], b1 = w[16kk + 8 + 2t, +1][gq]
    float wf[RT][4];
    float wmax = 0.f;
#pragma unroll
    for (int kk = 0; kk < RT; ++kk) {
      wf[kk][0] = wf[kk][1] = wf[kk][2] = wf[kk][3] = 0.f;
      if (kk < nrt) {
        const int r0 = 16 * kk + 2 * t;
        wf[kk][0] = wbw[r0 * 8 + gq];
        wf[kk][1] = wbw[(r0 + 1) * 8 + gq];
        if (r0 + 8 < r8) { wf[kk][2] = wbw[(r0 + 8) * 8 + gq]; wf[kk][3] = wbw[(r0 + 9) * 8 + gq]; }
      }
      wmax = fmaxf(wmax, fmaxf(fmaxf(fabsf(wf[kk][0]), fabsf(wf[kk][1])), fmaxf(fabsf(wf[kk][2]), fabsf(wf[kk][3]))));
    }
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, 1));
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, 2));
    const float wsc2 = pow2_down(wmax);
    uint32_t wh[RT][2], wl[RT][2];
#pragma unroll
    for (int kk = 0; kk < RT; ++kk) {
      split_half2(wf[kk][0] * wsc2, wf[kk][1] * wsc2, wh[kk][0], wl[kk][0]);
      split_half2(wf[kk][2] * wsc2, wf[kk][3] * wsc2, wh[kk][1], wl[kk][1]);
    }
    const float wus0 = 1.f / __shfl_sync(0xffffffffu, wsc2, 8 * t);
    const float wus1 = 1.f / __shfl_sync(0xffffffffu, wsc2, 8 * t + 4);
    float aL0, aX0, M0, aL1, aX1, M1;
    final_stats(2 * t, aL0, aX0, M0);
    final_stats(2 * t + 1, aL1, aX1, M1);
    const float LL0 = fin[8 + 2 * t], LL1 = fin[8 + 2 * t + 1];
    for (int md = warp; md < KT; md += kConsumers) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t mb = vv + (uint32_t)(md * 16 * r8 * 2);
#pragma unroll
      for (int kk = 0; kk < RT; ++kk) {
        if (kk < nkk) {
          const uint4 v = lds128(mb + (uint32_t)(kk * 512 + lane * 16));
          mma16816(c, v.x, v.y, v.z, v.w, wh[kk][0], wh[kk][1]);
          mma16816(c, v.x, v.y, v.z, v.w, wl[kk][0], wl[kk][1]);
        } else if (kk == nkk && rtail) {
          const uint2 v = lds64(mb + (uint32_t)(kk * 512 + lane * 8));
          mma1688(c, v.x, v.y, wh[kk][0]);
          mma1688(c, v.x, v.y, wl[kk][0]);
        }
      }
      const int d0 = md * 16 + gq, d1 = d0 + 8;
      const float av0 = __half2float(sm.av[d0]), av1 = __half2float(sm.av[d1]);
      const float2 x0 = *reinterpret_cast<const float2*>(obw + d0 * 8 + 2 * t);
      const float2 x1 = *reinterpret_cast<const float2*>(obw + d1 * 8 + 2 * t);
      const float r00 = aL0 * (c[0] * wus0 + LL0 * av0) + aX0 * x0.x;
      const float r01 = aL1 * (c[1] * wus1 + LL1 * av0) + aX1 * x0.y;
      const float r10 = aL0 * (c[2] * wus0 + LL0 * av1) + aX0 * x1.x;
      const float r11 = aL1 * (c[3] * wus1 + LL1 * av1) + aX1 * x1.y;
      if (gv0) { rec[16 + (2 * t) * D + d0] = ok ? r00 : 0.f; rec[16 + (2 * t) * D + d1] = ok ? r10 : 0.f; }
      if (gv1) { rec[16 + (2 * t + 1) * D + d0] = ok ? r01 : 0.f; rec[16 + (2 * t + 1) * D + d1] = ok ? r11 : 0.f; }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[vs]);  // this warp is done with the V_V slot
  } else {
    for (int e = tid; e < G * D; e += kConsumers * 32) {
      const int g = e / D, d = e % D;
      rec[16 + g * D + d] = ok ? obw[d * 8 + g] : 0.f;
    }
  }
  named_bar_sync(1, kConsumers * 32);  // the merge buffers are reused by the next item
}

// ---------------------------------------------------------------------------
// the persistent kernel
// ---------------------------------------------------------------------------
template <int D, int RT>
__global__ void __launch_bounds__(kThreads, 2) attend_kernel(AttendArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Smem sm = carve<D, RT>(smem, a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // full: the producer's arrival + the bulk copy's bytes; empty: one arrival per
    // consumer warp, so no slot is refilled before every warp has seen its data
    // (a parity wait is unambiguous only while no barrier runs two phases ahead)
    for (int i = 0; i < a.nslot; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], kConsumers); }
    for (int i = 0; i < kIQ; ++i) { mbar_init(&sm.iq_full[i], 1); mbar_init(&sm.iq_empty[i], 1); }
    fence_mbar_init();
  }
  __syncthreads();

  griddep_launch();  // the combine grid may be scheduled now; it waits for this grid's completion

  // =========================== producer warp
  if (warp == kConsumers) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      Ring rp = {0, 0};        // next chunk slot
      uint32_t k = 0;          // global ring index of the next chunk
      bool waited = false;     // the router's grid (and the previous launch) has completed
      for (int j = 0;; ++j) {
        int gi = blockIdx.x;
        if (j > 0) {
          if (!waited) { griddep_wait(); waited = true; }
          gi = (int)gridDim.x + (int)atomicAdd(&a.sched[0], 1u);
        }
        const int iq = j % kIQ;
        if (j >= kIQ && !mbar_wait(&sm.iq_empty[iq], ((j / kIQ) - 1) & 1, a.err)) break;
        ItemDesc& dsc = sm.iqd[iq];
        if (gi >= a.total) {
          dsc.stop = 1;
          mbar_arrive(&sm.iq_full[iq]);
          // the last CTA out resets the dynamic scheduler for the next call
          if (j > 0 && atomicAdd(&a.sched[1], 1u) == gridDim.x - 1) {
            a.sched[0] = 0u;
            a.sched[1] = 0u;
          }
          break;
        }
        if (needs_route(a, gi) && !waited) { griddep_wait(); waited = true; }
        ItemDesc it = decode_item(a, gi);
        it.k0 = k;
        dsc = it;
        if (it.ok) {
          // the descriptor (generic stores, released by the arrive) and the unit's query
          // rows (bulk copies into padded rows) complete the same barrier phase
          const int G = a.G;
          const uint32_t row = (uint32_t)(a.L.d * 2);
          mbar_arrive_expect_tx(&sm.iq_full[iq], row * (uint32_t)G);
          const __half* qsrc = a.q + ((size_t)(it.u / a.Hkv) * a.Hq + (size_t)(it.u % a.Hkv) * G) * a.L.d;
          __half* qdst = sm.qbuf + (size_t)iq * 8 * (a.L.d + 8);
          for (int g = 0; g < G; ++g)
            bulk_g2s(qdst + (size_t)g * (a.L.d + 8), qsrc + (size_t)g * a.L.d, row, &sm.iq_full[iq], pol);
        } else {
          mbar_arrive(&sm.iq_full[iq]);  // nothing to stream for this item
          continue;
        }
        for (int c = 0; c < it.n_chunks; ++c, ++k) {
          const int slot = rp.slot;
          if (rp.use > 0 && !mbar_wait(&sm.empty[slot], (rp.use - 1) & 1u, a.err)) return;
          rp.next(a.nslot);
          const Chunk ch = item_chunk(a, it, c);
          if (ch.bytes) {
            mbar_arrive_expect_tx(&sm.full[slot], ch.bytes);
            bulk_g2s(sm.slots + (size_t)slot * a.slot_bytes, a.cache + ch.src, ch.bytes, &sm.full[slot], pol);
          } else {
            mbar_arrive(&sm.full[slot]);
          }
        }
      }
    }
    return;
  }

  // =========================== consumer warps
  Ring rc = {0, 0};
  for (int j = 0;; ++j) {
    const int iq = j % kIQ;
    if (!mbar_wait(&sm.iq_full[iq], (j / kIQ) & 1, a.err)) break;
    const ItemDesc it = sm.iqd[iq];
    named_bar_sync(1, kConsumers * 32);  // every consumer has its copy of the descriptor
    if (it.stop) break;
    if (it.ok) {
      consume_item<D, RT>(a, sm, it, rc, iq);  // releases the query slot itself
    } else {
      // an out-of-range routed index (raised in the device error word): an empty
      // partial keeps the unit's merge well defined
      if (warp == 0 && lane == 0) mbar_arrive(&sm.iq_empty[iq]);
      float* rec = a.partials + ((size_t)it.u * a.n_items + it.item) * (16 + 8 * D);
      for (int e = threadIdx.x; e < 16 + 8 * D; e += kConsumers * 32) rec[e] = e < 8 ? -INFINITY : 0.f;
    }
  }
}

template <int D, int RT>
cudaError_t launch_one(const AttendArgs& a, int grid, size_t smem, cudaStream_t s) {
  static size_t configured = 0;  // largest dynamic shared memory size enabled so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the router's grid
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_kernel<D, RT>, a);
}

}  // namespace

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev] = v;
  }
  return n[dev];
}

DecodePlan plan_decode(const Layout& L, int n_q_heads, int n_kv_heads, int top_k) {
  DecodePlan P;
  P.K_eff = (top_k == 0 || top_k >= L.NB) ? L.NB : top_k;
  P.wchunk_tokens = tc_eligible(L, n_q_heads, n_kv_heads) ? tc_window_tokens() : kWindowChunk;
  P.n_wchunks = (L.W16 + P.wchunk_tokens - 1) / P.wchunk_tokens;
  P.n_items = P.K_eff + P.n_wchunks;
  P.off_sched = kWsHeader;  // attention scheduler: work counter, finished-CTA counter
  P.off_routed = round_up(P.off_sched + 8, 256);
  P.off_partials = round_up(P.off_routed + (size_t)L.units * P.K_eff * 4, 256);
  P.ws_bytes = P.off_partials + (size_t)L.units * P.n_items * (16 + 8 * L.d) * 4;
  return P;
}

cudaError_t launch_attend(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s) {
  if (tc_eligible(L, n_q_heads, n_kv_heads)) return launch_attend_tc(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, s);
  AttendArgs a;
  a.L = L;
  a.G = n_q_heads / n_kv_heads;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.K_eff = P.K_eff;
  a.n_items = P.n_items;
  a.n_wchunks = P.n_wchunks;
  a.n_wfront = (P.n_wchunks + 1) / 2;
  a.total = P.n_items * L.units;
  a.xtok = 16384 / (4 * L.d);
  const int head = (int)L.off_u;
  int slot = 16384;
  slot = head > slot ? head : slot;
  slot = kUTok * 2 * L.r8 > slot ? kUTok * 2 * L.r8 : slot;
  slot = 2 * L.r8 * L.d > slot ? 2 * L.r8 * L.d : slot;
  slot = (int)round_up((uint64_t)slot, 128);
  const int RT = L.r8 <= 32 ? 2 : (L.r8 <= 64 ? 4 : 8);
  size_t extra;
  if (L.d == 128) extra = RT == 2 ? smem_extra<128, 2>() : (RT == 4 ? smem_extra<128, 4>() : smem_extra<128, 8>());
  else extra = RT == 2 ? smem_extra<64, 2>() : (RT == 4 ? smem_extra<64, 4>() : smem_extra<64, 8>());
  const size_t budget = 113 * 1024;  // two CTAs per SM
  int nslot = (int)((budget - extra) / slot);
  nslot = nslot > kMaxSlots ? kMaxSlots : nslot;
  if (nslot < 2) nslot = 2;
  a.nslot = nslot;
  a.slot_bytes = slot;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)L.d);
  a.q = q;
  a.cache = cache;
  a.routed = reinterpret_cast<const int32_t*>(ws + P.off_routed);
  a.partials = reinterpret_cast<float*>(ws + P.off_partials);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.sched = reinterpret_cast<uint32_t*>(ws + P.off_sched);
  const size_t smem = (size_t)nslot * slot + extra;
  if (a.total == 0) return cudaSuccess;
  int grid = 2 * sm_count();
  grid = grid < a.total ? grid : a.total;
  cudaError_t e;
  if (L.d == 128) {
    e = RT == 2 ? launch_one<128, 2>(a, grid, smem, s)
                : (RT == 4 ? launch_one<128, 4>(a, grid, smem, s) : launch_one<128, 8>(a, grid, smem, s));
  } else {
    e = RT == 2 ? launch_one<64, 2>(a, grid, smem, s)
                : (RT == 4 ? launch_one<64, 4>(a, grid, smem, s) : launch_one<64, 8>(a, grid, smem, s));
  }
  if (e != cudaSuccess || out == nullptr) return e;
  return launch_combine(L, P, L.units / n_kv_heads, n_q_heads, n_kv_heads, a.partials, out, lse, s);
}

}  // namespace dkv
