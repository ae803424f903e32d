// Block + window attention of the DKV decode path (fragment cache layout).
//
// Per routed block ("Low-Rank Space Query Scoring" / "Flash-Style LSE
// Combine", Differential-KV README, section "Core Architecture & Paper
// Overview"; DKV Zenodo abstract):
//   z_g   = V_K (c q_g)                          (per block, r numbers per query)
//   s_0   = c q_g . a_k                          (the anchor: U row 0 is zero)
//   s_i   = c q_g . a_k + U_i . z_g,  i not in S (K is never materialised)
//   s_j   = c q_g . k_j,              j in S     (exact residual rows)
//   o_g  += (sum_lowrank p) a_v + V_V^T (sum_lowrank p_i U_i) + sum_S p_j v_j
// and the exact recency window is attended like the residual rows.
//
// Work split.  Every unit (sequence, KV head) has the same list of work: its
// window in 64-token stages, then for each routed block the low-rank part
// (three chunks: anchors + mask + V_K, U, V_V) and the residual rows in
// 64-token stages.  The host cuts the list into n_r ranges of about equal
// bytes, each range starting with its share of the window (which needs no
// routing, so it overlaps the router's grid).  One CTA takes one (unit, range).
//
// Inside a CTA, warp 4's lane 0 streams the range's chunks with 1-D TMA bulk
// copies (cp.async.bulk + mbarrier complete_tx, L2 evict-first) into a byte
// ring of variable-size chunks that fills the CTA's shared memory; the four
// consumer warps take every chunk together (one 16-token group each of an
// exact stage, 64 U rows each of a block), so a chunk is released as soon as
// the four quarters are done and most of the ring is in flight.  Each
// consumer warp keeps one online-softmax state (m, l, o) over every token it
// scores, low-rank and exact alike: a block's p-weighted U sum w stays in
// the warp's registers from the U chunk to the V_V chunk, where the warp adds
// V_V^T w + (sum p) a_v to its own o, so no cross-warp merge is needed until
// the end of the range.  There the four states merge once into the range's
// partial record (m, l, o in base-2 units), in a ring chunk reserved for it;
// the combine kernel merges a unit's records with an fp32 log-sum-exp.
//
// Every matrix product runs on mma.sync m16n8k16 (fp16 operands, fp32
// accumulate) with tokens (or the head dimension) in M and the GQA group in
// N = 8.  fp32 operands of a product (z, p, w) are split into an fp16 pair
// hi + lo, so each product carries about 22 bits.
#include <float.h>
#include <math.h>

#include <atomic>
#include <vector>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kConsumers = 4;                 // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kNBar = 16;                     // chunk barrier pairs: chunks in the ring at most
constexpr int kStageTok = 16 * kConsumers;    // exact tokens per stage (one 16-token group per warp)
constexpr int kMaxRanges = 128;               // ranges per unit
constexpr int kCtasPerSm = 2;                 // resident CTAs per SM (registers and shared memory)
// 2 x (108 + 1 reserved) KB leaves an SM room for one router CTA of the same
// call (programmatic launch lets the two grids overlap)
constexpr size_t kSmemPerCta = 108 * 1024;

enum ChunkKind { kWin = 0, kRes = 1, kHead = 2, kU = 3, kVV = 4 };

// Every block is routed (top-K >= NB): slot j is block j, and no router grid runs.
constexpr int kModeAll = 2;

struct AttendArgs {
  Layout L;
  int G, Hq, Hkv, K_eff, n_r, nres, n_wst, ring, mode;
  uint32_t inflight;  // bytes a CTA keeps in flight (issued, not yet landed) at most
  uint32_t wait_limit;  // polls of a bounded wait (kWaitLimit unless a diagnostic limit is set)
  int stop_after;       // diagnostic: chunks a producer issues at most (negative: all)
  float scale_log2;  // log2(e) / sqrt(d)
  const __half* q;
  const uint8_t* cache;
  const int32_t* routed;  // [units][K_eff], written by the router grid
  int32_t* routed_out;    // kModeAll, optional: the caller's copy of the routed indices (0 .. NB-1)
  float* partials;        // [units][n_r][4 consumer warps] records [m 8][l 8][o 8][d]
  uint32_t* err;
  int tab[kMaxRanges][4];  // per range: window stages [0, 1), block items [2, 3)
};

// One chunk of a range's list, as both the producer and the consumers see it.
struct Chunk {
  int kind;
  int j;          // routed block slot (block chunks)
  int tok0, ntok; // exact stages: first token and token count (a multiple of 8)
  uint32_t bytes; // bytes in shared memory (and of the copy)
  uint64_t off;   // source offset inside the block record / the unit's window
};

// What the consumer warps need of a chunk, written by the producer into the
// chunk's slot of a small shared-memory queue before it arrives on the chunk's
// full barrier (whose completion releases the descriptor with the data).
struct ChunkDesc {
  int kind;
  uint32_t off;   // byte offset in the ring
  int tok0, ntok; // exact stages
  int blk;        // block index (block chunks; an un-rotated pool rotates by position)
};

// Walks the chunks of one range in order: window stages, then block items
// (item x: block slot x / (1 + nres), part x % (1 + nres); counters kept
// incrementally, so a step costs no division).
struct Cursor {
  int ws, ws1, it, it1, j, k, sub;
  __device__ inline void init(const AttendArgs& a, int range) {
    ws = a.tab[range][0];
    ws1 = a.tab[range][1];
    it = a.tab[range][2];
    it1 = a.tab[range][3];
    j = it / (1 + a.nres);
    k = it % (1 + a.nres);
    sub = 0;
  }
  __device__ inline bool next(const AttendArgs& a, Chunk& c) {
    const Layout& L = a.L;
    c.j = 0; c.tok0 = 0; c.ntok = 0; c.off = 0;
    if (ws < ws1) {
      c.kind = kWin;
      c.tok0 = ws * kStageTok;
      c.ntok = min(kStageTok, L.W16 - c.tok0);
      c.bytes = (uint32_t)(c.ntok * 4 * L.d);
      c.off = (uint64_t)c.tok0 * 4 * L.d;
      ++ws;
      return true;
    }
    if (it >= it1) return false;
    c.j = j;
    if (k == 0) {
      if (sub == 0) {
        c.kind = kHead; c.bytes = (uint32_t)L.off_u; c.off = 0;
      } else if (sub == 1) {
        c.kind = kU; c.bytes = (uint32_t)(L.off_res - L.off_u); c.off = L.off_u;
      } else {
        c.kind = kVV; c.bytes = (uint32_t)(L.block_bytes - L.off_vv); c.off = L.off_vv;
      }
      if (++sub < 3) return true;
      sub = 0;
    } else {
      c.kind = kRes;
      c.tok0 = (k - 1) * kStageTok;
      c.ntok = min(kStageTok, L.R8 - c.tok0);
      // fp16 rows: 4d bytes a token; quantised rows: whole 16-token groups of L.qgb bytes
      c.bytes = L.qbits ? (uint32_t)(c.ntok / 16 * L.qgb) : (uint32_t)(c.ntok * 4 * L.d);
      c.off = L.off_res + (L.qbits ? (uint64_t)(c.tok0 / 16) * L.qgb : (uint64_t)c.tok0 * 4 * L.d);
    }
    ++it;
    if (++k > a.nres) { k = 0; ++j; }
    return true;
  }
};

// Chunks of one range (window stages, block items, and two more chunks per low-rank part)
__device__ inline int range_chunks(const AttendArgs& a, int range) {
  const int per = 1 + a.nres, it0 = a.tab[range][2], it1 = a.tab[range][3];
  const int n_lr = (it1 + per - 1) / per - (it0 + per - 1) / per;  // multiples of per in [it0, it1)
  return (a.tab[range][1] - a.tab[range][0]) + (it1 - it0) + 2 * n_lr;
}

// Place a chunk of `bytes` in the ring: chunks are contiguous, 128-byte aligned,
// and never wrap (a chunk that would wrap starts at the ring's beginning; the
// skipped tail counts as part of it).  pos: running byte count; off: pos in the ring.
struct RingPos {
  uint32_t pos, off;
  __device__ inline uint32_t place(uint32_t bytes, uint32_t ring) {
    const uint32_t b = (bytes + 127u) & ~127u;
    if (off + b > ring) { pos += ring - off; off = 0; }
    const uint32_t at = off;
    pos += b;
    off += b;
    if (off >= ring) off = 0;
    return at;
  }
};

__device__ inline float warp_max_rows(float v) {  // over lanes with the same lane % 4
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
// 8 bytes per lane (at lane * 8), returned in .x, .y.
__device__ inline uint4 ld_tile(uint32_t base, int lane, bool full) {
  const uint4 v = lds128(base + (uint32_t)(full ? lane * 16 : (lane >> 1) * 16));
  const bool odd = (lane & 1) != 0;
  return make_uint4(full ? v.x : (odd ? v.z : v.x), full ? v.y : (odd ? v.w : v.y), v.z, v.w);
}

// ldmatrix: four (x4) or two (x2) 8x8 b16 matrices, row addresses from lanes 8i..8i+7
// for matrix i; .trans gives the transposed matrices' fragments
__device__ inline uint4 ldsm4(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ inline uint4 ldsm4t(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ inline uint2 ldsm2(uint32_t addr) {
  uint2 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ inline uint2 ldsm2t(uint32_t addr) {
  uint2 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// C fragment (rows = k, two columns per lane) -> B fragments (k, n = group), hi and lo
__device__ inline void c_to_b(float c0, float c1, float c2, float c3, uint32_t& bh0, uint32_t& bl0, uint32_t& bh1,
                              uint32_t& bl1) {
  uint32_t h01, l01, h23, l23;
  split_half2(c0, c1, h01, l01);
  split_half2(c2, c3, h23, l23);
  bh0 = movtrans(h01); bl0 = movtrans(l01);
  bh1 = movtrans(h23); bl1 = movtrans(l23);
}

// Online-softmax state of one consumer warp for its two C-fragment columns
// (g = 2t, 2t + 1): running maximum m (base 2), per-lane partial normaliser l
// (summed over the warp's rows at the end) and the output accumulator o[d][g].
template <int D>
struct WarpState {
  float m0, m1, l0, l1;
  float o[D / 16][4];
};

// Scores may exceed the running maximum by up to kSlack (base 2) before it is
// moved: p = 2^(s - m) then stays below 2^kSlack, which fp32 sums and the
// hi + lo fp16 splits carry exactly as well, and most 16-token groups skip the
// rescale of o.  The record's (m, l, o) stays consistent whatever m is.
constexpr float kSlack = 8.f;

// Include this lane's tile maxima (mx0, mx1) of its two columns.  Returns
// whether the accumulated state was rescaled (a warp-uniform answer), the
// rescale factors (1 if not) and the subtrahends of the new p.
template <int D>
__device__ inline bool raise_max(WarpState<D>& st, float mx0, float mx1, float& sc0, float& sc1, float& ms0,
                                 float& ms1) {
  // st.m is the same on every lane of a column, so the vote can take each lane's own
  // tile maximum: the reduction over the column's lanes runs only when the maximum moves
  const bool up = __any_sync(0xffffffffu, mx0 > st.m0 + kSlack || mx1 > st.m1 + kSlack);
  if (up) {
    mx0 = warp_max_rows(mx0);
    mx1 = warp_max_rows(mx1);
    const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
    ms0 = n0 == -INFINITY ? 0.f : n0;
    ms1 = n1 == -INFINITY ? 0.f : n1;
    sc0 = fast_exp2(st.m0 - ms0);  // 2^(-inf) = 0
    sc1 = fast_exp2(st.m1 - ms1);
    st.m0 = n0;
    st.m1 = n1;
    st.l0 *= sc0;
    st.l1 *= sc1;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) { st.o[i][0] *= sc0; st.o[i][1] *= sc1; st.o[i][2] *= sc0; st.o[i][3] *= sc1; }
  } else {
    ms0 = st.m0 == -INFINITY ? 0.f : st.m0;
    ms1 = st.m1 == -INFINITY ? 0.f : st.m1;
    sc0 = sc1 = 1.f;
  }
  return up;
}

// RoPE at read of an un-rotated pool, for one lane: the positions of its two
// key rows (gq, gq + 8 of the 16-token tile) and the cache's RoPE tables.
// float2 per in-page factor row: h <= 64 pairs, padded so that the 8-byte loads of a half
// warp (rows gq, pairs 2t + e) fall in distinct bank pairs (row stride = 8 banks mod 32)
constexpr int kRopeRow = 64 + 4;
struct RopeRows {
  const float2* tab;       // the cache's page table [pages][h] (global)
  const float2* s16;       // shared: (cos, sin)(16 m theta_j), [16][kRopeRow]
  const float2* s1;        // shared: (cos, sin)(i theta_j), [16][kRopeRow]
  int pages, h;            // h = rope channels / 2: channel j < h pairs with j + h
  int P0, P1;
};
__device__ inline float2 cmul(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// (cos, sin) of P theta_j: page entry of P >> 8 (256 p theta_j) turned by 16 m theta_j and
// i theta_j, P = 256 p + 16 m + i
__device__ inline float2 rope_angle(const RopeRows& rr, int P, int j) {
  const float2 a = __ldg(rr.tab + (size_t)(P >> 8) * rr.h + j);
  return cmul(cmul(a, rr.s16[((P >> 4) & 15) * kRopeRow + j]), rr.s1[(P & 15) * kRopeRow + j]);
}
// turn the pair (x, y) = (channel j, channel j + h) by the angle whose (cos, sin) is cs
__device__ inline void rot_pair(float& x, float& y, float2 cs) {
  const float xr = fmaf(x, cs.x, -y * cs.y);
  y = fmaf(y, cs.x, x * cs.y);
  x = xr;
}
// rotate one register pair of key fragments: ra holds channels (j, j + 1) of a row, rb
// the same row's channels (j + h, j + h + 1); returns them rotated as fp32
__device__ inline void rot_regs(uint32_t ra, uint32_t rb, const RopeRows& rr, int P, int j, float2& xa, float2& xb) {
  xa = __half22float2(*reinterpret_cast<const __half2*>(&ra));
  xb = __half22float2(*reinterpret_cast<const __half2*>(&rb));
  rot_pair(xa.x, xb.x, rope_angle(rr, P, j));
  rot_pair(xa.y, xb.y, rope_angle(rr, P, j + 1));
}

// One 16-token exact group (residual rows or window tokens) of one warp:
// K tile [in_g x D] then V^T tile [D x in_g] at gb, in_g = 16 or 8.  With ROPE
// the key rows are rotated to their positions (rr) first: k tiles kt < h/16 pair
// with kt + h/16, and each rotated tile enters the product as fp16 hi + lo.
template <int D, bool FULL, bool ROPE = false>
__device__ __forceinline__ void exact_group(WarpState<D>& st, uint32_t qrow, uint32_t gb, int tok, int nvalid,
                                            float slog2, bool gv0, bool gv1, int lane, const RopeRows* rr = nullptr) {
  constexpr int KT = D / 16;
  constexpr int in_g = FULL ? 16 : 8;
  constexpr bool full = FULL;
  const int gq = lane >> 2, t = lane & 3;
  constexpr uint32_t kst = full ? 512u : 256u;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if constexpr (ROPE) {
    const int hk = rr->h / 16;  // rotated k-tile pairs
    auto qfrag = [&](int kt, uint32_t& b0, uint32_t& b1) {
      b0 = lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u);
      b1 = lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u);
    };
#pragma unroll 1
    for (int kt = 0; kt < hk; ++kt) {
      const uint4 va = ld_tile(gb + (uint32_t)kt * kst, lane, full);
      const uint4 vb = ld_tile(gb + (uint32_t)(kt + hk) * kst, lane, full);
      // a0 / a2: row gq, channels 16 kt + 2t.. / 16 kt + 8 + 2t..; a1 / a3: row gq + 8
      const int j0 = 16 * kt + 2 * t;
      float2 xa0, xb0, xa2, xb2, xa1 = make_float2(0.f, 0.f), xb1 = xa1, xa3 = xa1, xb3 = xa1;
      rot_regs(va.x, vb.x, *rr, rr->P0, j0, xa0, xb0);
      rot_regs(full ? va.z : va.y, full ? vb.z : vb.y, *rr, rr->P0, j0 + 8, xa2, xb2);
      if (full) {
        rot_regs(va.y, vb.y, *rr, rr->P1, j0, xa1, xb1);
        rot_regs(va.w, vb.w, *rr, rr->P1, j0 + 8, xa3, xb3);
      }
      uint32_t h0, l0, h1, l1, h2, l2, h3, l3, b0, b1;
      split_half2(xa0.x, xa0.y, h0, l0);
      split_half2(xa1.x, xa1.y, h1, l1);
      split_half2(xa2.x, xa2.y, h2, l2);
      split_half2(xa3.x, xa3.y, h3, l3);
      qfrag(kt, b0, b1);
      mma16816(acc[0], h0, h1, h2, h3, b0, b1);
      mma16816(acc[0], l0, l1, l2, l3, b0, b1);
      split_half2(xb0.x, xb0.y, h0, l0);
      split_half2(xb1.x, xb1.y, h1, l1);
      split_half2(xb2.x, xb2.y, h2, l2);
      split_half2(xb3.x, xb3.y, h3, l3);
      qfrag(kt + hk, b0, b1);
      mma16816(acc[1], h0, h1, h2, h3, b0, b1);
      mma16816(acc[1], l0, l1, l2, l3, b0, b1);
    }
#pragma unroll 1
    for (int kt = 2 * hk; kt < KT; ++kt) {  // channels past the rotated ones, exact fp16
      const uint4 v = ld_tile(gb + (uint32_t)kt * kst, lane, full);
      uint32_t b0, b1;
      qfrag(kt, b0, b1);
      mma16816(acc[kt & 1], v.x, full ? v.y : 0u, full ? v.z : v.y, full ? v.w : 0u, b0, b1);
    }
  } else {
    uint32_t qb[KT][2];
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      qb[kt][0] = lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u);
      qb[kt][1] = lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u);
    }
    uint4 kv[KT];
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) kv[kt] = ld_tile(gb + (uint32_t)kt * kst, lane, full);
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      // K tile (m = tokens, k = d): a half group holds rows gq only: (x, y) = k 2t.., 2t + 8..
      const uint4 v = kv[kt];
      const uint32_t a0 = v.x, a1 = full ? v.y : 0u, a2 = full ? v.z : v.y, a3 = full ? v.w : 0u;
      mma16816(acc[kt & 1], a0, a1, a2, a3, qb[kt][0], qb[kt][1]);
    }
  }
  const int tk0 = tok + gq, tk1 = tk0 + 8;
  const bool v0 = tk0 < nvalid, v1 = tk1 < nvalid && (gq + 8 < in_g);
  float s[4];
  s[0] = v0 ? (acc[0][0] + acc[1][0]) * slog2 : -INFINITY;
  s[1] = v0 ? (acc[0][1] + acc[1][1]) * slog2 : -INFINITY;
  s[2] = v1 ? (acc[0][2] + acc[1][2]) * slog2 : -INFINITY;
  s[3] = v1 ? (acc[0][3] + acc[1][3]) * slog2 : -INFINITY;
  const uint32_t vb = gb + (uint32_t)(in_g * D * 2);
  float sc0, sc1, ms0, ms1;
  raise_max<D>(st, fmaxf(s[0], s[2]), fmaxf(s[1], s[3]), sc0, sc1, ms0, ms1);
  float p[4];
  p[0] = gv0 ? fast_exp2(s[0] - ms0) : 0.f;
  p[1] = gv1 ? fast_exp2(s[1] - ms1) : 0.f;
  p[2] = gv0 ? fast_exp2(s[2] - ms0) : 0.f;
  p[3] = gv1 ? fast_exp2(s[3] - ms1) : 0.f;
  st.l0 += p[0] + p[2];
  st.l1 += p[1] + p[3];
  uint32_t bh0, bl0, bh1, bl1;
  c_to_b(p[0], p[1], p[2], p[3], bh0, bl0, bh1, bl1);
#pragma unroll
  for (int md = 0; md < KT; ++md) {
    // V^T tile (m = d, k = tokens): a half group holds k 0..7 only
    const uint4 v = ld_tile(vb + (uint32_t)md * kst, lane, full);
    const uint32_t a2 = full ? v.z : 0u, a3 = full ? v.w : 0u;
    mma16816(st.o[md], v.x, v.y, a2, a3, bh0, bh1);
    mma16816(st.o[md], v.x, v.y, a2, a3, bl0, bl1);
  }
}

// One 16-token group of group-quantised residual rows (Layout.qbits = BITS) of
// one warp: the same products as exact_group, with each operand register
// rebuilt from its codes in registers: (code | 0x6400) is the half 1024 + code,
// so h - 1024 is the code exactly and fma(scale, code, bias) rounds the
// dequantised value to fp16 once.  Key rows take their row's scale (rows gq,
// gq + 8 of the tile); value columns (tokens 2t, 2t + 1 and 2t + 8, 2t + 9)
// their tokens' scales, per 64-channel group.
__device__ inline __half2 lds_h2(uint32_t addr) {  // one fp16 from shared memory, in both halves
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __half2half2(__ushort_as_half(v));
}
__device__ inline uint32_t deq2(uint32_t codes, __half2 s, __half2 b) {
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&codes), __float2half2_rn(1024.f));
  const __half2 x = __hfma2(s, c, b);
  return *reinterpret_cast<const uint32_t*>(&x);
}
template <int BITS>
__device__ inline uint32_t qfield(uint32_t w, int sh) {  // the half2 1024 + codes of one register
  return ((w >> sh) & (BITS == 8 ? 0x00FF00FFu : 0x000F000Fu)) | 0x64006400u;
}
template <int D, int BITS>
__device__ __forceinline__ void exact_group_q(WarpState<D>& st, uint32_t qrow, uint32_t gb, int tok, int nvalid,
                                              float slog2, bool gv0, bool gv1, int lane) {
  constexpr int KT = D / 16;
  constexpr int G = D / kQuantGroup;
  constexpr uint32_t CB = 16u * D * BITS / 8u;
  constexpr int TPC = BITS == 8 ? 2 : 4;  // k tiles per 512-byte chunk
  const int gq = lane >> 2, t = lane & 3;
  uint32_t qb[KT][2];
#pragma unroll
  for (int kt = 0; kt < KT; ++kt) {
    qb[kt][0] = lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u);
    qb[kt][1] = lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u);
  }
  const uint32_t ksc = gb + 2 * CB, vsc = ksc + 64u * G;  // [scale G x 16][bias G x 16] of K, then of V
  uint4 kw[KT / TPC];
#pragma unroll
  for (int c = 0; c < KT / TPC; ++c) kw[c] = lds128(gb + (uint32_t)c * 512u + (uint32_t)lane * 16u);
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int g = 0; g < G; ++g) {
    // this lane's key rows gq and gq + 8: one scale and one bias each, for both halves
    const __half2 s0 = lds_h2(ksc + (uint32_t)(g * 16 + gq) * 2u), s1 = lds_h2(ksc + (uint32_t)(g * 16 + gq + 8) * 2u);
    const __half2 b0 = lds_h2(ksc + 32u * G + (uint32_t)(g * 16 + gq) * 2u);
    const __half2 b1 = lds_h2(ksc + 32u * G + (uint32_t)(g * 16 + gq + 8) * 2u);
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {  // the four k tiles of this 64-channel group
      const int kt = 4 * g + kq;
      const uint4 v = kw[kt / TPC];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t a0, a1, a2, a3;
      if (BITS == 8) {
        const uint32_t wa = wv[2 * (kt % 2)], wb = wv[2 * (kt % 2) + 1];
        a0 = deq2(qfield<8>(wa, 0), s0, b0);
        a1 = deq2(qfield<8>(wa, 8), s1, b1);
        a2 = deq2(qfield<8>(wb, 0), s0, b0);
        a3 = deq2(qfield<8>(wb, 8), s1, b1);
      } else {
        const uint32_t w = wv[kt % 4];
        a0 = deq2(qfield<4>(w, 0), s0, b0);
        a1 = deq2(qfield<4>(w, 4), s1, b1);
        a2 = deq2(qfield<4>(w, 8), s0, b0);
        a3 = deq2(qfield<4>(w, 12), s1, b1);
      }
      mma16816(acc[kt & 1], a0, a1, a2, a3, qb[kt][0], qb[kt][1]);
    }
  }
  const int tk0 = tok + gq, tk1 = tk0 + 8;
  const bool v0 = tk0 < nvalid, v1 = tk1 < nvalid;
  float s[4];
  s[0] = v0 ? (acc[0][0] + acc[1][0]) * slog2 : -INFINITY;
  s[1] = v0 ? (acc[0][1] + acc[1][1]) * slog2 : -INFINITY;
  s[2] = v1 ? (acc[0][2] + acc[1][2]) * slog2 : -INFINITY;
  s[3] = v1 ? (acc[0][3] + acc[1][3]) * slog2 : -INFINITY;
  float sc0, sc1, ms0, ms1;
  raise_max<D>(st, fmaxf(s[0], s[2]), fmaxf(s[1], s[3]), sc0, sc1, ms0, ms1);
  float p[4];
  p[0] = gv0 ? fast_exp2(s[0] - ms0) : 0.f;
  p[1] = gv1 ? fast_exp2(s[1] - ms1) : 0.f;
  p[2] = gv0 ? fast_exp2(s[2] - ms0) : 0.f;
  p[3] = gv1 ? fast_exp2(s[3] - ms1) : 0.f;
  st.l0 += p[0] + p[2];
  st.l1 += p[1] + p[3];
  uint32_t bh0, bl0, bh1, bl1;
  c_to_b(p[0], p[1], p[2], p[3], bh0, bl0, bh1, bl1);
  uint4 vw[KT / TPC];
#pragma unroll
  for (int c = 0; c < KT / TPC; ++c) vw[c] = lds128(gb + CB + (uint32_t)c * 512u + (uint32_t)lane * 16u);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    // value columns: tokens (2t, 2t + 1) and (2t + 8, 2t + 9), their own scales and biases
    const uint32_t sl = lds32(vsc + (uint32_t)(g * 16 + 2 * t) * 2u), sh = lds32(vsc + (uint32_t)(g * 16 + 2 * t + 8) * 2u);
    const uint32_t bl = lds32(vsc + 32u * G + (uint32_t)(g * 16 + 2 * t) * 2u);
    const uint32_t bhh = lds32(vsc + 32u * G + (uint32_t)(g * 16 + 2 * t + 8) * 2u);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sl), s89 = *reinterpret_cast<const __half2*>(&sh);
    const __half2 b01 = *reinterpret_cast<const __half2*>(&bl), b89 = *reinterpret_cast<const __half2*>(&bhh);
#pragma unroll
    for (int mq = 0; mq < 4; ++mq) {
      const int md = 4 * g + mq;
      const uint4 v = vw[md / TPC];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      uint32_t a0, a1, a2, a3;
      if (BITS == 8) {
        const uint32_t wa = wv[2 * (md % 2)], wb = wv[2 * (md % 2) + 1];
        a0 = deq2(qfield<8>(wa, 0), s01, b01);
        a1 = deq2(qfield<8>(wa, 8), s01, b01);
        a2 = deq2(qfield<8>(wb, 0), s89, b89);
        a3 = deq2(qfield<8>(wb, 8), s89, b89);
      } else {
        const uint32_t w = wv[md % 4];
        a0 = deq2(qfield<4>(w, 0), s01, b01);
        a1 = deq2(qfield<4>(w, 4), s01, b01);
        a2 = deq2(qfield<4>(w, 8), s89, b89);
        a3 = deq2(qfield<4>(w, 12), s89, b89);
      }
      mma16816(st.o[md], a0, a1, a2, a3, bh0, bh1);
      mma16816(st.o[md], a0, a1, a2, a3, bl0, bl1);
    }
  }
}

// Low-rank state of one routed block, live from its head chunk to its V_V chunk.
// Padded rank of a kernel instance: R8S > 0 fixes it at compile time (every
// tile test then folds away); R8S < 0 reads it at run time, up to 16 * (-R8S).
template <int R8S>
struct RankTiles {
  static constexpr int RT = R8S > 0 ? (R8S + 15) / 16 : -R8S;  // r tiles of 16 (the last may be 8 wide)
};

template <int D, int RT>
struct BlockState {
  uint32_t zh[RT][2], zl[RT][2];  // z as B fragments (k = r, n = group), hi and lo
  float us0, us1;                 // unscale of z for columns 2t, 2t + 1
  float base0, base1;             // c q . a_k (base 2) for columns 2t, 2t + 1
  uint32_t mk0, mk1;              // residual-row mask of this warp's 64 U rows
  float w[RT][4];                 // sum p_i U_i (C fragment: rows = r, columns = group)
  float pa0, pa1;                 // per-lane partial sum of the low-rank p
  uint32_t hsb;                   // un-rotated pool: the block's head chunk (a_k, V_K), held until U is scored
};


// shared memory: [ring][full kNBar][empty kNBar][query barrier][ends kNBar]
// [query rows 8 x (D + 8) fp16][a_v, one copy per consumer warp: 4 x D fp16]
// [chunk descriptors kNBar] and, for an un-rotated pool, [RoPE in-page factors]:
// (cos, sin) of 16 m theta_j and of i theta_j for m, i < 16 (rows of kRopeRow float2)
constexpr size_t kRopeSmem = 2 * 16 * kRopeRow * 8;
__host__ __device__ inline size_t smem_extra(bool rope) {
  return (size_t)kNBar * 8 * 2 + 16 + (size_t)kNBar * 4 + 8 * 136 * 2 + kConsumers * 128 * 2 +
         kNBar * sizeof(ChunkDesc) + 64 + (rope ? kRopeSmem : 0);
}

template <int D, int R8S, bool ROPE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) attend_kernel(AttendArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int KT = D / 16;
  constexpr int RT = RankTiles<R8S>::RT;
  const Layout& L = a.L;
  const uint32_t ring = (uint32_t)a.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring);
  uint64_t* empty = full + kNBar;
  uint64_t* qbar = empty + kNBar;
  uint32_t* ends = reinterpret_cast<uint32_t*>(qbar + 2);
  __half* qsm = reinterpret_cast<__half*>(ends + kNBar);  // [8][D + 8]: 16-byte aligned rows
  __half* avw = qsm + 8 * (D + 8);                        // [4][D]
  ChunkDesc* cdq = reinterpret_cast<ChunkDesc*>(avw + kConsumers * 128);  // [kNBar] chunk descriptors
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / a.n_r, range = blockIdx.x % a.n_r;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNBar; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kConsumers); }
    mbar_init(qbar, 1);
    fence_mbar_init();
  }
  // query rows past the group stay zero (the bulk copies fill rows 0 .. G-1)
  for (int e = threadIdx.x; e < (8 - a.G) * (D + 8); e += kThreads) qsm[a.G * (D + 8) + e] = __float2half(0.f);
  float2* rsm = reinterpret_cast<float2*>(cdq + kNBar);  // ROPE: [16][kRopeRow] x 2
  if constexpr (ROPE) {
    // rows 16 m and i (m, i < 16) of the cache's in-page table
    const int h = L.rope / 2;
    const float2* inpage = reinterpret_cast<const float2*>(a.cache + L.off_rope) + (size_t)L.rope_pages * h;
    for (int e = threadIdx.x; e < 32 * h; e += kThreads) {
      const int row = e / h, j = e % h;
      rsm[row * kRopeRow + j] = inpage[(size_t)(row < 16 ? 16 * row : row - 16) * h + j];
    }
  }
  __syncthreads();
  griddep_launch();  // the combine grid may be scheduled now; it waits for this grid's completion

  // =========================== producer (warp 4, lane 0)
  if (warp == kConsumers) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    const uint8_t* unit = a.cache + (uint64_t)u * L.unit_stride;
    const __half* qsrc = a.q + ((size_t)(u / a.Hkv) * a.Hq + (size_t)(u % a.Hkv) * a.G) * L.d;
    // the unit's G query rows, into padded shared-memory rows
    mbar_arrive_expect_tx(qbar, (uint32_t)(a.G * L.d * 2));
    for (int g = 0; g < a.G; ++g) bulk_g2s(qsm + g * (D + 8), qsrc + (size_t)g * L.d, (uint32_t)(L.d * 2), qbar, pol);
    Cursor cur;
    cur.init(a, range);
    Chunk ch;
    RingPos rp = {0u, 0u};
    uint32_t rel_end = 0, land_end = 0;
    int c = 0, rel = 0, land = 0;  // chunks issued; released (seen); landed (seen)
    bool routed_ready = false, ok = true;
    int jb = -1, bcur = 0;
    const uint8_t* blk = unit;
    while (ok && cur.next(a, ch)) {
      if (a.stop_after >= 0 && c >= a.stop_after) break;  // diagnostic: nothing further is issued
      const uint32_t off = rp.place(ch.bytes, ring);
      // wait until the chunk's bytes and barrier pair are free: the chunks not yet
      // released occupy [rel_end, start) of the running byte count (releases come in order)
      while (ok && (c - rel >= kNBar || (rel < c && rp.pos - rel_end > ring))) {
        const int rb = rel & (kNBar - 1);
        ok = mbar_wait(&empty[rb], (uint32_t)(rel / kNBar) & 1u, a.err, a.wait_limit);
        if (ok) { rel_end = ends[rb]; ++rel; }
      }
      // keep at most a.inflight bytes in flight: more only lengthens the queues of the
      // memory system (every CTA's first chunks land later) without adding bandwidth
      if (land < rel) { land = rel; land_end = rel_end; }
      while (ok && land < c && rp.pos - land_end > a.inflight) {
        const int lb = land & (kNBar - 1);
        ok = mbar_wait(&full[lb], (uint32_t)(land / kNBar) & 1u, a.err, a.wait_limit);
        if (ok) { land_end = ends[lb]; ++land; }
      }
      if (!ok) break;  // a wait gave up: nothing further is issued
      const int cb = c & (kNBar - 1);
      ends[cb] = rp.pos;
      if (ch.kind != kWin && ch.j != jb) {
        int b = ch.j;  // kModeAll: slot j is block j
        if (!(a.mode & kModeAll)) {
          if (!routed_ready) { griddep_wait(); routed_ready = true; }  // the router's grid has completed
          b = a.routed[(size_t)u * a.K_eff + ch.j];
        }
        if (b < 0 || b >= L.NB) {
          raise_error(a.err, DKV_DEVERR_INDEX);
          b = 0;
        }
        jb = ch.j;
        bcur = b;
        blk = unit + L.off_blocks + (uint64_t)b * L.block_stride;
      }
      ChunkDesc dsc;
      dsc.kind = ch.kind;
      dsc.off = off;
      dsc.tok0 = ch.tok0;
      dsc.ntok = ch.ntok;
      dsc.blk = ch.kind == kWin ? -1 : bcur;
      cdq[cb] = dsc;  // released to the consumers by this chunk's barrier phase
      uint64_t* fb = &full[cb];
      uint8_t* dst = smem + off;
      if (ch.kind == kWin) {
        mbar_arrive_expect_tx(fb, ch.bytes);
        bulk_g2s(dst, unit + L.off_window + ch.off, ch.bytes, fb, pol);
      } else if (ch.bytes == 0) {
        mbar_arrive(fb);  // an empty section (rank 0)
      } else {
        mbar_arrive_expect_tx(fb, ch.bytes);
        bulk_g2s(dst, blk + ch.off, ch.bytes, fb, pol);
      }
      ++c;
    }
    // every copy this CTA issued lands before the producer (and with it the CTA) may
    // finish, whether or not a wait gave up: the chunks not seen released, fewer than
    // kNBar of them, each on its own barrier
    for (int x = rel; x < c; ++x)
      if (!mbar_wait(&full[x & (kNBar - 1)], (uint32_t)(x / kNBar) & 1u, a.err, a.wait_limit)) break;
    return;
  }

  // =========================== consumer warps
  const int t = lane & 3, gq = lane >> 2;
  const int G = a.G;
  const bool gv0 = (2 * t) < G, gv1 = (2 * t + 1) < G;
  const float slog2 = a.scale_log2;
  const int r8 = R8S > 0 ? R8S : L.r8;
  const int nkk = r8 >> 4;                 // full 16-wide k tiles of r
  const bool rtail = (r8 & 15) != 0;       // one 8-wide tail
  const int nrt = nkk + (rtail ? 1 : 0);   // r tiles
  const uint32_t sbase = smem_u32(smem);
  bool alive = true;                       // false after a bounded wait gave up
  WarpState<D> st;
  BlockState<D, RT> bs;
  const uint32_t qrow = smem_u32(qsm + gq * (D + 8));  // this lane's query row (B fragments of q)
  __half* av = avw + warp * D;                         // this warp's copy of the block's a_v
  alive = __all_sync(0xffffffffu, mbar_wait(qbar, 0u, a.err, a.wait_limit));
  const int tid = threadIdx.x;
  if ((a.mode & kModeAll) && a.routed_out && range == 0)
    for (int j = tid; j < a.K_eff; j += kConsumers * 32) a.routed_out[(size_t)u * a.K_eff + j] = j;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
#pragma unroll
  for (int i = 0; i < KT; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
  RopeRows rr;
  const uint8_t* unit_g = a.cache + (uint64_t)u * L.unit_stride;
  if constexpr (ROPE) {
    rr.tab = reinterpret_cast<const float2*>(a.cache + L.off_rope);
    rr.s16 = rsm;
    rr.s1 = rsm + 16 * kRopeRow;
    rr.pages = L.rope_pages;
    rr.h = L.rope / 2;
  }
  int held = -1;  // ROPE: ring slot of the block head this warp still holds
  const int n_chunks = range_chunks(a, range);
  for (int c = 0; c < n_chunks; ++c) {
    const int bi = c & (kNBar - 1);
    if (alive) alive = __all_sync(0xffffffffu, mbar_wait(&full[bi], (uint32_t)(c / kNBar) & 1u, a.err, a.wait_limit));
    const ChunkDesc ch = cdq[bi];  // kind, ring offset and tokens, from the producer
    const uint32_t sb = sbase + ch.off;
    const uint8_t* sp = smem + ch.off;
    switch (alive ? ch.kind : -1) {
      case kWin:
      case kRes: {
        const int in_g = max(0, min(16, ch.ntok - 16 * warp));
        const int nvalid = ch.kind == kWin ? L.W : L.R;
        if (ch.kind == kRes && L.qbits) {  // quantised residual rows: whole 16-token groups
          const uint32_t qg = sb + (uint32_t)(warp * L.qgb);
          if (alive && in_g == 16 && L.qbits == 8)
            exact_group_q<D, 8>(st, qrow, qg, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane);
          else if (alive && in_g == 16)
            exact_group_q<D, 4>(st, qrow, qg, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane);
          break;
        }
        const uint32_t gb = sb + (uint32_t)(warp * 64 * D);
        if constexpr (ROPE) {
          // positions: window token w at 256 NB + w; residual row i of block b at 256 b + its token
          const int tk = ch.tok0 + 16 * warp + gq;
          if (ch.kind == kWin) {
            rr.P0 = 256 * L.NB + tk;
            rr.P1 = rr.P0 + 8;
          } else {
            const uint16_t* cold = reinterpret_cast<const uint16_t*>(unit_g + L.off_cold) + (size_t)ch.blk * L.R8;
            rr.P0 = 256 * ch.blk + (tk < L.R8 ? (int)cold[tk] : 0);
            rr.P1 = 256 * ch.blk + (tk + 8 < L.R8 ? (int)cold[tk + 8] : 0);
          }
          if (alive && in_g == 16)
            exact_group<D, true, true>(st, qrow, gb, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane, &rr);
          else if (alive && in_g == 8)
            exact_group<D, false, true>(st, qrow, gb, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane, &rr);
        } else {
          if (alive && in_g == 16)
            exact_group<D, true>(st, qrow, gb, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane);
          else if (alive && in_g == 8)
            exact_group<D, false>(st, qrow, gb, ch.tok0 + 16 * warp, nvalid, slog2, gv0, gv1, lane);
        }
        break;
      }
      case kHead: {
        if constexpr (ROPE) {
          const uint32_t* mask = reinterpret_cast<const uint32_t*>(sp + L.off_mask);
          bs.mk0 = alive ? mask[2 * warp] : 0u;
          bs.mk1 = alive ? mask[2 * warp + 1] : 0u;
          const __half* ak = reinterpret_cast<const __half*>(sp);
          for (int j = lane; j < D; j += 32) av[j] = ak[D + j];  // read back at the V_V chunk
          bs.hsb = sb;
#pragma unroll
          for (int i = 0; i < RT; ++i) bs.w[i][0] = bs.w[i][1] = bs.w[i][2] = bs.w[i][3] = 0.f;
          bs.pa0 = bs.pa1 = 0.f;
        } else {
        uint32_t qb[KT][2];
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
          qb[kt][0] = lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u);
          qb[kt][1] = lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u);
        }
        // base = c q . a_k for this lane's query row gq (four partial sums), then columns 2t, 2t + 1
        const __half* ak = reinterpret_cast<const __half*>(sp);
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
          const float2 q0 = __half22float2(*reinterpret_cast<const __half2*>(&qb[kt][0]));
          const float2 q1 = __half22float2(*reinterpret_cast<const __half2*>(&qb[kt][1]));
          const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(ak + 16 * kt + 2 * t));
          const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(ak + 16 * kt + 8 + 2 * t));
          part[kt & 3] = fmaf(q0.x, a0.x, fmaf(q0.y, a0.y, fmaf(q1.x, a1.x, fmaf(q1.y, a1.y, part[kt & 3]))));
        }
        float pb = (part[0] + part[1]) + (part[2] + part[3]);
        pb += __shfl_xor_sync(0xffffffffu, pb, 1);
        pb += __shfl_xor_sync(0xffffffffu, pb, 2);
        bs.base0 = __shfl_sync(0xffffffffu, pb, 8 * t) * slog2;
        bs.base1 = __shfl_sync(0xffffffffu, pb, 8 * t + 4) * slog2;
        const uint32_t* mask = reinterpret_cast<const uint32_t*>(sp + L.off_mask);
        bs.mk0 = alive ? mask[2 * warp] : 0u;
        bs.mk1 = alive ? mask[2 * warp + 1] : 0u;
        for (int j = lane; j < D; j += 32) av[j] = ak[D + j];  // read back at the V_V chunk
        // z = V_K (c q): V_K (stored as 8-row B^T tiles) read as the A operand, two tiles per
        // 16-row m-tile; q as B.  The C fragments (rows = r, columns = group) become the B
        // fragments of U z through movmatrix, with a per-column power-of-two scale.
        const uint32_t vk = sb + (uint32_t)L.off_vk;
        const int nt8 = r8 >> 3;
        float zc[RT][4];
#pragma unroll
        for (int mt = 0; mt < RT; ++mt) {
          zc[mt][0] = zc[mt][1] = zc[mt][2] = zc[mt][3] = 0.f;
          if (mt < nrt) {
            const bool lo_rows = 2 * mt + 1 < nt8;  // the m-tile's rows 8..15 exist
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
              const uint4 b0 = lds128(vk + (uint32_t)((2 * mt) * 8 * D * 2 + kp * 512 + lane * 16));
              const uint4 b1 = lo_rows ? lds128(vk + (uint32_t)((2 * mt + 1) * 8 * D * 2 + kp * 512 + lane * 16))
                                       : make_uint4(0u, 0u, 0u, 0u);
              mma16816(zc[mt], b0.x, b1.x, b0.y, b1.y, qb[2 * kp][0], qb[2 * kp][1]);
              mma16816(zc[mt], b0.z, b1.z, b0.w, b1.w, qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
            }
          }
        }
        float zm0 = 0.f, zm1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < RT; ++mt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) zc[mt][e] *= slog2;
          zm0 = fmaxf(zm0, fmaxf(fabsf(zc[mt][0]), fabsf(zc[mt][2])));
          zm1 = fmaxf(zm1, fmaxf(fabsf(zc[mt][1]), fabsf(zc[mt][3])));
        }
        zm0 = warp_max_rows(zm0);
        zm1 = warp_max_rows(zm1);
        const float zs0 = pow2_down(zm0), zs1 = pow2_down(zm1);  // per column 2t, 2t + 1
#pragma unroll
        for (int mt = 0; mt < RT; ++mt)
          c_to_b(zc[mt][0] * zs0, zc[mt][1] * zs1, zc[mt][2] * zs0, zc[mt][3] * zs1, bs.zh[mt][0], bs.zl[mt][0],
                 bs.zh[mt][1], bs.zl[mt][1]);
        bs.us0 = 1.f / zs0;
        bs.us1 = 1.f / zs1;
#pragma unroll
        for (int i = 0; i < RT; ++i) bs.w[i][0] = bs.w[i][1] = bs.w[i][2] = bs.w[i][3] = 0.f;
        bs.pa0 = bs.pa1 = 0.f;
        }
        break;
      }
      case kU: {
        if (!alive) break;
        // this warp's 64 U rows: m-tiles 4 warp .. 4 warp + 3.  U is stored as 8x8 core
        // matrices (8 tokens x 8 r, 128 contiguous bytes; tc_u_off): ldmatrix gives the A
        // fragments of U (m = tokens, k = r) and, transposed, those of U^T (m = r, k = tokens).
        constexpr int MT = 4;
        const int mi = lane >> 3, mrow = lane & 7;  // this lane's matrix and row of an ldmatrix
        // byte offset of core matrix (8-token group starting at token tk, r group rg)
        auto core = [&](int tk, int rg) -> uint32_t {
          return (uint32_t)((tk >> 7) * 256 * r8 + ((tk & 127) >> 3) * 16 * r8 + rg * 128 + mrow * 16);
        };
        float s[MT][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
        // A fragments of U for m-tile mt (m = tokens, k = r)
        auto load_u = [&](int mt, uint4 (&uv)[RT]) {
          const int t0 = 64 * warp + 16 * mt;
#pragma unroll
          for (int kk = 0; kk < RT; ++kk) {
            uv[kk] = make_uint4(0u, 0u, 0u, 0u);
            if (kk < nkk) {  // a0..a3: (tokens 0-7 | 8-15) x (r 0-7 | 8-15) of the tile
              uv[kk] = ldsm4(sb + core(t0 + 8 * (mi & 1), 2 * kk + (mi >> 1)));
            } else if (kk < nrt) {  // a half-width tile: a0, a1 (r 0-7)
              const uint2 h = ldsm2(sb + core(t0 + 8 * (mi & 1), 2 * kk));
              uv[kk].x = h.x;
              uv[kk].y = h.y;
            }
          }
        };
        if constexpr (ROPE) {
          // Un-rotated pool: score against the rebuilt keys K_hat = a_k + U V_K (m = tokens,
          // n = channels, fp32 accumulators), each pair (j, j + h) turned to its token's
          // position 256 b + i, then S = K_hat q with K_hat as fp16 hi + lo (its accumulators
          // are the A fragments).  Channels go in chunks of two k tiles: a rotated pair
          // (kt, kt + h/16) or two unrotated ones, so that V_K's operand registers serve
          // all four m-tiles of the warp.
          const uint32_t vk = bs.hsb + (uint32_t)L.off_vk;
          const __half* akp = reinterpret_cast<const __half*>(smem + (bs.hsb - sbase));
          const int hk = rr.h / 16, nro = r8 >> 3;
          const int P00 = 256 * ch.blk + 64 * warp + gq;  // position of row gq of m-tile 0
          float sacc[MT][4];
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            const bool rot = c < hk;
            const int ka = rot ? c : 2 * c, kb = rot ? c + hk : 2 * c + 1;
            const int nts[4] = {2 * ka, 2 * ka + 1, 2 * kb, 2 * kb + 1};
            // V_K as B fragments (k = r, n = channel): its stored 8x8 blocks (r octet x
            // channel octet, lane L holding r 8o + L/4, channels 2(L%4)..) transposed in registers
            // (n-tiles 2k, 2k + 1 sit in the same 16-byte lane word of their 32-channel group)
            uint32_t bf[4][RT][2];
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
              const int kx = p2 ? kb : ka;
              const uint32_t col = (uint32_t)((kx >> 1) * 512 + lane * 16);
              const bool hi = (kx & 1) != 0;  // n-tiles 2kx, 2kx + 1 are words 2, 3 (else 0, 1)
#pragma unroll
              for (int kk = 0; kk < RT; ++kk) {
                bf[2 * p2][kk][0] = bf[2 * p2][kk][1] = bf[2 * p2 + 1][kk][0] = bf[2 * p2 + 1][kk][1] = 0u;
                if (kk < nrt) {
                  const uint4 w0 = lds128(vk + (uint32_t)(2 * kk) * 16u * D + col);
                  bf[2 * p2][kk][0] = movtrans(hi ? w0.z : w0.x);
                  bf[2 * p2 + 1][kk][0] = movtrans(hi ? w0.w : w0.y);
                  if (2 * kk + 1 < nro) {
                    const uint4 w1 = lds128(vk + (uint32_t)(2 * kk + 1) * 16u * D + col);
                    bf[2 * p2][kk][1] = movtrans(hi ? w1.z : w1.x);
                    bf[2 * p2 + 1][kk][1] = movtrans(hi ? w1.w : w1.y);
                  }
                }
              }
            }
            float2 akv[4], pg[2][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) akv[i] = __half22float2(*reinterpret_cast<const __half2*>(akp + 8 * nts[i] + 2 * t));
            if (rot) {  // page entries of block b for this lane's pairs j = 8 n + 2t + e, n = nts[0], nts[1]
#pragma unroll
              for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e) pg[i][e] = __ldg(rr.tab + (size_t)ch.blk * rr.h + 8 * nts[i] + 2 * t + e);
            }
            const uint32_t qa0 = lds32(qrow + (uint32_t)(16 * ka + 2 * t) * 2u);
            const uint32_t qa1 = lds32(qrow + (uint32_t)(16 * ka + 8 + 2 * t) * 2u);
            const uint32_t qb0 = lds32(qrow + (uint32_t)(16 * kb + 2 * t) * 2u);
            const uint32_t qb1 = lds32(qrow + (uint32_t)(16 * kb + 8 + 2 * t) * 2u);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              uint4 uv[RT];
              load_u(mt, uv);
              float kh[4][4];  // [n-tile][row gq: channels 2t, 2t+1 | row gq + 8: the same]
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                kh[i][0] = akv[i].x;
                kh[i][1] = akv[i].y;
                kh[i][2] = akv[i].x;
                kh[i][3] = akv[i].y;
#pragma unroll
                for (int kk = 0; kk < RT; ++kk)
                  if (kk < nrt) mma16816(kh[i], uv[kk].x, uv[kk].y, uv[kk].z, uv[kk].w, bf[i][kk][0], bf[i][kk][1]);
              }
              if (rot) {
                // position 256 b + 16 m + i: m = 4 warp + mt, i = gq or gq + 8
                const int m16 = ((P00 + 16 * mt) >> 4) & 15;
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const int j = 8 * nts[i] + 2 * t + e;
                    const float2 pm = cmul(pg[i][e], rr.s16[m16 * kRopeRow + j]);
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                      rot_pair(kh[i][2 * r + e], kh[i + 2][2 * r + e], cmul(pm, rr.s1[(gq + 8 * r) * kRopeRow + j]));
                  }
              }
              uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
              split_half2(kh[0][0], kh[0][1], h0, l0);  // a0: row gq, channels 16 ka + 2t..
              split_half2(kh[0][2], kh[0][3], h1, l1);  // a1: row gq + 8
              split_half2(kh[1][0], kh[1][1], h2, l2);  // a2: row gq, channels 16 ka + 8 + 2t..
              split_half2(kh[1][2], kh[1][3], h3, l3);  // a3: row gq + 8
              mma16816(sacc[mt], h0, h1, h2, h3, qa0, qa1);
              mma16816(sacc[mt], l0, l1, l2, l3, qa0, qa1);
              split_half2(kh[2][0], kh[2][1], h0, l0);
              split_half2(kh[2][2], kh[2][3], h1, l1);
              split_half2(kh[3][0], kh[3][1], h2, l2);
              split_half2(kh[3][2], kh[3][3], h3, l3);
              mma16816(sacc[mt], h0, h1, h2, h3, qb0, qb1);
              mma16816(sacc[mt], l0, l1, l2, l3, qb0, qb1);
            }
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t wsel = mt < 2 ? bs.mk0 : bs.mk1;
            const bool m0 = (wsel >> ((mt & 1) * 16 + gq)) & 1u;
            const bool m1 = (wsel >> ((mt & 1) * 16 + gq + 8)) & 1u;
            s[mt][0] = m0 ? -INFINITY : sacc[mt][0] * slog2;
            s[mt][1] = m0 ? -INFINITY : sacc[mt][1] * slog2;
            s[mt][2] = m1 ? -INFINITY : sacc[mt][2] * slog2;
            s[mt][3] = m1 ? -INFINITY : sacc[mt][3] * slog2;
            mx0 = fmaxf(mx0, fmaxf(s[mt][0], s[mt][2]));
            mx1 = fmaxf(mx1, fmaxf(s[mt][1], s[mt][3]));
          }
        } else {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint4 uv[RT];
          load_u(mt, uv);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < RT; ++kk) {
            if (kk < nrt) {
              mma16816(acc, uv[kk].x, uv[kk].y, uv[kk].z, uv[kk].w, bs.zh[kk][0], bs.zh[kk][1]);
              mma16816(acc, uv[kk].x, uv[kk].y, uv[kk].z, uv[kk].w, bs.zl[kk][0], bs.zl[kk][1]);
            }
          }
          const uint32_t wsel = mt < 2 ? bs.mk0 : bs.mk1;
          const bool m0 = (wsel >> ((mt & 1) * 16 + gq)) & 1u;
          const bool m1 = (wsel >> ((mt & 1) * 16 + gq + 8)) & 1u;
          s[mt][0] = m0 ? -INFINITY : fmaf(acc[0], bs.us0, bs.base0);
          s[mt][1] = m0 ? -INFINITY : fmaf(acc[1], bs.us1, bs.base1);
          s[mt][2] = m1 ? -INFINITY : fmaf(acc[2], bs.us0, bs.base0);
          s[mt][3] = m1 ? -INFINITY : fmaf(acc[3], bs.us1, bs.base1);
          mx0 = fmaxf(mx0, fmaxf(s[mt][0], s[mt][2]));
          mx1 = fmaxf(mx1, fmaxf(s[mt][1], s[mt][3]));
        }
        }
        float sc0, sc1, ms0, ms1;
        raise_max<D>(st, mx0, mx1, sc0, sc1, ms0, ms1);
        bs.pa0 *= sc0;
        bs.pa1 *= sc1;
#pragma unroll
        for (int i = 0; i < RT; ++i) { bs.w[i][0] *= sc0; bs.w[i][1] *= sc1; bs.w[i][2] *= sc0; bs.w[i][3] *= sc1; }
        // p, and w += U^T p (U^T fragments straight from shared memory)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int t0 = 64 * warp + 16 * mt;
          uint4 uv[RT];
#pragma unroll
          for (int mr = 0; mr < RT; ++mr) {
            uv[mr] = make_uint4(0u, 0u, 0u, 0u);
            if (mr < nkk) {  // a0..a3: (r 0-7 | 8-15) x (tokens 0-7 | 8-15), transposed core matrices
              uv[mr] = ldsm4t(sb + core(t0 + 8 * (mi >> 1), 2 * mr + (mi & 1)));
            } else if (mr < nrt) {  // a half-width tile: a0, a2 (r 0-7)
              const uint2 h = ldsm2t(sb + core(t0 + 8 * (mi & 1), 2 * mr));
              uv[mr].x = h.x;
              uv[mr].z = h.y;
            }
          }
          float p[4];
          p[0] = gv0 ? fast_exp2(s[mt][0] - ms0) : 0.f;
          p[1] = gv1 ? fast_exp2(s[mt][1] - ms1) : 0.f;
          p[2] = gv0 ? fast_exp2(s[mt][2] - ms0) : 0.f;
          p[3] = gv1 ? fast_exp2(s[mt][3] - ms1) : 0.f;
          st.l0 += p[0] + p[2];
          st.l1 += p[1] + p[3];
          bs.pa0 += p[0] + p[2];
          bs.pa1 += p[1] + p[3];
          uint32_t bh0, bl0, bh1, bl1;
          c_to_b(p[0], p[1], p[2], p[3], bh0, bl0, bh1, bl1);
#pragma unroll
          for (int mr = 0; mr < RT; ++mr) {
            if (mr < nrt) {
              mma16816(bs.w[mr], uv[mr].x, uv[mr].y, uv[mr].z, uv[mr].w, bh0, bh1);
              mma16816(bs.w[mr], uv[mr].x, uv[mr].y, uv[mr].z, uv[mr].w, bl0, bl1);
            }
          }
        }
        break;
      }
      case kVV: {
        // o += V_V^T w + (sum p) a_v, in this warp's own frame
        const float pa0 = warp_sum_rows(bs.pa0), pa1 = warp_sum_rows(bs.pa1);
        float wm0 = 0.f, wm1 = 0.f;
#pragma unroll
        for (int kk = 0; kk < RT; ++kk) {
          wm0 = fmaxf(wm0, fmaxf(fabsf(bs.w[kk][0]), fabsf(bs.w[kk][2])));
          wm1 = fmaxf(wm1, fmaxf(fabsf(bs.w[kk][1]), fabsf(bs.w[kk][3])));
        }
        wm0 = warp_max_rows(wm0);
        wm1 = warp_max_rows(wm1);
        const float ws0 = pow2_down(wm0), ws1 = pow2_down(wm1);  // per column 2t, 2t + 1
        uint32_t wh[RT][2], wl[RT][2];
#pragma unroll
        for (int kk = 0; kk < RT; ++kk)
          c_to_b(bs.w[kk][0] * ws0, bs.w[kk][1] * ws1, bs.w[kk][2] * ws0, bs.w[kk][3] * ws1, wh[kk][0], wl[kk][0],
                 wh[kk][1], wl[kk][1]);
        const float wu0 = 1.f / ws0, wu1 = 1.f / ws1;
        const __half* avp = av;  // this block's a_v (this warp's copy, written at its head)
#pragma unroll
        for (int md = 0; md < KT; ++md) {
          float cv[4] = {0.f, 0.f, 0.f, 0.f};
          const uint32_t mb = sb + (uint32_t)(md * 16 * r8 * 2);
#pragma unroll
          for (int kk = 0; kk < RT; ++kk) {
            if (alive && kk < nkk) {
              const uint4 v = lds128(mb + (uint32_t)(kk * 512 + lane * 16));
              mma16816(cv, v.x, v.y, v.z, v.w, wh[kk][0], wh[kk][1]);
              mma16816(cv, v.x, v.y, v.z, v.w, wl[kk][0], wl[kk][1]);
            } else if (alive && kk == nkk && rtail) {
              const uint2 v = lds64(mb + (uint32_t)(kk * 512 + lane * 8));
              mma1688(cv, v.x, v.y, wh[kk][0]);
              mma1688(cv, v.x, v.y, wl[kk][0]);
            }
          }
          const float av0 = __half2float(avp[16 * md + gq]), av1 = __half2float(avp[16 * md + gq + 8]);
          st.o[md][0] += fmaf(cv[0], wu0, pa0 * av0);
          st.o[md][1] += fmaf(cv[1], wu1, pa1 * av0);
          st.o[md][2] += fmaf(cv[2], wu0, pa0 * av1);
          st.o[md][3] += fmaf(cv[3], wu1, pa1 * av1);
        }
        break;
      }
      default:
        break;
    }
    __syncwarp();
    if constexpr (ROPE) {
      if (alive && ch.kind == kHead) {
        held = bi;  // its a_k and V_K are read at the U chunk
      } else {
        if (lane == 0) mbar_arrive(&empty[bi]);
        if (held >= 0 && (ch.kind == kU || !alive)) {
          if (lane == 0) mbar_arrive(&empty[held]);
          held = -1;
        }
      }
    } else {
      if (lane == 0) mbar_arrive(&empty[bi]);
    }
  }
  if (ROPE && held >= 0 && lane == 0) mbar_arrive(&empty[held]);
  // this warp's partial record (m, l, o) over every token it scored; the combine merges them
  const float l0 = warp_sum_rows(st.l0), l1 = warp_sum_rows(st.l1);
  float* rec = a.partials + (((size_t)u * a.n_r + range) * kConsumers + warp) * (16 + 8 * D);
  if (lane < 4) {
    rec[2 * t] = alive ? st.m0 : -INFINITY;
    rec[2 * t + 1] = alive ? st.m1 : -INFINITY;
    rec[8 + 2 * t] = alive ? l0 : 0.f;
    rec[8 + 2 * t + 1] = alive ? l1 : 0.f;
  }
#pragma unroll
  for (int md = 0; md < KT; ++md) {
    const int d0 = 16 * md + gq;
    if (gv0) {
      rec[16 + (2 * t) * D + d0] = alive ? st.o[md][0] : 0.f;
      rec[16 + (2 * t) * D + d0 + 8] = alive ? st.o[md][2] : 0.f;
    }
    if (gv1) {
      rec[16 + (2 * t + 1) * D + d0] = alive ? st.o[md][1] : 0.f;
      rec[16 + (2 * t + 1) * D + d0 + 8] = alive ? st.o[md][3] : 0.f;
    }
  }
}

// ranges per unit: fill whole waves of kCtasPerSm CTAs per SM, preferring one wave
int ranges_per_unit(int units) {
  const long target = (long)kCtasPerSm * sm_count();
  int best = 1;
  double best_score = -1.0;
  for (int n = 1; n <= kMaxRanges; ++n) {
    const long ctas = (long)units * n;
    const long waves = (ctas + target - 1) / target;
    const double score = (double)ctas / (double)(waves * target) - 0.06 * (double)(waves - 1);
    if (score > best_score + 1e-9) { best_score = score; best = n; }
  }
  return best;
}

// bytes of the work list's pieces
uint64_t win_stage_bytes(const Layout& L, int s) {
  const int n = L.W16 - s * kStageTok < kStageTok ? L.W16 - s * kStageTok : kStageTok;
  return (uint64_t)n * 4 * L.d;
}
// Balancing weight of a block item: its bytes, the low-rank part's times
// kLowRankWeight (its z, U and V_V products cost the consumer warps about
// three times as long per byte as an exact stage; measured on GB300).
constexpr uint64_t kLowRankWeight = 3;
uint64_t block_item_bytes(const Layout& L, int k) {  // k = 0: low-rank part; k >= 1: residual stage k - 1
  if (k == 0) return kLowRankWeight * (L.off_u + (L.off_res - L.off_u) + (L.block_bytes - L.off_vv));
  const int t0 = (k - 1) * kStageTok;
  const int n = L.R8 - t0 < kStageTok ? L.R8 - t0 : kStageTok;
  // quantised rows: their bytes, weighted 2x for the dequantisation in registers
  return L.qbits ? (uint64_t)(n / 16) * L.qgb * 2 : (uint64_t)n * 4 * L.d;
}

// Cut one unit's work list into n_r ranges.  Every range starts with one
// window stage where there are enough (so it has work while the router runs);
// the block items are cut into contiguous runs and the other window stages are
// spread over the ranges, for the smallest capacity (largest range, in weight)
// that holds everything: binary search on the capacity, with the block runs
// filled in order up to it (exact for contiguous runs) and the spare window
// stages placed in whatever room is left.  Range i reads window stages
// [tab 0, tab 1) and block items [tab 2, tab 3).
void fill_ranges(const Layout& L, int K_eff, int nres, int n_wst, int n_r, int (*tab)[4]) {
  const int per = 1 + nres;
  const int n_it = K_eff * per;
  const uint64_t wst = win_stage_bytes(L, 0);  // the last stage may be shorter: counted as full
  const int base = n_wst >= n_r ? 1 : 0;
  const int spare = n_wst - base * n_r;
  std::vector<uint64_t> load(n_r, 0);
  std::vector<int> nw(n_r, base);
  uint64_t lo = base * wst, hi = (uint64_t)n_wst * wst;
  for (int k = 0; k < per; ++k) {
    const uint64_t b = block_item_bytes(L, k);
    lo = b > lo ? b : lo;
    hi += b * (uint64_t)K_eff;
  }
  auto fill = [&](uint64_t cap, bool write) {
    int x = 0;
    uint64_t room = 0;  // window stages that still fit
    for (int i = 0; i < n_r; ++i) {
      uint64_t acc = base * wst;
      if (write) tab[i][2] = x;
      while (x < n_it && acc + block_item_bytes(L, x % per) <= cap) acc += block_item_bytes(L, x++ % per);
      if (write) { tab[i][3] = x; load[i] = acc; }
      room += (wst && cap >= acc) ? (cap - acc) / wst : 0;
    }
    return x == n_it && room >= (uint64_t)spare;
  };
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo) / 2;
    if (fill(mid, false)) hi = mid; else lo = mid + 1;
  }
  fill(lo, true);
  for (int s = 0; s < spare; ++s) {  // lightest range first
    int best = 0;
    for (int i = 1; i < n_r; ++i) best = load[i] < load[best] ? i : best;
    ++nw[best];
    load[best] += wst;
  }
  int w = 0;
  for (int i = 0; i < n_r; ++i) {
    tab[i][0] = w;
    w += nw[i];
    tab[i][1] = w;
  }
}

template <int D, int R8S, bool ROPE>
cudaError_t launch_one(const AttendArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attend_kernel<D, R8S, ROPE>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the router's grid
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attend_kernel<D, R8S, ROPE>, a);
}

// Kernel instance for a layout: compile-time ranks for the padded ranks of the
// Qwen2.5-shaped workloads at head_dim 128 (16, 24, 32, 48), otherwise the
// run-time rank with 2, 4 or 8 r tiles.
int instance_r8s(int d, int r8) {
  if (d == 128 && (r8 == 16 || r8 == 24 || r8 == 32 || r8 == 48)) return r8;
  return r8 <= 32 ? -2 : (r8 <= 64 ? -4 : -8);
}

#define DKV_INSTANCES(X)                                                                                  \
  X(128, 16) X(128, 24) X(128, 32) X(128, 48) X(128, -2) X(128, -4) X(128, -8) X(64, -2) X(64, -4) X(64, -8)
// the un-rotated pool's instances (ranks up to 64)
#define DKV_ROPE_INSTANCES(X) \
  X(128, 16) X(128, 24) X(128, 32) X(128, 48) X(128, -2) X(128, -4) X(64, -2) X(64, -4)

cudaError_t launch_instance(int d, int r8s, bool rope, const AttendArgs& a, int grid, size_t smem, cudaStream_t s) {
#define DKV_LAUNCH(D_, R_) \
  if (!rope && d == D_ && r8s == R_) return launch_one<D_, R_, false>(a, grid, smem, s);
  DKV_INSTANCES(DKV_LAUNCH)
#undef DKV_LAUNCH
#define DKV_LAUNCH_ROPE(D_, R_) \
  if (rope && d == D_ && r8s == R_) return launch_one<D_, R_, true>(a, grid, smem, s);
  DKV_ROPE_INSTANCES(DKV_LAUNCH_ROPE)
#undef DKV_LAUNCH_ROPE
  return cudaErrorInvalidValue;
}
// Arguments shared by every attention launch of a call (mode and outputs set by the caller).
AttendArgs make_args(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                     const uint8_t* cache, uint8_t* ws, size_t* smem) {
  AttendArgs a;
  a.L = L;
  a.G = n_q_heads / n_kv_heads;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.K_eff = P.K_eff;
  a.n_r = P.n_items / kConsumers;
  a.nres = (L.R8 + kStageTok - 1) / kStageTok;
  a.n_wst = P.n_wchunks;
  a.mode = 0;
  if (a.n_r <= kMaxRanges) fill_ranges(L, a.K_eff, a.nres, a.n_wst, a.n_r, a.tab);
  const size_t extra = smem_extra(L.rope != 0);
  a.ring = (int)((kSmemPerCta - extra) / 128 * 128);
  // 64 KB in flight per CTA (about 19 MB over the grid) covers the memory latency at full
  // bandwidth; measured on GB300 against 16, 24, 40 KB and the whole ring (about 103 KB)
  a.inflight = a.ring < 65536 ? (uint32_t)a.ring : 65536u;
  debug_limits(&a.stop_after, &a.wait_limit);
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)L.d);
  a.q = q;
  a.cache = cache;
  a.routed = reinterpret_cast<const int32_t*>(ws + P.off_routed);
  a.routed_out = nullptr;
  a.partials = reinterpret_cast<float*>(ws + P.off_partials);
  a.err = reinterpret_cast<uint32_t*>(ws);
  *smem = (size_t)a.ring + extra;
  return a;
}

}  // namespace

namespace {
std::atomic<int> g_stop_after{-1};
std::atomic<uint32_t> g_wait_polls{kWaitLimit};
}  // namespace
void debug_limits(int* stop_after, uint32_t* wait_polls) {
  *stop_after = g_stop_after.load(std::memory_order_relaxed);
  *wait_polls = g_wait_polls.load(std::memory_order_relaxed);
}
namespace {
std::atomic<int> g_programmatic{1};
}  // namespace
bool programmatic_launch() { return g_programmatic.load(std::memory_order_relaxed) != 0; }
void set_programmatic_launch(bool on) { g_programmatic.store(on ? 1 : 0, std::memory_order_relaxed); }
void set_debug_limits(int stop_after, uint32_t wait_polls) {
  g_stop_after.store(stop_after < 0 ? -1 : stop_after, std::memory_order_relaxed);
  g_wait_polls.store(wait_polls ? wait_polls : kWaitLimit, std::memory_order_relaxed);
}

// Multiprocessors of the current device (cached per device; a host without a
// usable device plans for 148).
int sm_count() {
  static std::atomic<int> n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = n[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    n[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

DecodePlan plan_decode(const Layout& L, int n_q_heads, int n_kv_heads, int top_k) {
  DecodePlan P;
  P.K_eff = (top_k == 0 || top_k >= L.NB) ? L.NB : top_k;
  const bool tc = tc_eligible(L, n_q_heads, n_kv_heads);
  P.wchunk_tokens = tc ? tc_window_tokens() : kStageTok;
  P.n_wchunks = (L.W16 + P.wchunk_tokens - 1) / P.wchunk_tokens;
  if (tc) {
    P.n_items = P.K_eff + P.n_wchunks;
  } else {
    // one partial record per (unit, range, consumer warp)
    const int nres = (L.R8 + kStageTok - 1) / kStageTok;
    const int n_list = P.n_wchunks + P.K_eff * (1 + nres);
    int n_r = ranges_per_unit(L.units);
    n_r = n_r < n_list ? n_r : n_list;
    P.n_items = (n_r < 1 ? 1 : n_r) * kConsumers;
  }
  P.off_sched = kWsHeader;  // scheduler counters of the tensor-core kernel
  P.off_routed = round_up(P.off_sched + 8, 256);
  P.off_partials = round_up(P.off_routed + (size_t)L.units * P.K_eff * 4, 256);
  P.ws_bytes = P.off_partials + (size_t)L.units * P.n_items * (16 + 8 * L.d) * 4;
  return P;
}

cudaError_t launch_attend_mode(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                               const uint8_t* cache, uint8_t* ws, float* out, float* lse, int mode,
                               int32_t* routed_out, cudaStream_t s) {
  size_t smem;
  AttendArgs a = make_args(L, P, n_q_heads, n_kv_heads, q, cache, ws, &smem);
  if (a.n_r > kMaxRanges) return cudaErrorInvalidValue;
  a.mode = mode;
  a.routed_out = routed_out;
  const cudaError_t e = launch_instance(L.d, instance_r8s(L.d, L.r8), L.rope != 0, a, L.units * a.n_r, smem, s);
  if (e != cudaSuccess || out == nullptr) return e;
  return launch_combine(L, P, L.units / n_kv_heads, n_q_heads, n_kv_heads, a.partials, out, lse, s);
}

cudaError_t launch_attend(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s) {
  if (tc_eligible(L, n_q_heads, n_kv_heads)) return launch_attend_tc(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, s);
  return launch_attend_mode(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, 0, nullptr, s);
}

int decode_launches(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads) {
  const bool all = P.K_eff == L.NB && !tc_eligible(L, n_q_heads, n_kv_heads);  // no router grid
  return (P.K_eff > 0 && !all) ? 3 : 2;  // router, attention, combine
}

cudaError_t launch_decode(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, int32_t* routed_out,
                          cudaStream_t s) {
  if (tc_eligible(L, n_q_heads, n_kv_heads)) {
    cudaError_t e = cudaSuccess;
    if (P.K_eff > 0) e = launch_route(L, P, n_q_heads, n_kv_heads, q, cache, ws, routed_out, s);
    return e == cudaSuccess ? launch_attend_tc(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, s) : e;
  }
  if (P.K_eff == L.NB)  // every block (or none) is routed: no router grid
    return launch_attend_mode(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, kModeAll, routed_out, s);
  const cudaError_t e = launch_route(L, P, n_q_heads, n_kv_heads, q, cache, ws, routed_out, s);
  return e == cudaSuccess ? launch_attend_mode(L, P, n_q_heads, n_kv_heads, q, cache, ws, out, lse, 0, nullptr, s) : e;
}

}  // namespace dkv
