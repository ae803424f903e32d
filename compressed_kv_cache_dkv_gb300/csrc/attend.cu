// Block + window attention of the DKV decode path.
//
// One CTA per work item of a unit (a routed block, or a chunk of the exact
// recency window).  Warp 4 is the producer: its lane 0 streams the item's
// packed bytes, chunk by chunk, into a ring of shared-memory slots with 1-D
// TMA bulk copies (cp.async.bulk + mbarrier complete_tx).  Warps 0-3 are the
// consumers; every matrix product runs on the tensor cores through
// mma.sync m16n8k16 / m16n8k8 (fp16 operands, fp32 accumulate) with the
// tokens (or the head dimension) in M and the GQA group in N = 8.
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
// partials with an fp32 log-sum-exp reduction.  Scores are kept in fp32; the
// fp32 operands of a product (z, p, w) are split into an fp16 pair hi + lo so
// the tensor-core products carry about 22 bits.
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

struct AttendArgs {
  Layout L;
  int G, Hq, Hkv, K_eff, n_items, nslot, slot_bytes, xtok;
  float scale_log2;  // log2(e) / sqrt(d)
  const __half* q;
  const uint8_t* cache;
  const int32_t* routed;
  float* partials;
  uint32_t* err;
  uint32_t* counters;  // per-unit arrival counters (fused merge)
  float* out;          // nullptr: partials only
  float* lse;
};

struct Chunk {
  uint64_t src;   // byte offset from the cache base
  uint32_t bytes;
  int kind;       // 0 head, 1 U, 2 exact, 3 V_V
  int tok0;       // first token (U row / residual row / window token)
  int ntok;       // stored tokens in the chunk (multiple of 8)
};

struct ItemInfo {
  bool is_block;
  int n_chunks;
  int n_u, n_x;          // U chunks and exact chunks
  uint64_t base;         // block record or window offset
  int tok0, ntok;        // window: first stored token and stored tokens of the item
  int nvalid;            // exact tokens that are real (R for residuals, W for the window)
};

__device__ inline Chunk item_chunk(const AttendArgs& a, const ItemInfo& it, int k) {
  const Layout& L = a.L;
  Chunk c;
  if (it.is_block) {
    if (k == 0) {
      c.src = it.base; c.bytes = (uint32_t)L.off_u; c.kind = 0; c.tok0 = 0; c.ntok = 0;
    } else if (k <= it.n_u) {
      int t0 = (k - 1) * kUTok;
      c.src = it.base + L.off_u + (uint64_t)t0 * 2 * L.r8;
      c.bytes = (uint32_t)(kUTok * 2 * L.r8); c.kind = 1; c.tok0 = t0; c.ntok = kUTok;
    } else if (k <= it.n_u + it.n_x) {
      int t0 = (k - 1 - it.n_u) * a.xtok;
      int n = min(a.xtok, L.R8 - t0);
      c.src = it.base + L.off_res + (uint64_t)t0 * 4 * L.d;
      c.bytes = (uint32_t)(n * 4 * L.d); c.kind = 2; c.tok0 = t0; c.ntok = n;
    } else {
      c.src = it.base + L.off_vv; c.bytes = (uint32_t)(2 * L.r8 * L.d); c.kind = 3; c.tok0 = 0; c.ntok = 0;
    }
  } else {
    int t0 = it.tok0 + k * a.xtok;
    int n = min(a.xtok, it.tok0 + it.ntok - t0);
    c.src = it.base + (uint64_t)t0 * 4 * L.d;
    c.bytes = (uint32_t)(n * 4 * L.d); c.kind = 2; c.tok0 = t0; c.ntok = n;
  }
  return c;
}

__device__ inline int chunk_owner(const ItemInfo& it, int k) {
  if (it.is_block) {
    if (k == 0 || k == it.n_chunks - 1) return -1;  // all consumer warps
    return (k - 1) % kConsumers;
  }
  return k % kConsumers;
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

// Online-softmax state of one consumer warp, columns g = 2t, 2t+1 of the C fragment.
template <int D, int RT>
struct WarpState {
  float m[2], l[2], pa[2];
  float w[RT][4];
  float o[D / 16][4];
};

template <int D, int RT>
__device__ inline void rescale(WarpState<D, RT>& st, const float (&s)[4], float (&p)[4], bool gv0, bool gv1) {
  float mx0 = warp_max_rows(fmaxf(s[0], s[2]));
  float mx1 = warp_max_rows(fmaxf(s[1], s[3]));
  float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
  float ms0 = (mn0 == -INFINITY) ? 0.f : mn0;
  float ms1 = (mn1 == -INFINITY) ? 0.f : mn1;
  float sc0 = exp2f(st.m[0] - ms0), sc1 = exp2f(st.m[1] - ms1);  // exp2(-inf) = 0
  p[0] = gv0 ? exp2f(s[0] - ms0) : 0.f;
  p[1] = gv1 ? exp2f(s[1] - ms1) : 0.f;
  p[2] = gv0 ? exp2f(s[2] - ms0) : 0.f;
  p[3] = gv1 ? exp2f(s[3] - ms1) : 0.f;
  st.m[0] = mn0;
  st.m[1] = mn1;
  st.l[0] *= sc0; st.l[1] *= sc1;
  st.pa[0] *= sc0; st.pa[1] *= sc1;
#pragma unroll
  for (int i = 0; i < RT; ++i) { st.w[i][0] *= sc0; st.w[i][1] *= sc1; st.w[i][2] *= sc0; st.w[i][3] *= sc1; }
#pragma unroll
  for (int i = 0; i < D / 16; ++i) { st.o[i][0] *= sc0; st.o[i][1] *= sc1; st.o[i][2] *= sc0; st.o[i][3] *= sc1; }
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

template <int D, int RT>
__global__ void __launch_bounds__(kThreads, 2) attend_kernel(AttendArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout& L = a.L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = lane & 3, gq = lane >> 2;
  const int u = blockIdx.y, item = blockIdx.x;
  const int bseq = u / a.Hkv, h = u % a.Hkv;
  const int r8 = L.r8;
  const int nkk = r8 >> 4;                 // full 16-wide k tiles of r
  const bool rtail = (r8 & 15) != 0;       // one 8-wide tail
  const int nrt = nkk + (rtail ? 1 : 0);   // r tiles

  // ---- shared memory carve-up
  uint8_t* slots = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.nslot * a.slot_bytes);
  uint64_t* empty = full + kMaxSlots;
  float2* zbuf = reinterpret_cast<float2*>(empty + kMaxSlots);          // [r8/8][32]
  float* wbuf = reinterpret_cast<float*>(zbuf + (RT * 2) * 32);         // [RT*16][8]
  float* obuf = wbuf + RT * 16 * 8;                                     // [D][8]
  float* mbuf = obuf + D * 8;                                           // [4][8]
  float* lbuf = mbuf + 32;
  float* pabuf = lbuf + 32;
  uint32_t* maskbuf = reinterpret_cast<uint32_t*>(pabuf + 32);         // [8] residual mask bits
  __half* av = reinterpret_cast<__half*>(maskbuf + 8);                  // [D]

  // ---- work item
  ItemInfo it;
  uint64_t unit_base = (uint64_t)u * L.unit_stride;
  bool item_ok = true;
  if (item < a.K_eff) {
    int blk = a.routed[u * a.K_eff + item];
    if (blk < 0 || blk >= L.NB) {
      item_ok = false;
      if (threadIdx.x == 0) raise_error(a.err, DKV_DEVERR_INDEX);
      blk = 0;
    }
    it.is_block = true;
    it.n_u = L.r8 > 0 ? 256 / kUTok : 256 / kUTok;
    it.n_x = (L.R8 + a.xtok - 1) / a.xtok;
    it.n_chunks = 1 + it.n_u + it.n_x + 1;
    it.base = unit_base + L.off_blocks + (uint64_t)blk * L.block_stride;
    it.tok0 = 0; it.ntok = 0; it.nvalid = L.R;
  } else {
    int wc = item - a.K_eff;
    it.is_block = false;
    it.n_u = 0;
    it.tok0 = wc * kWindowChunk;
    it.ntok = min(kWindowChunk, L.W16 - it.tok0);
    it.n_x = (it.ntok + a.xtok - 1) / a.xtok;
    it.n_chunks = it.n_x;
    it.base = unit_base + L.off_window;
    it.nvalid = L.W;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.nslot; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    fence_mbar_init();
  }
  __syncthreads();

  // =========================== producer warp
  if (warp == kConsumers) {
    if (lane == 0 && item_ok) {
      const uint64_t pol = policy_evict_first();
      for (int k = 0; k < it.n_chunks; ++k) {
        int slot = k % a.nslot;
        if (k >= a.nslot && !mbar_wait(&empty[slot], ((k / a.nslot) - 1) & 1, a.err)) break;
        Chunk c = item_chunk(a, it, k);
        if (c.bytes) {
          mbar_arrive_expect_tx(&full[slot], c.bytes);
          bulk_g2s(slots + (size_t)slot * a.slot_bytes, a.cache + c.src, c.bytes, &full[slot], pol);
        } else {
          mbar_arrive(&full[slot]);
        }
      }
    }
    return;
  }

  // =========================== consumer warps
  const int G = a.G;
  const bool gv0 = (2 * t) < G, gv1 = (2 * t + 1) < G;
  // q as B fragments (k = head dim, n = group): q[gq][16kt + 2t, +1] and [16kt + 8 + 2t, +1]
  uint32_t qb[D / 16][2];
  {
    const __half* qrow = a.q + ((size_t)bseq * a.Hq + (size_t)h * G + (gq < G ? gq : 0)) * D;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
      uint32_t x0 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kt + 2 * t);
      uint32_t x1 = *reinterpret_cast<const uint32_t*>(qrow + 16 * kt + 8 + 2 * t);
      qb[kt][0] = gq < G ? x0 : 0u;
      qb[kt][1] = gq < G ? x1 : 0u;
    }
  }
  WarpState<D, RT> st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = st.pa[0] = st.pa[1] = 0.f;
#pragma unroll
  for (int i = 0; i < RT; ++i) st.w[i][0] = st.w[i][1] = st.w[i][2] = st.w[i][3] = 0.f;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;

  bool ok = item_ok;
  float base0 = 0.f, base1 = 0.f;       // c q_g . a_k in base-2 units, columns 2t, 2t+1
  float us0 = 1.f, us1 = 1.f;           // power-of-two unscale of z, columns 2t, 2t+1
  uint32_t zh[RT][2], zl[RT][2];        // z as B fragments (k = r, n = group), hi and lo
  const uint32_t slot0 = smem_u32(slots);

  if (it.is_block) {
    // ---------------- head chunk: anchors, residual mask, V_K -> base and z
    ok = ok && mbar_wait(&full[0], 0, a.err);
    const __half* ak = reinterpret_cast<const __half*>(slots);
    float part = 0.f;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
      __half2 q0 = *reinterpret_cast<__half2*>(&qb[kt][0]);
      __half2 q1 = *reinterpret_cast<__half2*>(&qb[kt][1]);
      float2 qf0 = __half22float2(q0), qf1 = __half22float2(q1);
      int j0 = 16 * kt + 2 * t, j1 = j0 + 8;
      part += qf0.x * __half2float(ak[j0]) + qf0.y * __half2float(ak[j0 + 1]);
      part += qf1.x * __half2float(ak[j1]) + qf1.y * __half2float(ak[j1 + 1]);
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part *= a.scale_log2;  // base for g = gq
    base0 = __shfl_sync(0xffffffffu, part, 8 * t);
    base1 = __shfl_sync(0xffffffffu, part, 8 * t + 4);
    if (warp == 0) {
      for (int j = lane; j < D; j += 32) av[j] = reinterpret_cast<const __half*>(slots)[D + j];
      if (lane < 8) maskbuf[lane] = reinterpret_cast<const uint32_t*>(slots + L.off_mask)[lane];
    }
    // z^T = q^T V_K^T : n-tiles of 8 r-rows split across warps
    const uint32_t vk = slot0 + (uint32_t)L.off_vk;
    for (int nt = warp; nt < (r8 >> 3); nt += kConsumers) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        uint4 b = lds128(vk + (uint32_t)(nt * 8 * D * 2 + kp * 512 + lane * 16));
        mma16816(c, qb[2 * kp][0], 0u, qb[2 * kp][1], 0u, b.x, b.y);
        mma16816(c, qb[2 * kp + 1][0], 0u, qb[2 * kp + 1][1], 0u, b.z, b.w);
      }
      zbuf[nt * 32 + lane] = make_float2(c[0] * a.scale_log2, c[1] * a.scale_log2);
    }
    named_bar_sync(1, kConsumers * 32);
    if (warp == 0 && lane == 0) mbar_arrive(&empty[0]);
    // z B fragments: b0 = z[16kk + 2t, +1][gq] = zbuf[2kk][lane], b1 = zbuf[2kk+1][lane]
    float zf[RT][4];
    float zmax = 0.f;
#pragma unroll
    for (int kk = 0; kk < RT; ++kk) {
      float2 z0 = make_float2(0.f, 0.f), z1 = make_float2(0.f, 0.f);
      if (kk < nrt) {
        z0 = zbuf[(2 * kk) * 32 + lane];
        if (2 * kk + 1 < (r8 >> 3)) z1 = zbuf[(2 * kk + 1) * 32 + lane];
      }
      zf[kk][0] = z0.x; zf[kk][1] = z0.y; zf[kk][2] = z1.x; zf[kk][3] = z1.y;
      zmax = fmaxf(zmax, fmaxf(fmaxf(fabsf(z0.x), fabsf(z0.y)), fmaxf(fabsf(z1.x), fabsf(z1.y))));
    }
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

  // ---------------- private chunks (U rows and exact rows), round-robin over warps
  const int k_first = it.is_block ? 1 : 0;
  const int k_last = it.is_block ? it.n_chunks - 2 : it.n_chunks - 1;
  for (int k = k_first; k <= k_last && ok; ++k) {
    if (chunk_owner(it, k) != warp) continue;
    const int slot = k % a.nslot;
    if (!mbar_wait(&full[slot], (k / a.nslot) & 1, a.err)) { ok = false; break; }
    const Chunk c = item_chunk(a, it, k);
    const uint32_t sb = slot0 + (uint32_t)(slot * a.slot_bytes);
    if (c.kind == 1) {
      // ---- U rows: s = base + U z, online softmax, w += U^T p
#pragma unroll 1
      for (int mt = 0; mt < kUTok / 16; ++mt) {
        const uint32_t tb = sb + (uint32_t)(mt * 16 * r8 * 2);
        uint32_t ua[RT][4];
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < RT; ++kk) {
          if (kk < nkk) {
            uint4 v = lds128(tb + (uint32_t)(kk * 512 + lane * 16));
            ua[kk][0] = v.x; ua[kk][1] = v.y; ua[kk][2] = v.z; ua[kk][3] = v.w;
            mma16816(s, v.x, v.y, v.z, v.w, zh[kk][0], zh[kk][1]);
            mma16816(s, v.x, v.y, v.z, v.w, zl[kk][0], zl[kk][1]);
          } else if (kk == nkk && rtail) {
            uint2 v = lds64(tb + (uint32_t)(kk * 512 + lane * 8));
            ua[kk][0] = v.x; ua[kk][1] = v.y; ua[kk][2] = 0u; ua[kk][3] = 0u;
            mma1688(s, v.x, v.y, zh[kk][0]);
            mma1688(s, v.x, v.y, zl[kk][0]);
          }
        }
        const int tk0 = c.tok0 + mt * 16 + gq, tk1 = tk0 + 8;
        const bool m0 = (maskbuf[tk0 >> 5] >> (tk0 & 31)) & 1u;
        const bool m1 = (maskbuf[tk1 >> 5] >> (tk1 & 31)) & 1u;
        s[0] = m0 ? -INFINITY : fmaf(s[0], us0, base0);
        s[1] = m0 ? -INFINITY : fmaf(s[1], us1, base1);
        s[2] = m1 ? -INFINITY : fmaf(s[2], us0, base0);
        s[3] = m1 ? -INFINITY : fmaf(s[3], us1, base1);
        float p[4];
        rescale(st, s, p, gv0, gv1);
        st.pa[0] += p[0] + p[2];
        st.pa[1] += p[1] + p[3];
        uint32_t bh0, bl0, bh1, bl1;
        p_to_b(p, bh0, bl0, bh1, bl1);
#pragma unroll
        for (int mr = 0; mr < RT; ++mr) {
          if (mr < nrt) {
            uint32_t A0 = movtrans(ua[mr][0]);
            uint32_t A2 = movtrans(ua[mr][1]);
            uint32_t A1 = (mr < nkk) ? movtrans(ua[mr][2]) : 0u;
            uint32_t A3 = (mr < nkk) ? movtrans(ua[mr][3]) : 0u;
            mma16816(st.w[mr], A0, A1, A2, A3, bh0, bh1);
            mma16816(st.w[mr], A0, A1, A2, A3, bl0, bl1);
          }
        }
      }
    } else {
      // ---- exact rows (residuals or window): s = c q . k, online softmax, o += V^T p
      const int ng = (c.ntok + 15) >> 4;
#pragma unroll 1
      for (int gi = 0; gi < ng; ++gi) {
        const int in_g = min(16, c.ntok - gi * 16);
        const uint32_t gb = sb + (uint32_t)(gi * 64 * D);
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (in_g == 16) {
#pragma unroll
          for (int kt = 0; kt < D / 16; ++kt) {
            uint4 v = lds128(gb + (uint32_t)(kt * 512 + lane * 16));
            mma16816(s, v.x, v.y, v.z, v.w, qb[kt][0], qb[kt][1]);
          }
        } else {
#pragma unroll
          for (int kt = 0; kt < D / 16; ++kt) {
            uint2 v = lds64(gb + (uint32_t)(kt * 256 + lane * 8));
            mma16816(s, v.x, 0u, v.y, 0u, qb[kt][0], qb[kt][1]);
          }
        }
        const int tk0 = c.tok0 + gi * 16 + gq, tk1 = tk0 + 8;
        const bool v0 = tk0 < it.nvalid && (gq < in_g);
        const bool v1 = tk1 < it.nvalid && (gq + 8 < in_g);
        s[0] = v0 ? s[0] * a.scale_log2 : -INFINITY;
        s[1] = v0 ? s[1] * a.scale_log2 : -INFINITY;
        s[2] = v1 ? s[2] * a.scale_log2 : -INFINITY;
        s[3] = v1 ? s[3] * a.scale_log2 : -INFINITY;
        float p[4];
        rescale(st, s, p, gv0, gv1);
        uint32_t bh0, bl0, bh1, bl1;
        p_to_b(p, bh0, bl0, bh1, bl1);
        const uint32_t vb = gb + (uint32_t)(in_g * D * 2);
        if (in_g == 16) {
#pragma unroll
          for (int md = 0; md < D / 16; ++md) {
            uint4 v = lds128(vb + (uint32_t)(md * 512 + lane * 16));
            mma16816(st.o[md], v.x, v.y, v.z, v.w, bh0, bh1);
            mma16816(st.o[md], v.x, v.y, v.z, v.w, bl0, bl1);
          }
        } else {
#pragma unroll
          for (int md = 0; md < D / 16; ++md) {
            uint2 v = lds64(vb + (uint32_t)(md * 256 + lane * 8));
            mma1688(st.o[md], v.x, v.y, bh0);
            mma1688(st.o[md], v.x, v.y, bl0);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ---------------- merge the four warps
  st.l[0] = warp_sum_rows(st.l[0]);
  st.l[1] = warp_sum_rows(st.l[1]);
  st.pa[0] = warp_sum_rows(st.pa[0]);
  st.pa[1] = warp_sum_rows(st.pa[1]);
  if (lane < 4) { mbuf[warp * 8 + 2 * t] = st.m[0]; mbuf[warp * 8 + 2 * t + 1] = st.m[1]; }
  named_bar_sync(1, kConsumers * 32);
  float mf0 = -INFINITY, mf1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) { mf0 = fmaxf(mf0, mbuf[w * 8 + 2 * t]); mf1 = fmaxf(mf1, mbuf[w * 8 + 2 * t + 1]); }
  const float sc0 = exp2f(st.m[0] - (mf0 == -INFINITY ? 0.f : mf0));
  const float sc1 = exp2f(st.m[1] - (mf1 == -INFINITY ? 0.f : mf1));
  if (lane < 4) {
    lbuf[warp * 8 + 2 * t] = st.l[0] * sc0; lbuf[warp * 8 + 2 * t + 1] = st.l[1] * sc1;
    pabuf[warp * 8 + 2 * t] = st.pa[0] * sc0; pabuf[warp * 8 + 2 * t + 1] = st.pa[1] * sc1;
  }
  // sequential (deterministic) sum of w and o across warps
  for (int w = 0; w < kConsumers; ++w) {
    if (warp == w) {
#pragma unroll
      for (int mr = 0; mr < RT; ++mr) {
        if (it.is_block && mr < nrt) {
          const int r0 = mr * 16 + gq, r1 = r0 + 8;
          float* w0 = wbuf + r0 * 8 + 2 * t;
          float* w1 = wbuf + r1 * 8 + 2 * t;
          if (w == 0) {
            w0[0] = st.w[mr][0] * sc0; w0[1] = st.w[mr][1] * sc1;
            if (r1 < r8) { w1[0] = st.w[mr][2] * sc0; w1[1] = st.w[mr][3] * sc1; }
          } else {
            w0[0] += st.w[mr][0] * sc0; w0[1] += st.w[mr][1] * sc1;
            if (r1 < r8) { w1[0] += st.w[mr][2] * sc0; w1[1] += st.w[mr][3] * sc1; }
          }
        }
      }
#pragma unroll
      for (int md = 0; md < D / 16; ++md) {
        float* o0 = obuf + (md * 16 + gq) * 8 + 2 * t;
        float* o1 = o0 + 64;
        if (w == 0) {
          o0[0] = st.o[md][0] * sc0; o0[1] = st.o[md][1] * sc1; o1[0] = st.o[md][2] * sc0; o1[1] = st.o[md][3] * sc1;
        } else {
          o0[0] += st.o[md][0] * sc0; o0[1] += st.o[md][1] * sc1; o1[0] += st.o[md][2] * sc0; o1[1] += st.o[md][3] * sc1;
        }
      }
    }
    named_bar_sync(1, kConsumers * 32);
  }

  // ---------------- low-rank value: o += V_V^T w + (sum p) a_v
  if (it.is_block) {
    const int kv = it.n_chunks - 1;
    const int slot = kv % a.nslot;
    ok = ok && mbar_wait(&full[slot], (kv / a.nslot) & 1, a.err);
    const uint32_t vv = slot0 + (uint32_t)(slot * a.slot_bytes);
    // w as B fragments: b0 = w[16kk + 2t, +1][gq], b1 = w[16kk + 8 + 2t, +1][gq]
    float wf[RT][4];
    float wmax = 0.f;
#pragma unroll
    for (int kk = 0; kk < RT; ++kk) {
      wf[kk][0] = wf[kk][1] = wf[kk][2] = wf[kk][3] = 0.f;
      if (kk < nrt) {
        int r0 = 16 * kk + 2 * t;
        wf[kk][0] = wbuf[r0 * 8 + gq];
        wf[kk][1] = wbuf[(r0 + 1) * 8 + gq];
        if (r0 + 8 < r8) { wf[kk][2] = wbuf[(r0 + 8) * 8 + gq]; wf[kk][3] = wbuf[(r0 + 9) * 8 + gq]; }
      }
      wmax = fmaxf(wmax, fmaxf(fmaxf(fabsf(wf[kk][0]), fabsf(wf[kk][1])), fmaxf(fabsf(wf[kk][2]), fabsf(wf[kk][3]))));
    }
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, 1));
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, 2));
    const float wsc = pow2_down(wmax);
    uint32_t wh[RT][2], wl[RT][2];
#pragma unroll
    for (int kk = 0; kk < RT; ++kk) {
      split_half2(wf[kk][0] * wsc, wf[kk][1] * wsc, wh[kk][0], wl[kk][0]);
      split_half2(wf[kk][2] * wsc, wf[kk][3] * wsc, wh[kk][1], wl[kk][1]);
    }
    const float wus0 = 1.f / __shfl_sync(0xffffffffu, wsc, 8 * t);
    const float wus1 = 1.f / __shfl_sync(0xffffffffu, wsc, 8 * t + 4);
    float pa0 = 0.f, pa1 = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) { pa0 += pabuf[w * 8 + 2 * t]; pa1 += pabuf[w * 8 + 2 * t + 1]; }
    for (int md = warp; md < D / 16; md += kConsumers) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t mb = vv + (uint32_t)(md * 16 * r8 * 2);
#pragma unroll
      for (int kk = 0; kk < RT; ++kk) {
        if (kk < nkk) {
          uint4 v = lds128(mb + (uint32_t)(kk * 512 + lane * 16));
          mma16816(c, v.x, v.y, v.z, v.w, wh[kk][0], wh[kk][1]);
          mma16816(c, v.x, v.y, v.z, v.w, wl[kk][0], wl[kk][1]);
        } else if (kk == nkk && rtail) {
          uint2 v = lds64(mb + (uint32_t)(kk * 512 + lane * 8));
          mma1688(c, v.x, v.y, wh[kk][0]);
          mma1688(c, v.x, v.y, wl[kk][0]);
        }
      }
      const int d0 = md * 16 + gq, d1 = d0 + 8;
      const float av0 = __half2float(av[d0]), av1 = __half2float(av[d1]);
      float* o0 = obuf + d0 * 8 + 2 * t;
      float* o1 = obuf + d1 * 8 + 2 * t;
      o0[0] += c[0] * wus0 + pa0 * av0;
      o0[1] += c[1] * wus1 + pa1 * av0;
      o1[0] += c[2] * wus0 + pa0 * av1;
      o1[1] += c[3] * wus1 + pa1 * av1;
    }
    named_bar_sync(1, kConsumers * 32);
  }

  // ---------------- write the partial: m[8], l[8], o[8][D] (base-2 units)
  float* rec = a.partials + ((size_t)u * a.n_items + item) * (16 + 8 * D);
  const int tid = threadIdx.x;
  if (tid < 8) {
    float m = -INFINITY, l = 0.f;
    for (int w = 0; w < kConsumers; ++w) m = fmaxf(m, mbuf[w * 8 + tid]);
    for (int w = 0; w < kConsumers; ++w) l += lbuf[w * 8 + tid];
    if (!ok) { m = -INFINITY; l = 0.f; }
    rec[tid] = m;
    rec[8 + tid] = l;
  }
  for (int e = tid; e < G * D; e += kConsumers * 32) {
    int g = e / D, j = e % D;
    rec[16 + g * D + j] = ok ? obuf[j * 8 + g] : 0.f;
  }
  if (a.out == nullptr) return;

  // ---------------- fused split-LSE merge: the unit's last CTA to finish merges
  // all of the unit's partials (arrival counter, no waiting on other CTAs)
  __threadfence();
  named_bar_sync(1, kConsumers * 32);
  if (tid == 0) maskbuf[0] = atomicAdd(&a.counters[u], 1u) == (unsigned)(a.n_items - 1);
  named_bar_sync(1, kConsumers * 32);
  if (!maskbuf[0]) return;
  __threadfence();
  const size_t rs = 16 + 8 * (size_t)D;
  const float* base = a.partials + (size_t)u * a.n_items * rs;
  float* mstar = mbuf;          // [8] max of the unit's partials, per query of the group
  float* linv = mbuf + 8;       // [8] 1 / merged normaliser
  const size_t qrow0 = (size_t)bseq * a.Hq + (size_t)h * G;
  if (tid < G) {
    float m = -INFINITY;
    for (int i = 0; i < a.n_items; ++i) m = fmaxf(m, __ldcg(base + i * rs + tid));
    const float ms = m == -INFINITY ? 0.f : m;
    float l = 0.f;
    for (int i = 0; i < a.n_items; ++i) l += __ldcg(base + i * rs + 8 + tid) * exp2f(__ldcg(base + i * rs + tid) - ms);
    mstar[tid] = ms;
    linv[tid] = 1.f / l;
    if (a.lse) a.lse[qrow0 + tid] = (ms + log2f(l)) * 0.6931471805599453f;
  }
  named_bar_sync(1, kConsumers * 32);
  for (int e = tid; e < G * D; e += kConsumers * 32) {
    const int g = e / D, j = e % D;
    const float ms = mstar[g];
    float acc = 0.f;
    for (int i = 0; i < a.n_items; ++i)
      acc = fmaf(exp2f(__ldcg(base + i * rs + g) - ms), __ldcg(base + i * rs + 16 + g * D + j), acc);
    a.out[(qrow0 + g) * D + j] = acc * linv[g];
  }
  if (tid == 0) a.counters[u] = 0u;  // ready for the next call on this workspace
}

template <int D, int RT>
cudaError_t launch_one(const AttendArgs& a, size_t smem, cudaStream_t s) {
  static size_t configured = 0;  // largest dynamic shared memory size enabled so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  dim3 grid(a.n_items, a.L.units);
  attend_kernel<D, RT><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

DecodePlan plan_decode(const Layout& L, int n_q_heads, int n_kv_heads, int top_k) {
  (void)n_q_heads;
  (void)n_kv_heads;
  DecodePlan P;
  P.K_eff = (top_k == 0 || top_k >= L.NB) ? L.NB : top_k;
  P.wchunk_tokens = kWindowChunk;
  P.n_wchunks = (L.W16 + kWindowChunk - 1) / kWindowChunk;
  P.n_items = P.K_eff + P.n_wchunks;
  P.route_splits = L.NB > 0 ? (L.NB + 63) / 64 : 0;
  P.off_counters = kWsHeader;
  P.off_bounds = round_up(P.off_counters + (size_t)L.units * 8, 256);
  P.off_routed = round_up(P.off_bounds + (size_t)L.units * L.NB * 4, 256);
  P.off_partials = round_up(P.off_routed + (size_t)L.units * P.K_eff * 4, 256);
  P.ws_bytes = P.off_partials + (size_t)L.units * P.n_items * (16 + 8 * L.d) * 4;
  return P;
}

cudaError_t launch_attend(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                          const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s) {
  AttendArgs a;
  a.L = L;
  a.G = n_q_heads / n_kv_heads;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.K_eff = P.K_eff;
  a.n_items = P.n_items;
  a.xtok = 16384 / (4 * L.d);
  const int head = (int)L.off_u;
  int slot = 16384;
  slot = head > slot ? head : slot;
  slot = kUTok * 2 * L.r8 > slot ? kUTok * 2 * L.r8 : slot;
  slot = 2 * L.r8 * L.d > slot ? 2 * L.r8 * L.d : slot;
  slot = (int)round_up((uint64_t)slot, 128);
  const int RT = L.r8 <= 32 ? 2 : (L.r8 <= 64 ? 4 : 8);
  const size_t extra = 2 * kMaxSlots * 8 + (size_t)(RT * 2) * 32 * 8 + (size_t)RT * 16 * 8 * 4 + (size_t)L.d * 8 * 4 +
                       3 * 32 * 4 + 32 + (size_t)L.d * 2 + 128;
  const size_t budget = 113 * 1024;
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
  a.counters = reinterpret_cast<uint32_t*>(ws + P.off_counters) + L.units;
  a.out = out;
  a.lse = lse;
  const size_t smem = (size_t)nslot * slot + extra;
  if (P.n_items == 0) return cudaSuccess;
  if (L.d == 128) {
    if (RT == 2) return launch_one<128, 2>(a, smem, s);
    if (RT == 4) return launch_one<128, 4>(a, smem, s);
    return launch_one<128, 8>(a, smem, s);
  }
  if (RT == 2) return launch_one<64, 2>(a, smem, s);
  if (RT == 4) return launch_one<64, 4>(a, smem, s);
  return launch_one<64, 8>(a, smem, s);
}

}  // namespace dkv
