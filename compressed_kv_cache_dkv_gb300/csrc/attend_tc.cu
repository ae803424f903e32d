// Block + window attention of the DKV decode path on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory), for the tensor-core cache
// layout (head_dim 128, 8 <= r8 <= 48, 1 <= R <= 128).
//
// Per routed block ("Low-Rank Space Query Scoring" / "Flash-Style LSE Combine",
// Differential-KV README, section "Core Architecture & Paper Overview"; DKV
// Zenodo abstract), with M = 128 rows and N = 16 columns per product:
//   S_X    = K_res [q | 0]              tcgen05, A = K_res (K-major)
//   z      = V_K (c q)                  mma.sync (r x 8, small)
//   S_L    = U [z_hi | z_lo]            tcgen05, A = U (K-major), two 128-token tiles
//   p      = 2^(s - max) over the 255 low-rank tokens and the anchor (s = c q.a_k + U z)
//   W      = U^T [p_hi | p_lo]          tcgen05, A = U viewed MN-major (no transpose)
//   O_X    = V_res^T [p_hi | p_lo]      tcgen05, A = V_res viewed MN-major
//   O_L    = V_V^T [w_hi | w_lo]        tcgen05, A = V_V viewed MN-major
// and the partial (m, l, o) with o = 2^(m_L - m) (O_L + L_L a_v) + 2^(m_X - m) O_X.
// The fp32 operands of a product (z, p, w) enter as an fp16 pair hi + lo in the
// two 8-column halves of N, so one MMA carries about 22 bits.  A window item
// (128 tokens) is the exact half alone.
//
// Two CTAs share an SM.  Each has four consumer warps (warp w owns tensor-memory
// lanes 32w..32w+31, i.e. one token / r / d row per thread) and one producer
// warp that streams each item's chunks into a ring of 16 KB shared-memory units
// with 1-D TMA bulk copies.  A chunk takes one unit (anchors + V_K, one U tile,
// V_V) or two adjacent units (the exact rows' K or V, when more than 64 rows);
// a two-unit chunk never wraps around the ring.  Thread 0 issues the
// tcgen05.mma groups; tcgen05.commit completes both the group's own mbarrier
// and the "empty" mbarriers of the units the group was the last to read, so a
// unit returns to the producer as soon as its tensor-core reads are done.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kTcConsumers = 4;
constexpr int kTcThreads = (kTcConsumers + 1) * 32;
constexpr int kTcCtasPerSm = 2;
constexpr uint32_t kUnit = 16 * 1024;
constexpr int kUnits = 5;
constexpr int kTcIQ = 2;
constexpr int kTcWin = 128;          // window tokens per item
constexpr uint32_t kTmemCols = 128;  // S_L (2 x 16), S_X, W, O_X, O_L (16 each)
constexpr uint32_t kColSL = 0, kColSX = 32, kColW = 48, kColOX = 64, kColOL = 80;

struct TcArgs {
  Layout L;
  int G, Hq, Hkv, K_eff, n_items, n_wgroups, n_wfront, total;
  float scale_log2;  // log2(e) / sqrt(d)
  const __half* q;
  const uint8_t* cache;
  const int32_t* routed;
  float* partials;
  uint32_t* err;
  uint32_t* sched;  // [0] next dynamic item, [1] CTAs done fetching
};

struct TcItem {
  int stop, is_block, ok, u, item, n, nvalid;
  uint64_t base;  // block record or window group (bytes from the cache base)
};

// Shared memory: the ring, then the operand buffers.  A one-unit exact chunk
// is read as 128 rows by S_X (rows past its end are masked), so at least one
// unit's worth of allocated memory follows the ring.
constexpr uint32_t kOffBq = kUnits * kUnit;              // [16 x 128] K-major, 4 KB
constexpr uint32_t kOffBPL = kOffBq + 4096;              // [256 x 16] MN-major, 8 KB
constexpr uint32_t kOffBPX = kOffBPL + 8192;             // [128 x 16] MN-major, 4 KB
constexpr uint32_t kOffBz = kOffBPX + 4096;              // [16 x r16] K-major, <= 1.5 KB
constexpr uint32_t kOffBW = kOffBz + 2048;               // [r16 x 16] MN-major, <= 1.5 KB
constexpr uint32_t kOffQ = kOffBW + 2048;                // [kTcIQ][8][136] fp16 query rows
constexpr uint32_t kOffZ = kOffQ + kTcIQ * 8 * 136 * 2;  // [r8][8] fp32 z
constexpr uint32_t kOffMisc = kOffZ + 48 * 8 * 4;        // barriers and small arrays
constexpr uint32_t kTcSmem = kOffMisc + 2048;
static_assert(kTcSmem - kOffBq >= kUnit, "guard after the ring");
static_assert(kTcCtasPerSm * (kTcSmem + 1024) <= 228 * 1024, "two CTAs per SM");

struct TcSmem {
  uint8_t* base;
  uint64_t *full, *empty, *iq_full, *iq_empty, *mma;  // mma[4]: S_L, S_X, W, O
  TcItem* iqd;
  float* basebuf;  // [4][8] partial q . a_k
  float* red;      // [2][4][8] per-warp maxima / sums (low-rank half, exact half)
  float* st;       // [8] base, [8] (unused), [8] L_L
  __half* av;      // [128]
  uint32_t* mask;  // [8]
  uint32_t* tmem;  // allocated tensor-memory address
  int* flag;       // [1] a wait gave up
};

__device__ inline TcSmem tc_carve(uint8_t* smem) {
  TcSmem s;
  s.base = smem;
  uint8_t* p = smem + kOffMisc;
  s.full = reinterpret_cast<uint64_t*>(p);
  s.empty = s.full + kUnits;
  s.iq_full = s.empty + kUnits;
  s.iq_empty = s.iq_full + kTcIQ;
  s.mma = s.iq_empty + kTcIQ;
  s.iqd = reinterpret_cast<TcItem*>(s.mma + 4);
  s.basebuf = reinterpret_cast<float*>(s.iqd + kTcIQ);
  s.red = s.basebuf + 32;
  s.st = s.red + 64;
  s.av = reinterpret_cast<__half*>(s.st + 48);
  s.mask = reinterpret_cast<uint32_t*>(s.av + 128);
  s.tmem = s.mask + 8;
  s.flag = reinterpret_cast<int*>(s.tmem + 1);
  return s;
}

// ---------------------------------------------------------------- ring of units
// First unit of an s-unit chunk; a chunk that would run past the last unit
// starts again at unit 0 (the skipped units are left alone this time round).
// Producer and consumers call it in the same order and so agree on every
// chunk's place.
__device__ inline int ring_take(int& pos, int s) {
  if (pos + s > kUnits) pos = 0;
  const int u = pos;
  pos += s;
  if (pos == kUnits) pos = 0;
  return u;
}
// units of an exact chunk (K or V) of n rows
__device__ inline int exact_units(int n) { return n * 256 > (int)kUnit ? 2 : 1; }

// ---------------------------------------------------------------- tcgen05 helpers
// Shared-memory matrix descriptor, no swizzle: start address, LBO = byte stride
// between core matrices along K, SBO = along M (or N); version field 1.
__device__ inline uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}
// Instruction descriptor: D f32, A and B f16, M = 128, N = 16; a_mn / b_mn = MN-major operand
__host__ __device__ constexpr uint32_t idesc(bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ inline void umma(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dt),
      "l"(ad), "l"(bd), "r"(id), "r"(acc)
      : "memory");
}
// arrive on `bar` once every tcgen05.mma issued so far by this thread has completed
__device__ inline void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ inline void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ inline void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 16 fp32 columns of this warp's 32 lanes
__device__ inline void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ inline void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
// 8 fp32 values -> (hi, lo) fp16 rows of 16 bytes each
__device__ inline void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_half2(x[2 * i], x[2 * i + 1], h[i], l[i]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// zero `bytes` (a multiple of 16 * 128) at shared address addr with the 128 consumer threads
__device__ inline void zero_smem(uint32_t addr, uint32_t bytes, int tid) {
  for (uint32_t o = (uint32_t)tid * 16u; o < bytes; o += kTcConsumers * 32 * 16u) sts128(addr + o, make_uint4(0u, 0u, 0u, 0u));
}

// per-column max / sum over the 128 consumer threads: warp butterfly, then the
// four warps through shared memory (caller provides the barrier between the
// store and the final read)
__device__ inline void warp_allmax8(float (&v)[8]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int g = 0; g < 8; ++g) v[g] = fmaxf(v[g], __shfl_xor_sync(0xffffffffu, v[g], o));
}
__device__ inline void warp_allsum8(float (&v)[8]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int g = 0; g < 8; ++g) v[g] += __shfl_xor_sync(0xffffffffu, v[g], o);
}
__device__ inline float pick8(const float (&v)[8], int i) {  // v[i] without dynamic indexing
  float x = v[0];
#pragma unroll
  for (int g = 1; g < 8; ++g) x = i == g ? v[g] : x;
  return x;
}

// Power of two 2^e with 2 L <= 2^e < 4 L for L >= 1 (its reciprocal scales w so
// that |w| <= max|U| < 65504 stays finite in fp16): from L's exponent field.
__device__ inline float w_unscale(float L) {
  const int E = (__float_as_int(fmaxf(L, 1.f)) >> 23) & 0xff;  // L in [2^(E-127), 2^(E-126))
  return __int_as_float((E + 2) << 23);                        // 2^(E-125)
}
__device__ inline float w_scale(float L) {
  const int E = (__float_as_int(fmaxf(L, 1.f)) >> 23) & 0xff;
  return __int_as_float((252 - E) << 23);  // 2^(125-E)
}

// Bounded wait on an MMA-group barrier; returns false on timeout.
__device__ inline bool mma_wait(uint64_t* bar, uint32_t& uses, uint32_t* err) {
  const bool ok = mbar_wait(bar, uses & 1u, err);
  ++uses;
  tc_fence_after();
  return ok;
}

// ---------------------------------------------------------------- item decode
__device__ inline TcItem tc_decode(const TcArgs& a, int gi) {
  const Layout& L = a.L;
  TcItem it;
  it.stop = 0;
  it.ok = 1;
  // n_wfront window groups of every unit, the routed blocks, the other window groups
  const int nfront = a.n_wfront * L.units, nblk = a.K_eff * L.units;
  if (gi < nfront || gi >= nfront + nblk) {
    const int wg = gi < nfront ? gi / L.units : a.n_wfront + (gi - nfront - nblk) / L.units;
    it.u = gi % L.units;
    it.item = a.K_eff + wg;
    it.is_block = 0;
    it.n = min(kTcWin, L.W16 - wg * kTcWin);
    it.nvalid = min(it.n, L.W - wg * kTcWin);
    it.base = (uint64_t)it.u * L.unit_stride + L.off_window + (uint64_t)wg * kTcWin * 4 * L.d;
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
    it.n = L.R8;
    it.nvalid = L.R;
    it.base = (uint64_t)it.u * L.unit_stride + L.off_blocks + (uint64_t)blk * L.block_stride;
  }
  return it;
}

// Ring places of one item's chunks, in streaming order: K, head (anchors, mask,
// V_K), U tile 0, U tile 1, V, V_V for a block; K, V for a window group.
struct Places {
  int k, head, u0, u1, v, vv, sx;  // first units; sx = units of K and of V
};
__device__ inline Places take_places(int& pos, const TcItem& it) {
  Places p;
  p.sx = exact_units(it.n);
  p.k = ring_take(pos, p.sx);
  p.head = p.u0 = p.u1 = p.vv = -1;
  if (it.is_block) {
    p.head = ring_take(pos, 1);
    p.u0 = ring_take(pos, 1);
    p.u1 = ring_take(pos, 1);
  }
  p.v = ring_take(pos, p.sx);
  if (it.is_block) p.vv = ring_take(pos, 1);
  return p;
}

// ---------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kTcThreads, kTcCtasPerSm) attend_tc_kernel(TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const TcSmem sm = tc_carve(smem);
  const Layout& L = a.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  constexpr int D = 128;

  if (tid == 0) {
    for (int i = 0; i < kUnits; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 1); }
    for (int i = 0; i < kTcIQ; ++i) { mbar_init(&sm.iq_full[i], 1); mbar_init(&sm.iq_empty[i], 1); }
    for (int i = 0; i < 4; ++i) mbar_init(&sm.mma[i], 1);
    sm.flag[0] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sm.tmem)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem;

  griddep_launch();  // the combine grid may be scheduled now; it waits for this grid's completion

  // =========================== producer warp
  if (warp == kTcConsumers) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int pos = 0;
      uint32_t eph = 0u, used = 0u;  // per unit: parity of its next release, filled at least once
      // per unit whose full barrier a fill armed (the first unit of the fill's span): the parity
      // of its next fill's phase and of its last one
      uint32_t armed = 0u, fpar = 0u, lastf = 0u;
      // per query slot: parity of its last phase (iteration j is phase j / kTcIQ of slot j % kTcIQ,
      // a copy or a plain arrival) and whether it had one; waiting on an older phase's parity
      // after a later one completed would sit out the whole bounded wait
      uint32_t qpar = 0u, qused = 0u;
      bool waited = false;
      const uint32_t r8 = (uint32_t)L.r8;
      // claim s units starting at u (waiting for their previous contents to be released) and fill them
      auto put = [&](int u, int s, const uint8_t* src, uint32_t bytes) -> bool {
        for (int v = u; v < u + s; ++v) {
          if ((used >> v) & 1u) {
            if (!mbar_wait(&sm.empty[v], (eph >> v) & 1u, a.err)) return false;
            eph ^= 1u << v;
          }
          used |= 1u << v;
        }
        mbar_arrive_expect_tx(&sm.full[u], bytes);
        bulk_g2s(smem + (size_t)u * kUnit, src, bytes, &sm.full[u], pol);
        lastf = (lastf & ~(1u << u)) | (fpar & (1u << u));
        fpar ^= 1u << u;
        armed |= 1u << u;
        return true;
      };
      for (int j = 0;; ++j) {
        int gi = blockIdx.x;
        if (j > 0) {
          if (!waited) { griddep_wait(); waited = true; }
          gi = (int)gridDim.x + (int)atomicAdd(&a.sched[0], 1u);
        }
        const int iq = j % kTcIQ;
        if (j >= kTcIQ && !mbar_wait(&sm.iq_empty[iq], ((j / kTcIQ) - 1) & 1, a.err)) break;
        qpar = (qpar & ~(1u << iq)) | ((uint32_t)((j / kTcIQ) & 1) << iq);  // every path below arrives once
        qused |= 1u << iq;
        TcItem& dsc = sm.iqd[iq];
        if (gi >= a.total) {
          dsc.stop = 1;
          mbar_arrive(&sm.iq_full[iq]);
          if (j > 0 && atomicAdd(&a.sched[1], 1u) == gridDim.x - 1) {  // the last CTA out resets the scheduler
            a.sched[0] = 0u;
            a.sched[1] = 0u;
          }
          break;
        }
        if (gi >= a.n_wfront * L.units && gi < (a.n_wfront + a.K_eff) * L.units && !waited) {
          griddep_wait();
          waited = true;
        }
        const TcItem it = tc_decode(a, gi);
        dsc = it;
        if (!it.ok) {
          mbar_arrive(&sm.iq_full[iq]);
          continue;
        }
        {
          const uint32_t row = (uint32_t)(D * 2);
          mbar_arrive_expect_tx(&sm.iq_full[iq], row * (uint32_t)a.G);
          const __half* qsrc = a.q + ((size_t)(it.u / a.Hkv) * a.Hq + (size_t)(it.u % a.Hkv) * a.G) * D;
          __half* qdst = reinterpret_cast<__half*>(smem + kOffQ) + (size_t)iq * 8 * 136;
          for (int g = 0; g < a.G; ++g) bulk_g2s(qdst + (size_t)g * 136, qsrc + (size_t)g * D, row, &sm.iq_full[iq], pol);
        }
        const Places p = take_places(pos, it);
        const uint8_t* src = a.cache + it.base;
        const uint32_t bx = (uint32_t)it.n * 2u * D;  // K (or V) bytes of the item
        const uint8_t* k0 = it.is_block ? src + L.off_res : src;
        bool ok = put(p.k, p.sx, k0, bx);
        if (ok && it.is_block) {
          ok = put(p.head, 1, src, (uint32_t)L.off_u) &&
               put(p.u0, 1, src + L.off_u, 256u * r8) &&
               put(p.u1, 1, src + L.off_u + 256u * r8, 256u * r8);
        }
        ok = ok && put(p.v, p.sx, k0 + bx, bx);
        if (ok && it.is_block) ok = put(p.vv, 1, src + L.off_vv, 256u * r8);
        if (!ok) break;
      }
      // every copy this CTA issued lands before it may finish, whether or not a wait gave
      // up: the last fill of every ring unit and the last phase of every query slot (fills of
      // a unit and phases of a slot complete in order: each waits for the release of the last)
      for (int v = 0; v < kUnits; ++v)
        if ((armed >> v) & 1u) mbar_wait(&sm.full[v], (lastf >> v) & 1u, a.err);
      for (int q = 0; q < kTcIQ; ++q)
        if ((qused >> q) & 1u) mbar_wait(&sm.iq_full[q], (qpar >> q) & 1u, a.err);
    }
    return;
  }

  // =========================== consumer warps
  int pos = 0;
  uint32_t fph = 0u;              // per unit: parity of its next fill
  uint32_t mu[4] = {0, 0, 0, 0};  // uses of the four MMA-group barriers
  const int G = a.G;
  const float slog2 = a.scale_log2;
  const int r8 = L.r8, r16 = (L.r8 + 15) & ~15;
  const int t = lane & 3, gq = lane >> 2;
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter
  float* st = sm.st;
  auto unit_addr = [&](int u) -> uint32_t { return sbase + (uint32_t)u * kUnit; };
  // wait for the fill of unit u taken with parity `par`
  auto wait_fill = [&](int u, uint32_t par) -> bool { return mbar_wait(&sm.full[u], par, a.err); };
  int j = 0;
  for (;; ++j) {
    const int iq = j % kTcIQ;
    const bool got = mbar_wait(&sm.iq_full[iq], (j / kTcIQ) & 1, a.err);
    if (!got && lane == 0) sm.flag[0] = 1;
    const TcItem it = sm.iqd[iq];
    named_bar_sync(1, kTcConsumers * 32);
    if (it.stop || *reinterpret_cast<volatile int*>(sm.flag)) break;
    float* rec = a.partials + ((size_t)it.u * a.n_items + it.item) * (16 + 8 * D);
    if (!it.ok) {
      if (tid == 0) mbar_arrive(&sm.iq_empty[iq]);
      for (int e = tid; e < 16 + 8 * D; e += kTcConsumers * 32) rec[e] = e < 8 ? -INFINITY : 0.f;
      continue;
    }
    bool ok = true;
    // ring places and fill parities of this item's chunks (a unit may serve two chunks of one item)
    const Places p = take_places(pos, it);
    uint32_t par_k, par_h = 0, par_u0 = 0, par_u1 = 0, par_v, par_vv = 0;
    par_k = (fph >> p.k) & 1u; fph ^= 1u << p.k;
    if (it.is_block) {
      par_h = (fph >> p.head) & 1u; fph ^= 1u << p.head;
      par_u0 = (fph >> p.u0) & 1u; fph ^= 1u << p.u0;
      par_u1 = (fph >> p.u1) & 1u; fph ^= 1u << p.u1;
    }
    par_v = (fph >> p.v) & 1u; fph ^= 1u << p.v;
    if (it.is_block) { par_vv = (fph >> p.vv) & 1u; fph ^= 1u << p.vv; }

    const __half* qrows = reinterpret_cast<const __half*>(smem + kOffQ) + (size_t)iq * 8 * 136;
    // ---- B_q [16 x 128] K-major: rows 0..G-1 the queries, the rest zero
    for (int e = tid; e < 256; e += kTcConsumers * 32) {
      const int n = e >> 4, kg = e & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < G) v = *reinterpret_cast<const uint4*>(qrows + n * 136 + kg * 8);
      sts128(sbase + kOffBq + (uint32_t)(n >> 3) * 2048u + (uint32_t)kg * 128u + (uint32_t)(n & 7) * 16u, v);
    }
    fence_async_smem();
    tc_fence_before();
    named_bar_sync(1, kTcConsumers * 32);  // B_q is visible to the tensor cores
    tc_fence_after();
    const int n16 = (it.n + 15) & ~15;
    if (tid == 0) {
      // S_X = K [q | 0]: K = head dim (8 k steps); then K's units go back to the producer
      ok = wait_fill(p.k, par_k) && ok;
      tc_fence_after();
      const uint64_t a0 = sdesc(unit_addr(p.k), 128u, 2048u), b0 = sdesc(sbase + kOffBq, 128u, 2048u);
      for (int ks = 0; ks < 8; ++ks)
        umma(tmem + kColSX, a0 + (uint64_t)(ks * 16), b0 + (uint64_t)(ks * 16), idesc(false, false), ks > 0 ? 1u : 0u);
      umma_commit(&sm.mma[1]);
      for (int v = p.k; v < p.k + p.sx; ++v) umma_commit(&sm.empty[v]);
      if (!it.is_block) mbar_arrive(&sm.iq_empty[iq]);  // the queries are in B_q
    }
    if (it.is_block) {
      // ======================= head chunk -> base, z; U tiles -> S_L
      ok = wait_fill(p.head, par_h) && ok;
      const uint8_t* head = smem + (size_t)p.head * kUnit;
      {
        // q fragments (B operand: k = head dim, n = group)
        uint32_t qb[8][2];
        const uint32_t qrow = smem_u32(qrows + gq * 136);
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          qb[kt][0] = gq < G ? lds32(qrow + (uint32_t)(16 * kt + 2 * t) * 2u) : 0u;
          qb[kt][1] = gq < G ? lds32(qrow + (uint32_t)(16 * kt + 8 + 2 * t) * 2u) : 0u;
        }
        // q . a_k: each warp two 16-wide k tiles
        const __half* ak = reinterpret_cast<const __half*>(head);
        float part = 0.f;
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          if (kt / 2 == warp) {
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
        if (tid < D) sm.av[tid] = reinterpret_cast<const __half*>(head)[D + tid];
        if (tid < 8) sm.mask[tid] = reinterpret_cast<const uint32_t*>(head + L.off_mask)[tid];
        // z^T = q^T V_K^T (V_K in the mma.sync B^T layout): n-tiles of 8 r-rows over the warps
        const uint32_t vk = smem_u32(head) + (uint32_t)L.off_vk;
        float* zb = reinterpret_cast<float*>(smem + kOffZ);
        for (int nt = warp; nt < (r8 >> 3); nt += kTcConsumers) {
          float c[4] = {0.f, 0.f, 0.f, 0.f};
          uint4 bv[4];
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) bv[kp] = lds128(vk + (uint32_t)(nt * 8 * D * 2 + kp * 512 + lane * 16));
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            mma16816(c, qb[2 * kp][0], 0u, qb[2 * kp][1], 0u, bv[kp].x, bv[kp].y);
            mma16816(c, qb[2 * kp + 1][0], 0u, qb[2 * kp + 1][1], 0u, bv[kp].z, bv[kp].w);
          }
          // C fragment: row gq = query, columns 2t, 2t+1 = r rows nt*8 + 2t, +1
          zb[(nt * 8 + 2 * t) * 8 + gq] = c[0] * slog2;
          zb[(nt * 8 + 2 * t + 1) * 8 + gq] = c[1] * slog2;
        }
      }
      named_bar_sync(1, kTcConsumers * 32);  // base, z, a_v, mask written; the head unit and the query rows are read
      if (tid == 0) {
        mbar_arrive(&sm.empty[p.head]);
        mbar_arrive(&sm.iq_empty[iq]);
      }
      // base score per query (base-2 units) and B_z [16 x r16] K-major: rows 0-7 z_hi, 8-15 z_lo
      if (tid < 8) st[tid] = (sm.basebuf[tid] + sm.basebuf[8 + tid] + sm.basebuf[16 + tid] + sm.basebuf[24 + tid]) * slog2;
      {
        const float* zb = reinterpret_cast<const float*>(smem + kOffZ);
        const int nkg = r16 >> 3;
        for (int e = tid; e < 8 * nkg; e += kTcConsumers * 32) {
          const int g = e / nkg, kg = e % nkg;
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int k = kg * 8 + i;
            x[i] = (k < r8 && g < G) ? zb[k * 8 + g] : 0.f;
          }
          uint4 hi, lo;
          split8(x, hi, lo);
          const uint32_t row_hi = sbase + kOffBz + (uint32_t)kg * 128u + (uint32_t)g * 16u;  // N group 0 (rows 0-7)
          sts128(row_hi, hi);
          sts128(row_hi + (uint32_t)nkg * 128u, lo);                                        // N group 1 (rows 8-15)
        }
      }
      // U tiles: with r8 % 16 == 8 the last 16-wide k step of the last token group reads one
      // core matrix past the tile; it multiplies zero rows of B_z but must hold finite values
      ok = wait_fill(p.u0, par_u0) && ok;
      ok = wait_fill(p.u1, par_u1) && ok;
      if (r16 > r8 && tid < 16) {
        const uint32_t tail = 256u * (uint32_t)r8 + (uint32_t)(tid & 7) * 16u;
        sts128(unit_addr(tid < 8 ? p.u0 : p.u1) + tail, make_uint4(0u, 0u, 0u, 0u));
      }
      fence_async_smem();
      tc_fence_before();
      named_bar_sync(1, kTcConsumers * 32);
      tc_fence_after();
      if (tid == 0) {
        // S_L = U [z_hi | z_lo] per 128-token tile: K = r16; A K-major (LBO = core matrices along r,
        // SBO = 8-token groups, r8 * 16 B apart)
        const uint32_t nkg = (uint32_t)(r16 >> 3);
        const uint64_t b0 = sdesc(sbase + kOffBz, 128u, nkg * 128u);
        for (int tile = 0; tile < 2; ++tile) {
          const uint64_t a0 = sdesc(unit_addr(tile == 0 ? p.u0 : p.u1), 128u, 16u * (uint32_t)r8);
          for (int ks = 0; ks < (r16 >> 4); ++ks)
            umma(tmem + kColSL + (uint32_t)tile * 16u, a0 + (uint64_t)(ks * 16), b0 + (uint64_t)(ks * 16),
                 idesc(false, false), ks > 0 ? 1u : 0u);
        }
        umma_commit(&sm.mma[0]);
      }
    }

    float ML[8], LL[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) { ML[g] = -INFINITY; LL[g] = 0.f; }
    if (it.is_block) {
      // ======================= low-rank softmax over the 256 rows (anchor + 255 tokens)
      ok = mma_wait(&sm.mma[0], mu[0], a.err) && ok;
      float s0[16], s1[16];
      tmem_ld16(tl + kColSL, s0);
      tmem_ld16(tl + kColSL + 16, s1);
      const int tk0 = warp * 32 + lane, tk1 = 128 + tk0;
      const bool m0 = (sm.mask[tk0 >> 5] >> (tk0 & 31)) & 1u, m1 = (sm.mask[tk1 >> 5] >> (tk1 & 31)) & 1u;
      float x0[8], x1[8], mx[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float b = st[g];
        x0[g] = (m0 || g >= G) ? -INFINITY : b + s0[g] + s0[8 + g];
        x1[g] = (m1 || g >= G) ? -INFINITY : b + s1[g] + s1[8 + g];
        mx[g] = fmaxf(x0[g], x1[g]);
      }
      warp_allmax8(mx);
      if (lane < 8) sm.red[warp * 8 + lane] = pick8(mx, lane);
      named_bar_sync(1, kTcConsumers * 32);
      float ps[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        ML[g] = fmaxf(fmaxf(sm.red[g], sm.red[8 + g]), fmaxf(sm.red[16 + g], sm.red[24 + g]));
        const float ms = ML[g] == -INFINITY ? 0.f : ML[g];
        x0[g] = fast_exp2(x0[g] - ms);
        x1[g] = fast_exp2(x1[g] - ms);
        ps[g] = x0[g] + x1[g];
      }
      uint4 hi, lo;
      split8(x0, hi, lo);
      sts128(sbase + kOffBPL + (uint32_t)(tk0 >> 3) * 256u + (uint32_t)(tk0 & 7) * 16u, hi);
      sts128(sbase + kOffBPL + (uint32_t)(tk0 >> 3) * 256u + 128u + (uint32_t)(tk0 & 7) * 16u, lo);
      split8(x1, hi, lo);
      sts128(sbase + kOffBPL + (uint32_t)(tk1 >> 3) * 256u + (uint32_t)(tk1 & 7) * 16u, hi);
      sts128(sbase + kOffBPL + (uint32_t)(tk1 >> 3) * 256u + 128u + (uint32_t)(tk1 & 7) * 16u, lo);
      warp_allsum8(ps);
      fence_async_smem();
      tc_fence_before();
      named_bar_sync(1, kTcConsumers * 32);  // the maxima are read; B_P is written
      tc_fence_after();
      if (lane < 8) sm.red[warp * 8 + lane] = pick8(ps, lane);
      if (tid == 0) {
        // W = U^T [p_hi | p_lo]: A = U viewed MN-major (M = r, K = tokens; LBO = 8-token groups,
        // SBO = core matrices along r); 8 k steps of 16 tokens per tile.  Then the U units are free.
        const uint64_t b0 = sdesc(sbase + kOffBPL, 256u, 128u);
        for (int ks = 0; ks < 16; ++ks) {
          const uint32_t ua = unit_addr(ks < 8 ? p.u0 : p.u1) + (uint32_t)(ks & 7) * 32u * (uint32_t)r8;
          umma(tmem + kColW, sdesc(ua, 16u * (uint32_t)r8, 128u), b0 + (uint64_t)(ks * 32), idesc(true, true),
               ks > 0 ? 1u : 0u);
        }
        umma_commit(&sm.mma[2]);
        umma_commit(&sm.empty[p.u0]);
        umma_commit(&sm.empty[p.u1]);
      }
    }

    // ======================= exact softmax over the chunk's rows
    ok = mma_wait(&sm.mma[1], mu[1], a.err) && ok;
    float MX[8], LX[8];
    {
      float sx[16];
      tmem_ld16(tl + kColSX, sx);
      const int row = warp * 32 + lane;
      const bool valid = row < it.nvalid;
      float x[8], mx[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        x[g] = (valid && g < G) ? sx[g] * slog2 : -INFINITY;
        mx[g] = x[g];
      }
      warp_allmax8(mx);
      named_bar_sync(1, kTcConsumers * 32);  // the previous contents of red are read
      if (lane < 8) sm.red[32 + warp * 8 + lane] = pick8(mx, lane);  // second half of the scratch
      if (it.is_block) {
        // low-rank normaliser, from the per-warp sums stored before the barrier
        if (tid < 8) st[16 + tid] = sm.red[tid] + sm.red[8 + tid] + sm.red[16 + tid] + sm.red[24 + tid];
      }
      named_bar_sync(1, kTcConsumers * 32);
      const float* rx = sm.red + 32;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        MX[g] = fmaxf(fmaxf(rx[g], rx[8 + g]), fmaxf(rx[16 + g], rx[24 + g]));
        const float ms = MX[g] == -INFINITY ? 0.f : MX[g];
        x[g] = fast_exp2(x[g] - ms);
        mx[g] = x[g];
      }
      uint4 hi, lo;
      split8(x, hi, lo);
      sts128(sbase + kOffBPX + (uint32_t)(row >> 3) * 256u + (uint32_t)(row & 7) * 16u, hi);
      sts128(sbase + kOffBPX + (uint32_t)(row >> 3) * 256u + 128u + (uint32_t)(row & 7) * 16u, lo);
      warp_allsum8(mx);
      if (it.is_block) {
#pragma unroll
        for (int g = 0; g < 8; ++g) LL[g] = st[16 + g];
      }
      if (lane < 8) sm.basebuf[warp * 8 + lane] = pick8(mx, lane);  // per-warp exact sums
    }
    // V: zero the rows n .. n16-1 read by the 16-token k steps (one 8-row plane)
    ok = wait_fill(p.v, par_v) && ok;
    if (n16 > it.n) zero_smem(unit_addr(p.v) + (uint32_t)(it.n >> 3) * 2048u, 2048u, tid);
    if (it.is_block) {
      // ---- W (lane = r) -> B_W [r16 x 16] MN-major, scaled per query by 1 / w_unscale(L_L)
      ok = mma_wait(&sm.mma[2], mu[2], a.err) && ok;
      float wv[16];
      tmem_ld16(tl + kColW, wv);
      const int r = warp * 32 + lane;
      if (r < r16) {
        float x[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) x[g] = r < r8 ? (wv[g] + wv[8 + g]) * w_scale(LL[g]) : 0.f;
        uint4 hi, lo;
        split8(x, hi, lo);
        sts128(sbase + kOffBW + (uint32_t)(r >> 3) * 256u + (uint32_t)(r & 7) * 16u, hi);
        sts128(sbase + kOffBW + (uint32_t)(r >> 3) * 256u + 128u + (uint32_t)(r & 7) * 16u, lo);
      }
      // V_V: zero the r rows r8 .. r16-1 read by the last 16-wide k step (one 8-row plane)
      ok = wait_fill(p.vv, par_vv) && ok;
      if (r16 > r8) zero_smem(unit_addr(p.vv) + (uint32_t)(r8 >> 3) * 2048u, 2048u, tid);
    }
    fence_async_smem();
    tc_fence_before();
    named_bar_sync(1, kTcConsumers * 32);  // B_PX, B_W, the padding planes and the exact sums are written
    tc_fence_after();
#pragma unroll
    for (int g = 0; g < 8; ++g)
      LX[g] = sm.basebuf[g] + sm.basebuf[8 + g] + sm.basebuf[16 + g] + sm.basebuf[24 + g];
    if (tid == 0) {
      // O_X = V^T [p_hi | p_lo]: A = V viewed MN-major (M = d, K = n16 tokens)
      {
        const uint64_t a0 = sdesc(unit_addr(p.v), 2048u, 128u), b0 = sdesc(sbase + kOffBPX, 256u, 128u);
        for (int ks = 0; ks < (n16 >> 4); ++ks)
          umma(tmem + kColOX, a0 + (uint64_t)(ks * 256), b0 + (uint64_t)(ks * 32), idesc(true, true), ks > 0 ? 1u : 0u);
      }
      if (it.is_block) {
        // O_L = V_V^T [w_hi | w_lo]: A = V_V viewed MN-major (M = d, K = r16)
        const uint64_t a0 = sdesc(unit_addr(p.vv), 2048u, 128u), b0 = sdesc(sbase + kOffBW, 256u, 128u);
        for (int ks = 0; ks < (r16 >> 4); ++ks)
          umma(tmem + kColOL, a0 + (uint64_t)(ks * 256), b0 + (uint64_t)(ks * 32), idesc(true, true), ks > 0 ? 1u : 0u);
      }
      umma_commit(&sm.mma[3]);
      for (int v = p.v; v < p.v + p.sx; ++v) umma_commit(&sm.empty[v]);
      if (it.is_block) umma_commit(&sm.empty[p.vv]);
    }

    // ======================= epilogue: thread = head-dim row d
    ok = mma_wait(&sm.mma[3], mu[3], a.err) && ok;
    {
      float ox[16], ol[16];
      tmem_ld16(tl + kColOX, ox);
      if (it.is_block) tmem_ld16(tl + kColOL, ol);
      const int dd = warp * 32 + lane;
      const float av = it.is_block ? __half2float(sm.av[dd]) : 0.f;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float M = fmaxf(ML[g], MX[g]);
        const float ms = M == -INFINITY ? 0.f : M;
        const float aL = fast_exp2(ML[g] - ms), aX = fast_exp2(MX[g] - ms);
        float oL = 0.f;
        if (it.is_block) oL = (ol[g] + ol[8 + g]) * w_unscale(LL[g]) + LL[g] * av;
        const float o = aL * oL + aX * (ox[g] + ox[8 + g]);
        if (g < G) rec[16 + g * D + dd] = ok ? o : 0.f;
        if (dd == g) {
          rec[g] = ok ? M : -INFINITY;
          rec[8 + g] = ok ? aL * LL[g] + aX * LX[g] : 0.f;
        }
      }
    }
    if (!ok && lane == 0) sm.flag[0] = 1;
    // the tensor memory and the operand buffers are reused by the next item
    tc_fence_before();
    named_bar_sync(1, kTcConsumers * 32);
    tc_fence_after();
  }
  // all MMAs issued by thread 0 were waited for: free the tensor memory
  named_bar_sync(1, kTcConsumers * 32);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

}  // namespace

bool tc_eligible(const Layout& L, int n_q_heads, int n_kv_heads) {
  return L.tc != 0 && n_q_heads / n_kv_heads <= 8 && L.d == 128;
}

int tc_window_tokens() { return kTcWin; }

cudaError_t launch_attend_tc(const Layout& L, const DecodePlan& P, int n_q_heads, int n_kv_heads, const __half* q,
                             const uint8_t* cache, uint8_t* ws, float* out, float* lse, cudaStream_t s) {
  TcArgs a;
  a.L = L;
  a.G = n_q_heads / n_kv_heads;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.K_eff = P.K_eff;
  a.n_items = P.n_items;
  a.n_wgroups = P.n_wchunks;
  a.n_wfront = (P.n_wchunks + 1) / 2;
  a.total = L.units * P.n_items;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)L.d);
  a.q = q;
  a.cache = cache;
  a.routed = reinterpret_cast<const int32_t*>(ws + P.off_routed);
  a.partials = reinterpret_cast<float*>(ws + P.off_partials);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.sched = reinterpret_cast<uint32_t*>(ws + P.off_sched);
  if (a.total == 0) return cudaSuccess;
  {
    const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(attend_tc_kernel), kTcSmem);
    if (e != cudaSuccess) return e;
  }
  int grid = kTcCtasPerSm * sm_count();
  grid = grid < a.total ? grid : a.total;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap with the router's grid
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attend_tc_kernel, a);
  if (e != cudaSuccess || out == nullptr) return e;
  return launch_combine(L, P, L.units / n_kv_heads, n_q_heads, n_kv_heads, a.partials, out, lse, s);
}

}  // namespace dkv
