// GPU block compression (dkv_compress_layout): setup path, not timed.
//
// Per 256-token block ("Core Architecture & Paper Overview" of the
// Differential-KV README, items 1-3; DKV Zenodo abstract):
//   anchor (a_k, a_v) = the first token, kept exact;
//   X_i = [K_i - a_k | V_i - a_v], i = 1..255 (n = 2d columns);
//   the top-r right singular vectors W_r of X (joint K|V basis, V_K and V_V
//   are its key and value halves) and U = X W_r (the singular values folded
//   into U);
//   e_i = ||(K_i - a_k) - U_i V_K||_2 and the R largest are kept exact
//   (ties to the lower row), the "vanilla L2" criterion of the README's
//   "Content-Aware / Rarity-Aware Residual Selection";
//   per-channel key min / max over the 256 exact keys for the router.
//
// Eigen-solve of the Gram G = X^T X (fp32, accumulated with the anchor
// subtracted exactly):
//   head_dim 64  (n = 128): cyclic Jacobi on the whole Gram (exact up to fp32);
//   head_dim 128 (n = 256): subspace iteration Q <- orth(G Q) with p = r + 16
//     columns (at most 64) and classical Gram-Schmidt applied twice, then a
//     Rayleigh-Ritz step: cyclic Jacobi on Q^T G Q.
// The start block is a fixed +-1 pattern from an integer hash, so the result
// is deterministic.  One CTA (17 warps) per block; the extra CTA per unit
// (blockIdx.x == n_blocks) copies the exact recency window.
#include <math.h>

#include "dkv_internal.cuh"

namespace dkv {

namespace {

constexpr int kCThreads = 544;   // 17 warps: 528 threads own the 8x8 Gram tiles when n = 256
constexpr int kChunk = 16;       // tokens staged in shared memory at a time
constexpr int kIters = 12;       // subspace iterations after the start block
constexpr int kMaxSweeps = 16;

struct CArgs {
  Layout L;
  const __half* K;
  const __half* V;
  uint8_t* cache;
  uint32_t* err;
  int T;             // source tokens per unit (K, V are [units][T][D])
  int blk0, nblk;    // CTA x = i < nblk compresses source tokens [256 i, 256 i + 256) into block blk0 + i
  int with_window;   // CTA x = nblk copies the source tokens from 256 nblk on as the exact window
  int n, p, full;
  uint32_t off_q, off_xc, off_misc;  // byte offsets of the shared-memory regions (R1 at 0)
};

__device__ inline uint32_t hash32(uint32_t x) {  // integer avalanche hash (xorshift-multiply)
  x ^= x >> 16; x *= 0x7feb352du;
  x ^= x >> 15; x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

__device__ inline float h2f(__half h) { return __half2float(h); }

// round to fp16, saturating (and flagging) values outside the fp16 range
__device__ inline __half to_h(float x, uint32_t* err) {
  if (!(fabsf(x) <= 65504.f)) {
    raise_error(err, DKV_DEVERR_RANGE);
    x = isnan(x) ? 0.f : copysignf(65504.f, x);
  }
  return __float2half_rn(x);
}

__device__ inline float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < nw; ++w) s += red[w];
  return s;
}

// Cyclic Jacobi on the symmetric m x m matrix A (leading dim ld) accumulating
// the rotations into Z (leading dim ld, Z = I on entry).  Disjoint pairs of a
// round-robin round are rotated together.  On exit A is (nearly) diagonal and
// A0 = Z diag(A) Z^T.
__device__ void jacobi(float* A, float* Z, int m, int ld, float* red, float2* cs, int2* pr) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int half = m / 2;
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    float off = 0.f, dia = 0.f;
    for (int e = tid; e < m * m; e += nt) {
      int i = e / m, j = e % m;
      float v = A[i * ld + j];
      if (i == j) dia += v * v; else off += v * v;
    }
    off = block_sum(off, red);
    dia = block_sum(dia, red + 32);
    // converged for fp32 (and far below the fp16 the factors are stored in): the
    // off-diagonal norm is at most 1e-5 of the diagonal's
    if (!(off > 1e-10f * dia) || dia == 0.f) break;
    for (int round = 0; round < m - 1; ++round) {
      for (int k = tid; k < half; k += nt) {
        int p, q;
        if (k == 0) { p = round; q = m - 1; }
        else { p = (round + k) % (m - 1); q = (round - k + (m - 1)) % (m - 1); }
        if (p > q) { int t = p; p = q; q = t; }
        float apq = A[p * ld + q], app = A[p * ld + p], aqq = A[q * ld + q];
        float c = 1.f, s = 0.f;
        if (fabsf(apq) > 1e-30f && fabsf(apq) > 1e-9f * sqrtf(fabsf(app * aqq))) {
          float tau = (aqq - app) / (2.f * apq);
          float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
          c = rsqrtf(1.f + t * t);
          s = t * c;
        }
        cs[k] = make_float2(c, s);
        pr[k] = make_int2(p, q);
      }
      __syncthreads();
      for (int e = tid; e < half * m; e += nt) {  // rows: A <- J^T A
        int k = e / m, col = e % m;
        float2 r = cs[k];
        int2 pq = pr[k];
        float ap = A[pq.x * ld + col], aq = A[pq.y * ld + col];
        A[pq.x * ld + col] = r.x * ap - r.y * aq;
        A[pq.y * ld + col] = r.y * ap + r.x * aq;
      }
      __syncthreads();
      for (int e = tid; e < half * m; e += nt) {  // columns: A <- A J, Z <- Z J
        int k = e / m, row = e % m;
        float2 r = cs[k];
        int2 pq = pr[k];
        float ap = A[row * ld + pq.x], aq = A[row * ld + pq.y];
        A[row * ld + pq.x] = r.x * ap - r.y * aq;
        A[row * ld + pq.y] = r.y * ap + r.x * aq;
        float zp = Z[row * ld + pq.x], zq = Z[row * ld + pq.y];
        Z[row * ld + pq.x] = r.x * zp - r.y * zq;
        Z[row * ld + pq.y] = r.y * zp + r.x * zq;
      }
      __syncthreads();
    }
  }
}

// Orthonormalises columns b0 .. b0 + nb - 1 (nb <= 8) of Q (column c at Q + c ldq, RPL
// rows a lane: row lane + 32 k) inside one warp, one column after the other, each
// projected twice against the block's earlier columns (classical Gram-Schmidt, twice);
// the columns before the block are already projected out.  A column that is numerically
// in the span of the earlier ones (its norm falls below 1e-5 of what it was) restarts
// from a fixed +-1 pattern projected against every earlier column, and is zero if that
// fails too.
template <int RPL>
__device__ __noinline__ void orth_block_warp(float* Q, int ldq, int b0, int nb, int lane) {
  float x[8][RPL];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int k = 0; k < RPL; ++k) x[j][k] = j < nb ? Q[(b0 + j) * ldq + lane + 32 * k] : 0.f;
  auto warp_sum = [](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= nb) break;
    float n0 = 0.f;
#pragma unroll
    for (int k = 0; k < RPL; ++k) n0 = fmaf(x[j][k], x[j][k], n0);
    const float nrm0 = sqrtf(warp_sum(n0));
    for (int attempt = 0; attempt < 2; ++attempt) {
      for (int pass = 0; pass < 2; ++pass) {
        if (attempt == 1) {  // a restarted column: the columns before the block as well
          for (int cc = 0; cc < b0; ++cc) {
            float sd = 0.f;
#pragma unroll
            for (int k = 0; k < RPL; ++k) sd = fmaf(Q[cc * ldq + lane + 32 * k], x[j][k], sd);
            sd = warp_sum(sd);
#pragma unroll
            for (int k = 0; k < RPL; ++k) x[j][k] = fmaf(-sd, Q[cc * ldq + lane + 32 * k], x[j][k]);
          }
        }
        float sd[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          sd[jj] = 0.f;
          if (jj < j) {
#pragma unroll
            for (int k = 0; k < RPL; ++k) sd[jj] = fmaf(x[jj][k], x[j][k], sd[jj]);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (jj < j) sd[jj] += __shfl_xor_sync(0xffffffffu, sd[jj], o);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
          if (jj < j) {
#pragma unroll
            for (int k = 0; k < RPL; ++k) x[j][k] = fmaf(-sd[jj], x[jj][k], x[j][k]);
          }
      }
      float n1 = 0.f;
#pragma unroll
      for (int k = 0; k < RPL; ++k) n1 = fmaf(x[j][k], x[j][k], n1);
      const float nrm = sqrtf(warp_sum(n1));
      if (nrm > 1e-5f * nrm0 && nrm > 1e-30f) {
        const float inv = 1.f / nrm;
#pragma unroll
        for (int k = 0; k < RPL; ++k) x[j][k] *= inv;
        break;
      }
#pragma unroll
      for (int k = 0; k < RPL; ++k)
        x[j][k] = attempt == 0 ? ((hash32((uint32_t)((lane + 32 * k) * 7 + (b0 + j) * 104729 + 99991)) & 1u) ? 1.f : -1.f)
                               : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < nb) {
#pragma unroll
      for (int k = 0; k < RPL; ++k) Q[(b0 + j) * ldq + lane + 32 * k] = x[j][k];
    }
}

template <int D>
__global__ void __launch_bounds__(kCThreads, 1) compress_kernel(CArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const Layout& L = a.L;
  constexpr int n = 2 * D;
  const int p = a.p;
  const int r = L.r, r8 = L.r8, R = L.R, R8 = L.R8;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int u = blockIdx.y, sb = blockIdx.x, blk = a.blk0 + sb;
  uint8_t* unit = a.cache + (uint64_t)u * L.unit_stride;

  if (sb == a.nblk) {  // ---------------- exact recency window
    const __half* Kw = a.K + ((size_t)u * a.T + (size_t)a.nblk * 256) * D;
    const __half* Vw = a.V + ((size_t)u * a.T + (size_t)a.nblk * 256) * D;
    uint8_t* win = unit + L.off_window;
    for (int e = tid; e < L.W16 * D; e += nt) {
      int t = e / D, j = e % D;
      __half kv = __float2half(0.f), vv = kv;
      if (t < L.W) { kv = Kw[(size_t)t * D + j]; vv = Vw[(size_t)t * D + j]; }
      *reinterpret_cast<__half*>(win + win_k_off(L, t, j)) = kv;
      *reinterpret_cast<__half*>(win + win_v_off(L, t, j)) = vv;
    }
    return;
  }

  float* R1 = reinterpret_cast<float*>(sm);
  float* Qb = reinterpret_cast<float*>(sm + a.off_q);
  __half* Xc = reinterpret_cast<__half*>(sm + a.off_xc);
  float* anc = reinterpret_cast<float*>(sm + a.off_misc);  // [n]
  float* errv = anc + n;                                   // [256]
  float* red = errv + 256;                                 // [64]
  float* vec = red + 64;                                   // [128]
  float* ubuf = vec + 128;                                 // [17][128]
  float2* cs = reinterpret_cast<float2*>(ubuf + 17 * 128); // [64]
  int2* pr = reinterpret_cast<int2*>(cs + 64);             // [64]
  int* sel = reinterpret_cast<int*>(pr + 64);              // [256]
  int* flag = sel + 256;                                   // [256]

  const __half* Kb = a.K + ((size_t)u * a.T + (size_t)sb * 256) * D;
  const __half* Vb = a.V + ((size_t)u * a.T + (size_t)sb * 256) * D;
  uint8_t* bp = unit + L.off_blocks + (uint64_t)blk * L.block_stride;

  // ---- anchor, router min / max, anchors in the block record
  for (int i = tid; i < n; i += nt) anc[i] = i < D ? h2f(Kb[i]) : h2f(Vb[i - D]);
  for (int j = tid; j < D; j += nt) {
    if (L.rope) {
      // un-rotated pool: the box of the keys rotated to positions 256 blk + t, in fp32
      const int h = L.rope / 2, jj = j < h ? j : j - h, jp = j < h ? j + h : j - h;
      const float2* tab = reinterpret_cast<const float2*>(a.cache + L.off_rope);
      float mn = INFINITY, mx = -INFINITY;
      for (int t = 0; t < 256; ++t) {
        float x = h2f(Kb[(size_t)t * D + j]);
        if (j < L.rope) {
          const float y = h2f(Kb[(size_t)t * D + jp]);
          const float2 c = rope_cs(tab, L.rope_pages, h, 256 * blk + t, jj);
          x = j < h ? fmaf(x, c.x, -y * c.y) : fmaf(x, c.x, y * c.y);
        }
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      float* router = reinterpret_cast<float*>(unit + L.off_router + (uint64_t)blk * 8 * D);
      router[j] = mn;
      router[D + j] = mx;
    } else {
      __half mn = Kb[j], mx = Kb[j];
      for (int t = 1; t < 256; ++t) {
        __half v = Kb[(size_t)t * D + j];
        if (__hlt(v, mn)) mn = v;
        if (__hgt(v, mx)) mx = v;
      }
      __half* router = reinterpret_cast<__half*>(unit + L.off_router + (uint64_t)blk * 4 * D);
      router[j] = mn;
      router[D + j] = mx;
    }
    reinterpret_cast<__half*>(bp)[j] = Kb[j];
    reinterpret_cast<__half*>(bp)[D + j] = Vb[j];
  }
  __syncthreads();

  // ---- Gram G = X^T X, X = raw rows 1..255 minus the anchor (fp32)
  const int n8 = n / 8;
  const int ntiles = n8 * (n8 + 1) / 2;
  int TI = 0, TJ = 0;
  const bool owner = tid < ntiles;
  if (owner) {
    int rem = tid;
    while (rem >= n8 - TI) { rem -= n8 - TI; ++TI; }
    TJ = TI + rem;
  }
  float acc[8][8];
#pragma unroll
  for (int x = 0; x < 8; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
  float ai[8], aj[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) { ai[x] = anc[8 * TI + x]; aj[x] = anc[8 * TJ + x]; }
  for (int t0 = 1; t0 < 256; t0 += kChunk) {
    const int nv = min(kChunk, 256 - t0);
    __syncthreads();
    for (int e = tid; e < nv * (n / 8); e += nt) {  // 16-byte pieces of K|V rows
      int k = e / (n / 8), piece = e % (n / 8);
      int col = piece * 8;
      const __half* src = col < D ? Kb + (size_t)(t0 + k) * D + col : Vb + (size_t)(t0 + k) * D + (col - D);
      *reinterpret_cast<uint4*>(Xc + k * n + col) = *reinterpret_cast<const uint4*>(src);
    }
    __syncthreads();
    if (owner) {
      for (int k = 0; k < nv; ++k) {
        uint4 vi = *reinterpret_cast<const uint4*>(Xc + k * n + 8 * TI);
        uint4 vj = *reinterpret_cast<const uint4*>(Xc + k * n + 8 * TJ);
        const __half* hi = reinterpret_cast<const __half*>(&vi);
        const __half* hj = reinterpret_cast<const __half*>(&vj);
        float xi[8], xj[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) { xi[x] = h2f(hi[x]) - ai[x]; xj[x] = h2f(hj[x]) - aj[x]; }
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
          for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(xi[x], xj[y], acc[x][y]);
      }
    }
  }
  __syncthreads();

  const int ldh = a.full ? (n + 1) : (p + 1);  // leading dim of H and Z
  float* H = nullptr;
  float* Z = nullptr;
  if (a.full) {
    // whole Gram in full storage, then Jacobi on it
    H = R1;
    Z = R1 + n * ldh;
    if (owner) {
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) {
          H[(8 * TI + x) * ldh + 8 * TJ + y] = acc[x][y];
          H[(8 * TJ + y) * ldh + 8 * TI + x] = acc[x][y];
        }
    }
    for (int e = tid; e < n * n; e += nt) Z[(e / n) * ldh + e % n] = (e / n == e % n) ? 1.f : 0.f;
    __syncthreads();
    jacobi(H, Z, n, ldh, red, cs, pr);
  } else {
    // the Gram's upper triangle as 8x8 tiles: tile (TI, TJ), TI <= TJ, is the owner's, at
    // 64 tid floats (rows of the tile contiguous)
    if (owner) {
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; y += 4)
          *reinterpret_cast<float4*>(R1 + tid * 64 + 8 * x + y) =
              make_float4(acc[x][y], acc[x][y + 1], acc[x][y + 2], acc[x][y + 3]);
    }
    // start block: fixed +-1 pattern
    const int ldq = n + 1;
    for (int e = tid; e < n * p; e += nt) {
      int i = e % n, c = e / n;
      Qb[c * ldq + i] = (hash32((uint32_t)(i * 131 + c * 7919 + 17)) & 1u) ? 1.f : -1.f;
    }
    __syncthreads();
    for (int it = 0; it <= kIters + 1; ++it) {
      // ---- Y = G Q: warps 0..15 own the 8-row blocks w and w + 16, lanes the columns lane and
      // lane + 32; per 8-row block J of Q one Gram tile (a broadcast to the warp), read
      // transposed below the diagonal
      float y[2][8][2];
#pragma unroll
      for (int bb = 0; bb < 2; ++bb)
#pragma unroll
        for (int x = 0; x < 8; ++x) y[bb][x][0] = y[bb][x][1] = 0.f;
      const bool gw = warp < 16;
      const int c0 = lane, c1 = lane + 32;
      if (gw) {
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int I = warp + 16 * bb;
          for (int J = 0; J < n8; ++J) {
            float q0[8], q1[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              q0[e] = c0 < p ? Qb[c0 * ldq + 8 * J + e] : 0.f;
              q1[e] = c1 < p ? Qb[c1 * ldq + 8 * J + e] : 0.f;
            }
            const int lo = I < J ? I : J, hi = I < J ? J : I;
            const float4* T4 = reinterpret_cast<const float4*>(R1 + (lo * n8 - (lo * (lo - 1)) / 2 + (hi - lo)) * 64);
            if (I <= J) {  // G[8I + x][8J + e] = T[x][e]
#pragma unroll
              for (int x = 0; x < 8; ++x) {
                const float4 ga = T4[2 * x], gb = T4[2 * x + 1];
                const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  y[bb][x][0] = fmaf(g[e], q0[e], y[bb][x][0]);
                  y[bb][x][1] = fmaf(g[e], q1[e], y[bb][x][1]);
                }
              }
            } else {  // G[8I + x][8J + e] = T[e][x] of tile (J, I)
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 ga = T4[2 * e], gb = T4[2 * e + 1];
                const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                  y[bb][x][0] = fmaf(g[x], q0[e], y[bb][x][0]);
                  y[bb][x][1] = fmaf(g[x], q1[e], y[bb][x][1]);
                }
              }
            }
          }
        }
      }
      __syncthreads();
      if (it <= kIters) {
        // Q <- orth(Y): classical Gram-Schmidt, twice
        if (gw) {
#pragma unroll
          for (int bb = 0; bb < 2; ++bb)
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const int i = 8 * (warp + 16 * bb) + x;
              if (c0 < p) Qb[c0 * ldq + i] = y[bb][x][0];
              if (c1 < p) Qb[c1 * ldq + i] = y[bb][x][1];
            }
        }
        __syncthreads();
        // 8 columns at a time: the block is projected twice against the columns before it,
        // then warp 0 orthonormalises the block's columns one after the other, twice against
        // each earlier one.  For the projection the block also sits row-major in Yt (the
        // staging area of X, idle here): a dot-product thread (earlier column cc, half of the
        // rows) reads Q's column once and the block's row as two broadcast 16-byte loads,
        // and an update thread (row i) takes every earlier column's 8 coefficients the same way.
        float* Yt = reinterpret_cast<float*>(Xc);  // [n][8]
        float* part = ubuf;                         // [2 halves][64][8] partial coefficients
        for (int b0 = 0; b0 < p; b0 += 8) {
          const int nb = min(8, p - b0);
          if (b0 > 0) {
            for (int i = tid; i < n; i += nt) {
              float v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = j < nb ? Qb[(b0 + j) * ldq + i] : 0.f;
              *reinterpret_cast<float4*>(Yt + 8 * i) = make_float4(v[0], v[1], v[2], v[3]);
              *reinterpret_cast<float4*>(Yt + 8 * i + 4) = make_float4(v[4], v[5], v[6], v[7]);
            }
            __syncthreads();
            for (int pass = 0; pass < 2; ++pass) {
              if (tid < 2 * b0) {  // coefficients of column cc over one half of the rows
                const int cc = tid % b0, hh = tid / b0;
                const float* qp = Qb + cc * ldq;
                float c8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int i = hh * (n / 2); i < (hh + 1) * (n / 2); ++i) {
                  const float qv = qp[i];
                  const float4 ya = *reinterpret_cast<const float4*>(Yt + 8 * i);
                  const float4 yb = *reinterpret_cast<const float4*>(Yt + 8 * i + 4);
                  c8[0] = fmaf(qv, ya.x, c8[0]); c8[1] = fmaf(qv, ya.y, c8[1]);
                  c8[2] = fmaf(qv, ya.z, c8[2]); c8[3] = fmaf(qv, ya.w, c8[3]);
                  c8[4] = fmaf(qv, yb.x, c8[4]); c8[5] = fmaf(qv, yb.y, c8[5]);
                  c8[6] = fmaf(qv, yb.z, c8[6]); c8[7] = fmaf(qv, yb.w, c8[7]);
                }
                float* pc = part + (hh * 64 + cc) * 8;
                *reinterpret_cast<float4*>(pc) = make_float4(c8[0], c8[1], c8[2], c8[3]);
                *reinterpret_cast<float4*>(pc + 4) = make_float4(c8[4], c8[5], c8[6], c8[7]);
              }
              __syncthreads();
              for (int i = tid; i < n; i += nt) {  // row i of the block minus its projection
                const float4 ya = *reinterpret_cast<const float4*>(Yt + 8 * i);
                const float4 yb = *reinterpret_cast<const float4*>(Yt + 8 * i + 4);
                float v[8] = {ya.x, ya.y, ya.z, ya.w, yb.x, yb.y, yb.z, yb.w};
                for (int cc = 0; cc < b0; ++cc) {
                  const float qv = Qb[cc * ldq + i];
                  const float4 a0 = *reinterpret_cast<const float4*>(part + cc * 8);
                  const float4 a1 = *reinterpret_cast<const float4*>(part + cc * 8 + 4);
                  const float4 b0v = *reinterpret_cast<const float4*>(part + (64 + cc) * 8);
                  const float4 b1v = *reinterpret_cast<const float4*>(part + (64 + cc) * 8 + 4);
                  v[0] = fmaf(-(a0.x + b0v.x), qv, v[0]); v[1] = fmaf(-(a0.y + b0v.y), qv, v[1]);
                  v[2] = fmaf(-(a0.z + b0v.z), qv, v[2]); v[3] = fmaf(-(a0.w + b0v.w), qv, v[3]);
                  v[4] = fmaf(-(a1.x + b1v.x), qv, v[4]); v[5] = fmaf(-(a1.y + b1v.y), qv, v[5]);
                  v[6] = fmaf(-(a1.z + b1v.z), qv, v[6]); v[7] = fmaf(-(a1.w + b1v.w), qv, v[7]);
                }
                *reinterpret_cast<float4*>(Yt + 8 * i) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(Yt + 8 * i + 4) = make_float4(v[4], v[5], v[6], v[7]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (j < nb) Qb[(b0 + j) * ldq + i] = v[j];
              }
              __syncthreads();
            }
          }
          if (warp == 0) orth_block_warp<n / 32>(Qb, ldq, b0, nb, lane);
          __syncthreads();
        }
      } else {
        // ---- Rayleigh-Ritz: Y into R1 (the Gram is no longer needed), H = Q^T Y
        if (gw) {
#pragma unroll
          for (int bb = 0; bb < 2; ++bb)
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              const int i = 8 * (warp + 16 * bb) + x;
              if (c0 < p) R1[c0 * ldq + i] = y[bb][x][0];
              if (c1 < p) R1[c1 * ldq + i] = y[bb][x][1];
            }
        }
        __syncthreads();
        H = R1 + p * ldq;
        Z = H + p * ldh;
        for (int e = warp; e < p * p; e += nw) {
          const int c = e / p, c2 = e % p;
          if (c2 < c) continue;
          float s = 0.f;
          for (int i = lane; i < n; i += 32) s = fmaf(Qb[c * ldq + i], R1[c2 * ldq + i], s);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          if (lane == 0) { H[c * ldh + c2] = s; H[c2 * ldh + c] = s; }
        }
        for (int e = tid; e < p * p; e += nt) Z[(e / p) * ldh + e % p] = (e / p == e % p) ? 1.f : 0.f;
        __syncthreads();
        jacobi(H, Z, p, ldh, red, cs, pr);
      }
    }
  }

  // ---- top-r eigenpairs (eigenvalue desc, ties to the lower index)
  const int m = a.full ? n : p;
  for (int k = tid; k < 256; k += nt) sel[k] = 0;  // in-range even if non-finite values break the ranking
  __syncthreads();
  for (int c = tid; c < m; c += nt) {
    const float lc = H[c * ldh + c];
    int rank = 0;
    for (int c2 = 0; c2 < m; ++c2) {
      const float l2 = H[c2 * ldh + c2];
      rank += (l2 > lc) || (l2 == lc && c2 < c);
    }
    if (rank < r) sel[rank] = c;
  }
  __syncthreads();
  // W [n][r] (row-major) at the start of R1: W = Z[:, sel] (full) or Q Z[:, sel]
  float* Wm = R1;
  if (a.full) {
    // Z lives above the W area (n * r <= n * ldh), H is dead
    for (int e = tid; e < n * r; e += nt) {
      const int i = e / r, k = e % r;
      Wm[i * r + k] = Z[i * ldh + sel[k]];
    }
  } else {
    // Y (dead) occupies [0, p*ldq); W [n*r] fits there; H and Z sit above it
    const int ldq = n + 1;
    for (int e = tid; e < n * r; e += nt) {
      const int i = e / r, k = e % r;
      const int zc = sel[k];
      float s = 0.f;
      for (int c = 0; c < p; ++c) s = fmaf(Qb[c * ldq + i], Z[c * ldh + zc], s);
      Wm[i * r + k] = s;
    }
  }
  __syncthreads();

  // ---- U = X W per token, key error, U rows into the packed layout
  for (int t0 = 1; t0 < 256; t0 += kChunk) {
    const int nv = min(kChunk, 256 - t0);
    __syncthreads();
    for (int e = tid; e < nv * (n / 8); e += nt) {
      int k = e / (n / 8), piece = e % (n / 8);
      int col = piece * 8;
      const __half* src = col < D ? Kb + (size_t)(t0 + k) * D + col : Vb + (size_t)(t0 + k) * D + (col - D);
      *reinterpret_cast<uint4*>(Xc + k * n + col) = *reinterpret_cast<const uint4*>(src);
    }
    __syncthreads();
    for (int k = warp; k < nv; k += nw) {
      const int tok = t0 + k;
      const __half* xr = Xc + k * n;
      float* ub = ubuf + warp * 128;
      for (int kk = lane; kk < r; kk += 32) {
        float s = 0.f;
        for (int i = 0; i < n; ++i) s = fmaf(h2f(xr[i]) - anc[i], Wm[i * r + kk], s);
        ub[kk] = s;
      }
      __syncwarp();
      float e2 = 0.f;
      for (int j = lane; j < D; j += 32) {
        float kh = 0.f;
        for (int kk = 0; kk < r; ++kk) kh = fmaf(ub[kk], Wm[j * r + kk], kh);
        const float dlt = (h2f(xr[j]) - anc[j]) - kh;
        e2 = fmaf(dlt, dlt, e2);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) e2 += __shfl_xor_sync(0xffffffffu, e2, o);
      if (lane == 0) errv[tok - 1] = sqrtf(e2);
      for (int kk = lane; kk < r8; kk += 32) {
        const __half v = kk < r ? to_h(ub[kk], a.err) : __float2half(0.f);
        *reinterpret_cast<__half*>(bp + blk_u_off(L, tok, kk)) = v;
      }
      __syncwarp();
    }
  }
  // U row 0 (the anchor) is zero
  for (int kk = tid; kk < r8; kk += nt)
    *reinterpret_cast<__half*>(bp + blk_u_off(L, 0, kk)) = __float2half(0.f);
  __syncthreads();

  // ---- residual selection: R largest errors, ties to the lower token
  for (int i = tid; i < 255; i += nt) {
    const float ei = errv[i];
    int rank = 0;
    for (int j = 0; j < 255; ++j) {
      const float ej = errv[j];
      rank += (ej > ei) || (ej == ei && j < i);
    }
    flag[i] = rank < R;
  }
  __syncthreads();
  for (int i = tid; i < 255; i += nt) {
    if (!flag[i]) continue;
    int pos = 0;
    for (int j = 0; j < i; ++j) pos += flag[j];
    sel[pos] = i + 1;  // token position
  }
  if (tid < 8) {
    uint32_t w = 0;
    for (int b = 0; b < 32; ++b) {
      const int tok = tid * 32 + b;
      if (tok >= 1 && flag[tok - 1]) w |= 1u << b;
    }
    reinterpret_cast<uint32_t*>(bp + L.off_mask)[tid] = w;
  }
  __syncthreads();
  const int nres = min(R, 255);
  uint16_t* cold = reinterpret_cast<uint16_t*>(unit + L.off_cold) + (size_t)blk * R8;
  for (int i = tid; i < R8; i += nt) cold[i] = i < nres ? (uint16_t)sel[i] : 0;
  if (L.qbits) {  // group-quantised residual rows (every thread of the CTA takes part)
    write_quant_residuals(
        L, bp + L.off_res, nres, [&](int i, int j) { return Kb[(size_t)sel[i] * D + j]; },
        [&](int i, int j) { return Vb[(size_t)sel[i] * D + j]; });
  } else {
    for (int e = tid; e < R8 * D; e += nt) {
      const int i = e / D, j = e % D;
      __half kv = __float2half(0.f), vv = kv;
      if (i < nres) { kv = Kb[(size_t)sel[i] * D + j]; vv = Vb[(size_t)sel[i] * D + j]; }
      *reinterpret_cast<__half*>(bp + blk_resk_off(L, i, j)) = kv;
      *reinterpret_cast<__half*>(bp + blk_resv_off(L, i, j)) = vv;
    }
  }
  // ---- V_K (B^T layout) and V_V from W
  for (int e = tid; e < r8 * D; e += nt) {
    const int k = e / D, j = e % D;
    __half vk = __float2half(0.f), vv = vk;
    if (k < r) { vk = to_h(Wm[j * r + k], a.err); vv = to_h(Wm[(D + j) * r + k], a.err); }
    *reinterpret_cast<__half*>(bp + L.off_vk + bt_layout_off(r8, D, k, j)) = vk;
    *reinterpret_cast<__half*>(bp + blk_vv_off(L, k, j)) = vv;
  }
}

struct CPlan {
  int n, p, full;
  uint32_t off_q, off_xc, off_misc, smem;
};

CPlan plan(const Layout& L) {
  CPlan c;
  c.n = 2 * L.d;
  c.full = L.d == 64;
  c.p = c.full ? c.n : (L.r + 16 < 64 ? L.r + 16 : 64);
  if (c.p < 1) c.p = 1;
  uint32_t r1;
  if (c.full) {
    r1 = (uint32_t)(2 * c.n * (c.n + 1) * 4);
  } else {
    const uint32_t gram = (uint32_t)((c.n / 8) * (c.n / 8 + 1) / 2 * 64 * 4);  // 8x8 tiles of the upper triangle
    const uint32_t rr = (uint32_t)((c.p * (c.n + 1) + 2 * c.p * (c.p + 1)) * 4);
    r1 = gram > rr ? gram : rr;
  }
  r1 = (uint32_t)round_up(r1, 16);
  c.off_q = r1;
  const uint32_t q = c.full ? 0u : (uint32_t)(c.p * (c.n + 1) * 4);
  c.off_xc = (uint32_t)round_up(c.off_q + q, 16);
  c.off_misc = c.off_xc + (uint32_t)(kChunk * c.n * 2);
  const uint32_t misc = (uint32_t)((c.n + 256 + 64 + 128 + 17 * 128) * 4 + 64 * 8 + 64 * 8 + 2 * 256 * 4);
  c.smem = c.off_misc + misc;
  return c;
}

template <int D>
cudaError_t launch_t(const CArgs& a, uint32_t smem, cudaStream_t s) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(compress_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nblk + (a.with_window ? 1 : 0), a.L.units);
  if (grid.x == 0) return cudaSuccess;
  compress_kernel<D><<<grid, kCThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t compress_ws_bytes(const Layout& L) {
  (void)L;
  return kWsHeader;
}

cudaError_t launch_compress_blocks(const Layout& L, const __half* K, const __half* V, int T, int blk0, int nblk,
                                   uint8_t* cache, uint32_t* err, cudaStream_t s) {
  CPlan c = plan(L);
  CArgs a;
  a.L = L;
  a.K = K;
  a.V = V;
  a.cache = cache;
  a.err = err;
  a.T = T;
  a.blk0 = blk0;
  a.nblk = nblk;
  a.with_window = 0;
  a.n = c.n;
  a.p = c.p;
  a.full = c.full;
  a.off_q = c.off_q;
  a.off_xc = c.off_xc;
  a.off_misc = c.off_misc;
  if (L.d == 128) return launch_t<128>(a, c.smem, s);
  return launch_t<64>(a, c.smem, s);
}

cudaError_t launch_compress(const Layout& L, const __half* K, const __half* V, uint8_t* cache, uint8_t* ws,
                            uint32_t* err, cudaStream_t s) {
  (void)ws;
  cudaError_t e = cudaMemsetAsync(cache, 0, L.total, s);
  if (e != cudaSuccess) return e;
  e = launch_rope_tables(L, cache, s);  // the boxes of an un-rotated pool read them
  if (e != cudaSuccess) return e;
  CPlan c = plan(L);
  CArgs a;
  a.L = L;
  a.K = K;
  a.V = V;
  a.cache = cache;
  a.err = err;
  a.T = L.NB * 256 + L.W;
  a.blk0 = 0;
  a.nblk = L.NB;
  a.with_window = 1;
  a.n = c.n;
  a.p = c.p;
  a.full = c.full;
  a.off_q = c.off_q;
  a.off_xc = c.off_xc;
  a.off_misc = c.off_misc;
  if (L.d == 128) return launch_t<128>(a, c.smem, s);
  return launch_t<64>(a, c.smem, s);
}

}  // namespace dkv
