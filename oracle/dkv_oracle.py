"""Plain fp64 CPU oracle for DKV decode attention over an anchor + low-rank
differential KV cache.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``; the
product path never imports, links or runs anything in this directory.  It
shares no code, header, table or constant with the CUDA library.

Sources (cited by page title and section):

* [DKV-Z]   "DKV: Anchor + Low-Rank Differential KV-Cache Compression for
            Scalable Long-Context Inference" (Zenodo record), abstract.
* [README]  "Differential-KV (DKV): Anchor + Low-Rank KV-Cache Compression"
            (project README), sections "Core Architecture & Paper Overview"
            (Core), "Core Innovations" (Innov), "Key Environment Knobs"
            (Knobs), "Measured Paper Benchmarks" (Bench).

What is computed (and where the pages are silent, the reading taken):

* compression of one 256-token block: exact anchor = first token; joint K|V
  truncated SVD of the deltas to the anchor, S folded into U; exact residual
  rows = the R rows whose key the low-rank part reconstructs worst (plain L2
  key error, ties to the lower row); per-block key min/max (router bounds);
* decode: top-K routing on the per-block upper bound of the GQA-averaged
  query against the key box; attention over the routed blocks (anchor,
  low-rank rows, exact residual rows) and the exact recency window.  The
  plain definition is implemented by materialising the reconstructed keys and
  values of the routed blocks and taking one softmax; the factored form
  (low-rank scoring, low-rank value, split log-sum-exp merge) is implemented
  separately so that the two can pin each other.

Everything runs in float64 on float64 copies of the (fp16) inputs.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK_SIZE = 256  # [README Core] fixed micro-blocks of B_s = 256 tokens


# ---------------------------------------------------------------------------
# compression
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Block:
    """One compressed block (all fields float64 except ``S``).

    a_k, a_v   [d]        exact anchor token (the block's first token)
    U          [255, r]   low-rank coefficients of tokens 1..255, S folded in
    V_K, V_V   [r, d]     key / value halves of the joint right basis
    S          [R]        token positions (1..255, ascending) kept exact
    K_res,V_res[R, d]     the exact rows at those positions
    kmin, kmax [d]        per-channel key extremes over the 256 tokens
    sigma      [m]        singular values of the delta matrix (diagnostic)
    err        [255]      key reconstruction error of tokens 1..255
    """

    a_k: np.ndarray
    a_v: np.ndarray
    U: np.ndarray
    V_K: np.ndarray
    V_V: np.ndarray
    S: np.ndarray
    K_res: np.ndarray
    V_res: np.ndarray
    kmin: np.ndarray
    kmax: np.ndarray
    sigma: np.ndarray | None = None
    err: np.ndarray | None = None

    @property
    def rank(self) -> int:
        return self.U.shape[1]


def select_residuals(err: np.ndarray, n_residual: int) -> np.ndarray:
    """Exact-residual selection by worst reconstruction.

    [DKV-Z] keeps as exact residual tokens "the rows the low-rank basis
    reconstructs worst"; [README Innov, "Content-Aware / Rarity-Aware Residual
    Selection"] names the vanilla criterion arg max ||k - k_hat||_2.  ``err``
    holds that error for tokens 1..255; the R largest are kept, equal errors
    going to the lower token.  Returns token positions (1..255), ascending.
    """
    n = err.shape[0]
    R = max(0, min(int(n_residual), n))
    order = sorted(range(n), key=lambda i: (-float(err[i]), i))[:R]
    return np.array(sorted(i + 1 for i in order), dtype=np.int64)


def compress_block(Kb: np.ndarray, Vb: np.ndarray, rank: int, n_residual: int) -> Block:
    """Anchor + joint K|V truncated SVD + exact residuals for one block.

    [README Core] items 1-3 and [DKV-Z]: the anchor (a_k, a_v) is the block's
    first token kept exact; the other 255 tokens are stored as a rank-r joint
    K|V truncated SVD delta with U in R^{255 x r} and V_K, V_V in R^{r x d};
    a budget of R exact residual rows is kept beside it.

    Step by step:
    1. a_k = K[0], a_v = V[0].
    2. X_i = [K[i] - a_k | V[i] - a_v] for i = 1..255 (delta to the anchor).
    3. X = U_hat diag(sigma) W^T (LAPACK, fp64); U = U_hat[:, :r] diag(sigma[:r])
       (S folded into U); V_K = W^T[:r, :d], V_V = W^T[:r, d:].
    4. err_i = ||(K[i] - a_k) - U_i V_K||_2 and the R worst rows are kept exact.
    5. kmin, kmax = channel-wise min / max of the 256 exact keys ([README Bench],
       table "Per-Block Memory Breakdown": "Key Min/Max ... Decode router bounds").
    """
    Kb = np.asarray(Kb, dtype=np.float64)
    Vb = np.asarray(Vb, dtype=np.float64)
    n, d = Kb.shape
    if n != BLOCK_SIZE or Vb.shape != Kb.shape:
        raise ValueError("a block is 256 tokens of K and V with the same head_dim")
    a_k, a_v = Kb[0].copy(), Vb[0].copy()
    dK = Kb[1:] - a_k
    dV = Vb[1:] - a_v
    X = np.concatenate([dK, dV], axis=1)                      # [255, 2d]
    U_hat, sigma, Wt = np.linalg.svd(X, full_matrices=False)  # fp64 LAPACK
    r = max(0, min(int(rank), sigma.shape[0]))
    U = U_hat[:, :r] * sigma[:r]
    V_K = Wt[:r, :d].copy()
    V_V = Wt[:r, d:].copy()
    err = np.sqrt(((dK - U @ V_K) ** 2).sum(axis=1))
    S = select_residuals(err, n_residual)
    return Block(a_k=a_k, a_v=a_v, U=U, V_K=V_K, V_V=V_V, S=S,
                 K_res=Kb[S].copy(), V_res=Vb[S].copy(),
                 kmin=Kb.min(axis=0), kmax=Kb.max(axis=0), sigma=sigma, err=err)


@dataclasses.dataclass(frozen=True)
class Rope:
    """Rotary position embedding of an un-rotated pool ([README Knobs]
    DKV_ROTATED_POOL=0: the pool stores keys before RoPE and rotates them to
    their absolute positions at read).  The pages name RoPE without restating
    it; the reading taken is the rotate-half form of the models they measure
    (Qwen2.5 / Qwen3.5 under Hugging Face): the first ``dims`` channels are
    rotated in pairs (j, j + dims/2) by the angle pos * base^(-2j/dims); the
    channels from ``dims`` on are left alone (partial RoPE, "64 of 256 dims" on
    Qwen3.5 in the README's verification list)."""

    dims: int
    base: float


def rope_angles(pos: np.ndarray, rope: Rope) -> np.ndarray:
    """[n, dims/2] angles pos_t * base^(-2j/dims), j = 0 .. dims/2 - 1."""
    h = rope.dims // 2
    theta = float(rope.base) ** (-2.0 * np.arange(h, dtype=np.float64) / rope.dims)
    return np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]


def apply_rope(X: np.ndarray, pos: np.ndarray, rope: Rope) -> np.ndarray:
    """Rows of X [n, d] rotated to positions pos [n]: for j < h = dims/2
        x'_j     = x_j cos(a_tj) - x_{j+h} sin(a_tj)
        x'_{j+h} = x_{j+h} cos(a_tj) + x_j sin(a_tj)
    and x'_c = x_c for c >= dims."""
    X = np.asarray(X, dtype=np.float64)
    out = X.copy()
    if rope.dims == 0 or X.shape[0] == 0:
        return out
    h = rope.dims // 2
    a = rope_angles(pos, rope)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = X[:, :h], X[:, h:2 * h]
    out[:, :h] = x1 * c - x2 * s
    out[:, h:2 * h] = x2 * c + x1 * s
    return out


def rope_key_box(Kb: np.ndarray, block_index: int, rope: Rope) -> tuple[np.ndarray, np.ndarray]:
    """Router box of a block in an un-rotated pool: the channel-wise min / max
    of its 256 exact keys rotated to their absolute positions 256 b .. 256 b +
    255 (the keys the decode scores; reading of [README Bench] "Decode router
    bounds" for a pool that rotates at read)."""
    pos = np.arange(block_index * BLOCK_SIZE, (block_index + 1) * BLOCK_SIZE)
    Kr = apply_rope(Kb, pos, rope)
    return Kr.min(axis=0), Kr.max(axis=0)


@dataclasses.dataclass
class Unit:
    """Compressed cache of one (layer, sequence, KV head): blocks + window.
    With ``rope`` set the pool is un-rotated: every stored key (anchors,
    low-rank factors, residual rows, window) is the key before RoPE; block b's
    token i sits at absolute position 256 b + i and window token w at
    256 NB + w."""

    blocks: list
    win_K: np.ndarray  # [W, d] exact recency window ([README Core] item 4)
    win_V: np.ndarray
    rope: Rope | None = None


def compress_unit(K: np.ndarray, V: np.ndarray, n_blocks: int, rank: int, n_residual: int,
                  rope: Rope | None = None) -> Unit:
    """Split a unit's T = n_blocks*256 + W tokens into compressed blocks and the
    exact recency window ([DKV-Z]: recent tokens exact, older ones compressed).
    With ``rope`` K holds keys before RoPE (an un-rotated pool): the blocks
    compress them as they are and only the router box is taken over the
    rotated keys (``rope_key_box``)."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    nb = int(n_blocks)
    blocks = []
    for b in range(nb):
        Kb, Vb = K[b * BLOCK_SIZE:(b + 1) * BLOCK_SIZE], V[b * BLOCK_SIZE:(b + 1) * BLOCK_SIZE]
        blk = compress_block(Kb, Vb, rank, n_residual)
        if rope is not None:
            kmin, kmax = rope_key_box(Kb, b, rope)
            blk = dataclasses.replace(blk, kmin=kmin, kmax=kmax)
        blocks.append(blk)
    return Unit(blocks=blocks, win_K=K[nb * BLOCK_SIZE:].copy(), win_V=V[nb * BLOCK_SIZE:].copy(), rope=rope)


def append_tokens(unit: Unit, K_new: np.ndarray, V_new: np.ndarray, window_capacity: int, rank: int,
                  n_residual: int) -> Unit:
    """Streaming append: new tokens join the exact recency window; whenever the
    window has no free slot left, its oldest 256 tokens are compressed into a
    new block and leave the window ([DKV-Z]: recent tokens exact, older ones
    compressed; [README Core] items 1-4 applied as tokens arrive).  Raises
    ValueError when a compression step finds fewer than 256 window tokens."""
    blocks = list(unit.blocks)
    win_K = [row for row in np.asarray(unit.win_K, dtype=np.float64)]
    win_V = [row for row in np.asarray(unit.win_V, dtype=np.float64)]
    K_new = np.asarray(K_new, dtype=np.float64)
    V_new = np.asarray(V_new, dtype=np.float64)
    i = 0
    while i < len(K_new):
        if len(win_K) == window_capacity:
            if len(win_K) < BLOCK_SIZE:
                raise ValueError("window capacity below one block")
            Kb = np.array(win_K[:BLOCK_SIZE])
            blk = compress_block(Kb, np.array(win_V[:BLOCK_SIZE]), rank, n_residual)
            if unit.rope is not None:  # the window's oldest tokens become block len(blocks), same positions
                kmin, kmax = rope_key_box(Kb, len(blocks), unit.rope)
                blk = dataclasses.replace(blk, kmin=kmin, kmax=kmax)
            blocks.append(blk)
            win_K = win_K[BLOCK_SIZE:]
            win_V = win_V[BLOCK_SIZE:]
            continue
        win_K.append(K_new[i])
        win_V.append(V_new[i])
        i += 1
    d = K_new.shape[1] if K_new.ndim == 2 else np.asarray(unit.win_K).shape[-1]
    as_arr = lambda rows: np.array(rows).reshape(len(rows), d)
    return Unit(blocks=blocks, win_K=as_arr(win_K), win_V=as_arr(win_V), rope=unit.rope)


def reconstruct_block(blk: Block) -> tuple[np.ndarray, np.ndarray]:
    """K_hat, V_hat [256, d] of a compressed block: row 0 the anchor, rows in S
    the stored exact rows, every other row a + U_i [V_K | V_V] ([README Core])."""
    d = blk.a_k.shape[0]
    Kh = np.empty((BLOCK_SIZE, d))
    Vh = np.empty((BLOCK_SIZE, d))
    Kh[0], Vh[0] = blk.a_k, blk.a_v
    Kh[1:] = blk.a_k + blk.U @ blk.V_K
    Vh[1:] = blk.a_v + blk.U @ blk.V_V
    if blk.S.size:
        Kh[blk.S] = blk.K_res
        Vh[blk.S] = blk.V_res
    return Kh, Vh


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def effective_top_k(top_k: int, n_blocks: int) -> int:
    """[README Knobs] DKV_TOPK_BLOCKS: blocks routed per decode step; the README's
    benchmark section ("attend every block (DKV_TOPK_BLOCKS=0)") reads 0 as
    every block.  K >= NB also attends every block."""
    if top_k < 0:
        raise ValueError("top_k must be >= 0")
    return n_blocks if (top_k == 0 or top_k >= n_blocks) else int(top_k)


def router_bounds(q: np.ndarray, kmin: np.ndarray, kmax: np.ndarray) -> np.ndarray:
    """Per-block upper bound on the group-mean query score.

    q [G, d] are the GQA group's queries (one KV head).  [README Knobs]
    DKV_CB_GQA_ROUTE routes on the head-averaged query; [README Bench] stores
    per-block key min/max as the "Decode router bounds".  With
    qbar = mean_g (c q_g), c = 1/sqrt(d):
        bound_b = sum_j max(qbar_j * kmax_bj, qbar_j * kmin_bj)
    which is >= qbar . k for every key k in the block's box.
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[1]
    qbar = (q / math.sqrt(d)).mean(axis=0)
    kmin = np.asarray(kmin, dtype=np.float64)
    kmax = np.asarray(kmax, dtype=np.float64)
    return np.maximum(qbar[None, :] * kmax, qbar[None, :] * kmin).sum(axis=1)


def route(bounds: np.ndarray, top_k: int) -> np.ndarray:
    """Top-K blocks by (bound descending, block index ascending); the routed
    indices are returned in ascending order ([DKV-Z]: "routes to the top-K
    relevant blocks")."""
    nb = bounds.shape[0]
    k = effective_top_k(top_k, nb)
    order = sorted(range(nb), key=lambda b: (-float(bounds[b]), b))[:k]
    return np.array(sorted(order), dtype=np.int64)


# ---------------------------------------------------------------------------
# decode: plain definition
# ---------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """o_g = softmax(c q_g K^T) V and lse_g = log sum exp(c q_g K^T), c = 1/sqrt(d)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    s = (q / math.sqrt(q.shape[1])) @ K.T                   # [G, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return (e @ V) / l, (m + np.log(l))[:, 0]


def decode_unit(q: np.ndarray, unit: Unit, top_k: int) -> dict:
    """Decode attention of one unit, by definition.

    [DKV-Z]: route to the top-K relevant blocks, attend them and the dense
    recency window.  Token set = for each routed block its anchor, its
    reconstructed low-rank rows and its exact residual rows; then the W window
    tokens.  One softmax over that set (the split log-sum-exp merge the pages
    describe reaches the same value; see ``decode_unit_factored``).  In an
    un-rotated pool (``unit.rope``) every key of the set is rotated to its
    absolute position before it is scored; q is the query as the model gives
    it (already rotated to its own position); values are not rotated.
    Returns o [G, d], lse [G], idx (routed blocks, ascending), bounds [NB].
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[1]
    nb = len(unit.blocks)
    if nb:
        kmin = np.stack([b.kmin for b in unit.blocks])
        kmax = np.stack([b.kmax for b in unit.blocks])
        bounds = router_bounds(q, kmin, kmax)
        idx = route(bounds, top_k)
    else:
        bounds = np.zeros(0)
        idx = np.zeros(0, dtype=np.int64)
    Ks, Vs = [], []
    for b in idx:
        Kh, Vh = reconstruct_block(unit.blocks[b])
        if unit.rope is not None:
            Kh = apply_rope(Kh, np.arange(b * BLOCK_SIZE, (b + 1) * BLOCK_SIZE), unit.rope)
        Ks.append(Kh)
        Vs.append(Vh)
    Kw = np.asarray(unit.win_K, dtype=np.float64).reshape(-1, d)
    if unit.rope is not None:
        Kw = apply_rope(Kw, nb * BLOCK_SIZE + np.arange(Kw.shape[0]), unit.rope)
    Ks.append(Kw)
    Vs.append(np.asarray(unit.win_V, dtype=np.float64).reshape(-1, d))
    Kall = np.concatenate(Ks)
    Vall = np.concatenate(Vs)
    if Kall.shape[0] == 0:
        raise ValueError("nothing to attend: no routed block and an empty window")
    o, lse = softmax_attention(q, Kall, Vall)
    return {"o": o, "lse": lse, "idx": idx, "bounds": bounds}


# ---------------------------------------------------------------------------
# decode: factored form (low-rank scoring, low-rank value, split LSE merge)
# ---------------------------------------------------------------------------

def lse_merge(parts: list) -> tuple[np.ndarray, np.ndarray]:
    """Flash-style log-sum-exp merge ([DKV-Z]; [README Core] "Flash-Style LSE
    Combine").  Each part is (m [G], l [G], acc [G, d]) with
    l = sum exp(s - m) and acc = sum exp(s - m) v over that part's tokens:
        m* = max_j m_j,  l* = sum_j l_j e^{m_j - m*},
        o  = sum_j acc_j e^{m_j - m*} / l*,  lse = m* + log l*.
    """
    ms = np.stack([p[0] for p in parts])                     # [P, G]
    mstar = ms.max(axis=0)
    w = np.exp(ms - mstar[None, :])
    lstar = sum(wj * p[1] for wj, p in zip(w, parts))
    acc = sum(wj[:, None] * p[2] for wj, p in zip(w, parts))
    return acc / lstar[:, None], mstar + np.log(lstar)


def _part(s: np.ndarray, V: np.ndarray) -> tuple:
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    return m, e.sum(axis=1), e @ V


def block_partial(q: np.ndarray, blk: Block) -> tuple:
    """Partial (m, l, acc) of one routed block without materialising K.

    [README Core] "Low-Rank Space Query Scoring": with q~ = c q,
      z   = V_K q~                              (r numbers per query)
      s_0 = q~ . a_k                            (anchor)
      s_i = q~ . a_k + U_i . z                  (low-rank rows i not in S)
      s_j = q~ . k_j                            (exact residual rows j in S)
    and the value side
      acc = (sum_{low-rank incl. anchor} p) a_v + (sum p_i U_i) V_V + sum_{S} p_j v_j.
    """
    q = np.asarray(q, dtype=np.float64)
    qt = q / math.sqrt(q.shape[1])
    z = qt @ blk.V_K.T                                        # [G, r]
    base = qt @ blk.a_k                                       # [G]
    lowrank = np.ones(BLOCK_SIZE, dtype=bool)
    lowrank[blk.S] = False
    lr_rows = np.nonzero(lowrank[1:])[0]                      # indices into U (token - 1)
    s_lr = base[:, None] + z @ blk.U[lr_rows].T               # [G, n_lr]
    s_anchor = base[:, None]                                  # [G, 1]
    s_res = qt @ blk.K_res.T                                  # [G, R]
    s_all = np.concatenate([s_anchor, s_lr, s_res], axis=1)
    m = s_all.max(axis=1)
    p_anchor = np.exp(s_anchor - m[:, None])
    p_lr = np.exp(s_lr - m[:, None])
    p_res = np.exp(s_res - m[:, None])
    pa = p_anchor[:, 0] + p_lr.sum(axis=1)
    w = p_lr @ blk.U[lr_rows]                                 # [G, r]
    acc = pa[:, None] * blk.a_v[None, :] + w @ blk.V_V + p_res @ blk.V_res
    l = pa + p_res.sum(axis=1)
    return m, l, acc


def decode_unit_factored(q: np.ndarray, unit: Unit, top_k: int, window_chunk: int = 256) -> dict:
    """Same result as ``decode_unit`` through the factored steps: route, one
    partial per routed block (``block_partial``), exact window partials in
    chunks, then the split log-sum-exp merge."""
    if unit.rope is not None:
        # the scorer shares z = V_K q over a block's tokens, which needs one frame for all
        # of them ([README Knobs] DKV_ROTATED_POOL: the low-rank scorer refuses un-rotated keys)
        raise ValueError("the factored low-rank scorer needs a rotated pool")
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[1]
    qt = q / math.sqrt(d)
    nb = len(unit.blocks)
    if nb:
        bounds = router_bounds(q, np.stack([b.kmin for b in unit.blocks]), np.stack([b.kmax for b in unit.blocks]))
        idx = route(bounds, top_k)
    else:
        bounds, idx = np.zeros(0), np.zeros(0, dtype=np.int64)
    parts = [block_partial(q, unit.blocks[b]) for b in idx]
    W = unit.win_K.shape[0]
    for t0 in range(0, W, window_chunk):
        Kc = np.asarray(unit.win_K[t0:t0 + window_chunk], dtype=np.float64)
        Vc = np.asarray(unit.win_V[t0:t0 + window_chunk], dtype=np.float64)
        parts.append(_part(qt @ Kc.T, Vc))
    o, lse = lse_merge(parts)
    return {"o": o, "lse": lse, "idx": idx, "bounds": bounds}


# ---------------------------------------------------------------------------
# group-quantised residual rows
# ---------------------------------------------------------------------------

RESIDUAL_QUANT_GROUP = 64  # [README Innov] "asymmetric group quantization (group_size=64, ...)"


def quantize_groups(X: np.ndarray, bits: int, group: int = RESIDUAL_QUANT_GROUP):
    """Asymmetric group quantisation of the rows of X ([README Innov] "Physical
    4-Bit Group-Quantized Residual Buffers"; [README Knobs] DKV_RESIDUAL_QUANT,
    DKV_RESIDUAL_QUANT_GROUP_SIZE, DKV_RESIDUAL_QUANT_BITS).

    Every row is cut into groups of ``group`` consecutive channels.  Per group:
    bias = the group's minimum and scale = (maximum - minimum) / (2^bits - 1),
    both kept in fp16 (the pages' "half-precision scale and bias"); each value's
    code is the nearest integer to (x - bias) / scale, clamped to
    [0, 2^bits - 1]; a group whose fp16 scale is 0 has every code 0.  The code
    is an integer decision, taken in fp32 (the difference, the division and the
    range of the group are fp32 operations on the fp16 values; the rounding goes
    to the nearest integer, ties to even).

    X holds fp16 values (any float dtype).  Returns codes uint8 [n, d] and the
    fp16 scale and bias [n, d / group].
    """
    X = np.asarray(X, dtype=np.float32)  # exact for fp16 values
    n, d = X.shape
    if d % group:
        raise ValueError("head_dim must be a multiple of the group size")
    Xg = X.reshape(n, d // group, group)
    lo = Xg.min(axis=2)
    hi = Xg.max(axis=2)
    levels = np.float32(2 ** bits - 1)
    scale = ((hi - lo) / levels).astype(np.float16)
    bias = lo.astype(np.float16)  # exact: the minimum is one of the fp16 values
    s = scale.astype(np.float32)[:, :, None]
    b = bias.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.rint((Xg - b) / s)
    q = np.where(s == 0, 0.0, q)
    q = np.clip(q, 0, 2 ** bits - 1)
    return q.reshape(n, d).astype(np.uint8), scale, bias


def dequantize_groups(codes: np.ndarray, scale: np.ndarray, bias: np.ndarray,
                      group: int = RESIDUAL_QUANT_GROUP) -> np.ndarray:
    """x_hat = scale * code + bias per group of ``group`` channels, from the stored
    fp16 scale and bias, rounded once to fp16: [README Innov] dequantises the
    routed blocks "into transient scratchpads" for the attention, whose operands
    are fp16.  (scale * code + bias is exact in fp64, so the one rounding is the
    fp16 one.)  Returned as float64."""
    codes = np.asarray(codes, dtype=np.float64)
    n, d = codes.shape
    s = np.asarray(scale, dtype=np.float64)
    b = np.asarray(bias, dtype=np.float64)
    x = (codes.reshape(n, d // group, group) * s[:, :, None] + b[:, :, None]).reshape(n, d)
    return x.astype(np.float16).astype(np.float64)


def quantize_block_residuals(blk: Block, bits: int) -> Block:
    """The block as the decode reads it when its exact residual rows are stored
    group-quantised ([README Innov]: "only the gathered top-K routed blocks are
    dequantized ... during decode attention"): K_res and V_res are replaced by
    the dequantised (fp16) images of their own quantisation, each row on its own
    (keys and values separately); positions and every other part stay as they are."""
    if blk.S.size == 0:
        return dataclasses.replace(blk)
    Kq = dequantize_groups(*quantize_groups(blk.K_res, bits))
    Vq = dequantize_groups(*quantize_groups(blk.V_res, bits))
    return dataclasses.replace(blk, K_res=Kq, V_res=Vq)


def quant_residual_row_bytes(d: int, bits: int, group: int = RESIDUAL_QUANT_GROUP) -> int:
    """Bytes of one group-quantised residual row (a key or a value): d codes of
    ``bits`` bits packed in 32-bit words, plus an fp16 scale and an fp16 bias
    per group of ``group`` channels ([README Innov]: "head_dim * bits // 32 = 16
    words for D=128 alongside half-precision scale and bias vectors (8 bytes)")."""
    return d * bits // 32 * 4 + (d // group) * 4


# ---------------------------------------------------------------------------
# block-sparse prefill
# ---------------------------------------------------------------------------

def prefill_routes(Q: np.ndarray, K: np.ndarray, top_k: int) -> list:
    """Blocks each query block attends beside its own, for one unit ([DKV-Z]:
    "Prefill uses training-free block-sparse attention, so its cost grows
    sub-quadratically"; [README Core] "Sub-Quadratic Prefill": O(L^2) down to
    O(L * K)).  Q [G, T, d] are the GQA group's queries, K [T, d] the exact keys.

    Query block i (tokens 256 i .. 256 i + 255, the last one possibly shorter)
    scores every earlier key block j < i with the key-box bound of the decode
    router, taken with the block's mean query: qbar_i = mean over the block's
    tokens and the group's heads of c q, c = 1/sqrt(d), and
        bound_ij = sum_d max(qbar_id kmax_jd, qbar_id kmin_jd)
    over the channel extremes of block j's 256 keys; it keeps the top_k blocks
    by (bound desc, j asc), every earlier block when top_k is 0 or >= i.
    Returns, per query block, (routed blocks ascending, bounds [i]).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    G, T, d = Q.shape
    nb = -(-T // BLOCK_SIZE)
    out = []
    for i in range(nb):
        t0, t1 = i * BLOCK_SIZE, min(T, (i + 1) * BLOCK_SIZE)
        qbar = (Q[:, t0:t1, :] / math.sqrt(d)).mean(axis=(0, 1))
        bounds = np.array([np.maximum(qbar * K[j * BLOCK_SIZE:(j + 1) * BLOCK_SIZE].max(axis=0),
                                      qbar * K[j * BLOCK_SIZE:(j + 1) * BLOCK_SIZE].min(axis=0)).sum()
                           for j in range(i)])
        k = i if (top_k == 0 or top_k >= i) else int(top_k)
        order = sorted(range(i), key=lambda j: (-float(bounds[j]), j))[:k]
        out.append((np.array(sorted(order), dtype=np.int64), bounds))
    return out


def prefill_unit(Q: np.ndarray, K: np.ndarray, V: np.ndarray, top_k: int) -> dict:
    """Block-sparse prefill attention of one unit, by definition: the query at
    token t of query block i attends the keys of its own block up to t (causal)
    and every key of the blocks ``prefill_routes`` gives block i; one softmax of
    c q . k over that set.  Returns o [G, T, d], lse [G, T] and the routes."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    G, T, d = Q.shape
    routes = prefill_routes(Q, K, top_k)
    o = np.zeros((G, T, d))
    lse = np.zeros((G, T))
    for i, (idx, _) in enumerate(routes):
        t0, t1 = i * BLOCK_SIZE, min(T, (i + 1) * BLOCK_SIZE)
        keys = np.concatenate([np.arange(j * BLOCK_SIZE, (j + 1) * BLOCK_SIZE) for j in idx] +
                              [np.arange(t0, t1)]).astype(np.int64)
        s = np.einsum("gtd,kd->gtk", Q[:, t0:t1, :], K[keys]) / math.sqrt(d)
        own = keys >= t0
        causal = keys[None, :] > np.arange(t0, t1)[:, None]  # a key after the query
        s = np.where((own[None, :] & causal)[None, :, :], -np.inf, s)
        m = s.max(axis=2, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=2, keepdims=True)
        o[:, t0:t1, :] = np.einsum("gtk,kd->gtd", e, V[keys]) / l
        lse[:, t0:t1] = (m + np.log(l))[:, :, 0]
    return {"o": o, "lse": lse, "routes": [r for r, _ in routes], "bounds": [b for _, b in routes]}


def prefill_pairs(T: int, top_k: int) -> int:
    """(query, key) pairs block-sparse prefill scores for one query head: per query
    block its own causal triangle plus 256 keys of each routed earlier block; the
    cost the pages call O(L * K)."""
    nb = -(-T // BLOCK_SIZE)
    pairs = 0
    for i in range(nb):
        n = min(T, (i + 1) * BLOCK_SIZE) - i * BLOCK_SIZE
        k = i if (top_k == 0 or top_k >= i) else top_k
        pairs += n * (n + 1) // 2 + n * k * BLOCK_SIZE
    return pairs


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------

def pages_block_bytes(d: int, u_rank: int, R: int, elem_bytes: int = 4,
                      basis_bytes: int | None = None, meta_bytes: int = 8) -> dict:
    """Per-block byte accounting in the layout of [README Bench] table
    "Per-Block Memory Breakdown (B_s = 256 Tokens)": U coefficients [255, r],
    V_K/V_V bases [2, r, d], anchors [2, d], key min/max [2, d], scalars,
    exact residuals [R, 2, d]; the dense block is [256, 2, d] x 2.
    ``basis_bytes`` overrides the V_K/V_V row (the table prints a figure that
    does not follow from its own shape)."""
    u = (BLOCK_SIZE - 1) * u_rank * elem_bytes
    basis = basis_bytes if basis_bytes is not None else 2 * u_rank * d * elem_bytes
    anchors = 2 * d * elem_bytes
    minmax = 2 * d * elem_bytes
    core = u + basis + anchors + minmax + meta_bytes
    res = R * 2 * d * elem_bytes
    dense = BLOCK_SIZE * 2 * d * elem_bytes
    return {"U": u, "basis": basis, "anchors": anchors, "minmax": minmax, "meta": meta_bytes,
            "core": core, "residual": res, "block": core + res, "dense": dense,
            "ratio": dense / (core + res)}


def residual_row_bytes(d: int, elem_bytes: int = 2) -> int:
    """One exact residual token = its key and value rows."""
    return 2 * d * elem_bytes


def dense_kv_bytes(context: int, d: int, n_layers: int, n_kv_heads: int, elem_bytes: int = 2) -> int:
    """Uncompressed K and V of every layer and KV head."""
    return context * 2 * d * elem_bytes * n_layers * n_kv_heads
