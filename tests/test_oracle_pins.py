"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute itself:
a textbook routine it must reduce to (dense softmax attention via scipy), a
closed form, an invariant, brute force on tiny inputs, or the numbers the
pages print (tests/golden).  A plausible slip in the oracle (dropped anchor,
wrong sign of a delta, transposed basis, residual rows not substituted,
wrong tie order, a missing LSE rescale) fails at least one of them;
tests/test_oracle_mutants.py plants 58 such slips and checks exactly that.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import dkv_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = O.BLOCK_SIZE


def _kv(rng, n_tok, d, lat=3, outliers=2):
    """Small structured K/V: mean + low-rank latent + noise + a few outlier rows."""
    mu = rng.standard_normal((2, d))
    L = rng.standard_normal((2, n_tok, lat))
    Wm = rng.standard_normal((2, lat, d)) / math.sqrt(lat)
    X = mu[:, None, :] + L @ Wm + 0.05 * rng.standard_normal((2, n_tok, d))
    rows = rng.choice(n_tok, size=outliers, replace=False)
    X[:, rows, :] *= 8.0
    return X[0], X[1]


def _dense(q, K, V):
    """Textbook softmax attention via scipy (the routine the method must reduce to)."""
    s = (q / math.sqrt(q.shape[1])) @ K.T
    return scipy.special.softmax(s, axis=1) @ V, scipy.special.logsumexp(s, axis=1)


# ----------------------------------------------------------------- P1, P2

@pytest.mark.parametrize("d,nb,W", [(16, 3, 40), (8, 2, 0), (32, 1, 7)])
def test_full_rank_all_routed_equals_dense(d, nb, W):
    """r = rank(X) = min(255, 2d), R = 0, K = NB: the cache is lossless and the
    decode is dense softmax attention over the exact K, V."""
    rng = np.random.default_rng(10 + d)
    K, V = _kv(rng, nb * BS + W, d)
    q = rng.standard_normal((3, d))
    unit = O.compress_unit(K, V, nb, rank=min(255, 2 * d), n_residual=0)
    for top_k in (0, nb, nb + 5):
        got = O.decode_unit(q, unit, top_k)
        o, lse = _dense(q, K, V)
        np.testing.assert_allclose(got["o"], o, atol=1e-11, rtol=0)
        np.testing.assert_allclose(got["lse"], lse, atol=1e-11, rtol=0)


@pytest.mark.parametrize("rank", [0, 1, 5])
def test_all_residual_rows_is_exact(rank):
    """R = 255 keeps every non-anchor row exact: dense attention for any r."""
    rng = np.random.default_rng(rank)
    d, nb, W = 16, 2, 33
    K, V = _kv(rng, nb * BS + W, d)
    q = rng.standard_normal((2, d))
    unit = O.compress_unit(K, V, nb, rank=rank, n_residual=255)
    got = O.decode_unit(q, unit, 0)
    o, lse = _dense(q, K, V)
    np.testing.assert_allclose(got["o"], o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(got["lse"], lse, atol=1e-12, rtol=0)
    f = O.decode_unit_factored(q, unit, 0)
    np.testing.assert_allclose(f["o"], o, atol=1e-12, rtol=0)


# ----------------------------------------------------------------- P3

def test_split_lse_merge_equals_single_softmax():
    """Any partition of the token set merged by log-sum-exp = one softmax."""
    rng = np.random.default_rng(3)
    G, n, d = 4, 777, 12
    q = rng.standard_normal((G, d)) * 3.0
    K = rng.standard_normal((n, d)) * 2.0
    V = rng.standard_normal((n, d))
    s = (q / math.sqrt(d)) @ K.T
    o_ref = scipy.special.softmax(s, axis=1) @ V
    lse_ref = scipy.special.logsumexp(s, axis=1)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, n), size=trial + 1, replace=False))
        parts = []
        for a, b in zip(np.r_[0, cuts], np.r_[cuts, n]):
            sp = s[:, a:b]
            m = sp.max(axis=1)
            e = np.exp(sp - m[:, None])
            parts.append((m, e.sum(axis=1), e @ V[a:b]))
        o, lse = O.lse_merge(parts)
        np.testing.assert_allclose(o, o_ref, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse, lse_ref, atol=1e-12, rtol=0)


def test_lse_merge_single_part_and_order_invariance():
    rng = np.random.default_rng(4)
    parts = [(rng.standard_normal(2) * 5, rng.random(2) + 0.1, rng.standard_normal((2, 3))) for _ in range(4)]
    o1, l1 = O.lse_merge(parts)
    o2, l2 = O.lse_merge(parts[::-1])
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)
    m, l, acc = parts[0]
    o, lse = O.lse_merge([parts[0]])
    np.testing.assert_allclose(o, acc / l[:, None], atol=1e-15)
    np.testing.assert_allclose(lse, m + np.log(l), atol=1e-15)


# ----------------------------------------------------------------- P4

@pytest.mark.parametrize("rank,R", [(3, 10), (8, 0), (0, 4), (12, 100)])
def test_factored_equals_materialised(rank, R):
    """Low-rank scoring q.a_k + U_i.z and value (sum p) a_v + (sum p U) V_V equal
    attention over the reconstructed tokens, per block and per unit."""
    rng = np.random.default_rng(40 + rank + R)
    d, nb, W = 16, 4, 70
    K, V = _kv(rng, nb * BS + W, d)
    q = rng.standard_normal((6, d)) * 2
    unit = O.compress_unit(K, V, nb, rank, R)
    for blk in unit.blocks:
        m, l, acc = O.block_partial(q, blk)
        Kh, Vh = O.reconstruct_block(blk)
        o_ref, lse_ref = _dense(q, Kh, Vh)
        np.testing.assert_allclose(acc / l[:, None], o_ref, atol=1e-12, rtol=0)
        np.testing.assert_allclose(m + np.log(l), lse_ref, atol=1e-12, rtol=0)
    for top_k in (1, 2, 0):
        a = O.decode_unit(q, unit, top_k)
        b = O.decode_unit_factored(q, unit, top_k, window_chunk=32)
        np.testing.assert_array_equal(a["idx"], b["idx"])
        np.testing.assert_allclose(a["o"], b["o"], atol=1e-12, rtol=0)
        np.testing.assert_allclose(a["lse"], b["lse"], atol=1e-12, rtol=0)


# ----------------------------------------------------------------- P5

def test_router_bound_is_an_upper_bound_on_every_key():
    rng = np.random.default_rng(5)
    d = 24
    for _ in range(20):
        keys = rng.standard_normal((BS, d)) * rng.uniform(0.1, 5)
        q = rng.standard_normal((5, d))
        b = O.router_bounds(q, keys.min(0)[None], keys.max(0)[None])[0]
        qbar = (q / math.sqrt(d)).mean(0)
        assert b >= (keys @ qbar).max() - 1e-12
        # the bound is attained when the block's box corners are keys
        corner = np.where(qbar >= 0, keys.max(0), keys.min(0))
        np.testing.assert_allclose(b, corner @ qbar, atol=1e-12)


def test_route_brute_force_and_ties():
    rng = np.random.default_rng(6)
    for nb in (1, 2, 5, 7):
        for k in range(0, nb + 2):
            bounds = rng.integers(0, 4, size=nb).astype(float)  # many ties
            got = O.route(bounds, k)
            kk = nb if (k == 0 or k >= nb) else k
            # brute force: best subset by sum of bounds, ties broken toward lower indices
            best = None
            for sub in itertools.combinations(range(nb), kk):
                key = (-sum(bounds[list(sub)]), list(sub))
                if best is None or key < best[0]:
                    best = (key, sub)
            assert list(got) == sorted(best[1])
    # explicit tie order: equal bounds keep the lower block index
    assert list(O.route(np.array([1.0, 2.0, 2.0, 2.0]), 2)) == [1, 2]
    assert list(O.route(np.array([5.0, 1.0, 5.0]), 1)) == [0]


def test_all_routed_makes_routing_irrelevant():
    rng = np.random.default_rng(7)
    d, nb = 16, 5
    K, V = _kv(rng, nb * BS + 20, d)
    unit = O.compress_unit(K, V, nb, 4, 6)
    q = rng.standard_normal((2, d))
    a = O.decode_unit(q, unit, 0)
    # permute the blocks: attending all of them gives the same answer
    perm = O.Unit(blocks=unit.blocks[::-1], win_K=unit.win_K, win_V=unit.win_V)
    b = O.decode_unit(q, perm, nb)
    np.testing.assert_allclose(a["o"], b["o"], atol=1e-13)
    assert list(a["idx"]) == list(range(nb))


def test_routing_picks_blocks_with_the_largest_bound():
    """A block whose keys align with the query must be routed."""
    rng = np.random.default_rng(8)
    d, nb = 16, 6
    K, V = _kv(rng, nb * BS, d)
    q = rng.standard_normal((3, d))
    qbar = q.mean(0)
    K[3 * BS + 17] = 40 * qbar / np.linalg.norm(qbar)  # one very aligned key in block 3
    unit = O.compress_unit(K, V, nb, 4, 4)
    assert 3 in O.decode_unit(q, unit, 1)["idx"]


# ----------------------------------------------------------------- P6

def test_rank_zero_closed_form():
    """r = 0: every low-rank row is the anchor, so a block's partial is
    (n_lr e^{s0}) a_v + sum_S e^{s_j} v_j over l = n_lr e^{s0} + sum_S e^{s_j}."""
    rng = np.random.default_rng(9)
    d = 16
    K, V = _kv(rng, BS, d)
    blk = O.compress_block(K, V, rank=0, n_residual=7)
    q = rng.standard_normal((2, d))
    qt = q / math.sqrt(d)
    s0 = qt @ K[0]
    sres = qt @ K[blk.S].T
    n_lr = BS - len(blk.S)
    num = (n_lr * np.exp(s0))[:, None] * V[0][None] + np.exp(sres) @ V[blk.S]
    den = n_lr * np.exp(s0) + np.exp(sres).sum(1)
    m, l, acc = O.block_partial(q, blk)
    np.testing.assert_allclose(acc / l[:, None], num / den[:, None], atol=1e-12)
    np.testing.assert_allclose(m + np.log(l), np.log(den), atol=1e-12)


# ----------------------------------------------------------------- P7, P8 (the pages' printed numbers)

def test_per_block_bytes_match_the_pages_table():
    g = json.load(open(os.path.join(GOLDEN, "per_block_bytes.json")))
    rows = g["rows"]
    for R in (128, 64):
        acc = O.pages_block_bytes(g["head_dim"], g["u_rank"], R, elem_bytes=g["elem_bytes"],
                                  basis_bytes=g["basis_bytes_as_printed"])
        assert acc["U"] == rows["U"]
        assert acc["anchors"] == rows["anchors"]
        assert acc["minmax"] == rows["minmax"]
        assert acc["core"] == rows["core"]
        assert acc["residual"] == rows[f"residual_R{R}"]
        assert acc["block"] == rows[f"block_R{R}"]
        assert acc["dense"] == rows["dense"]
        assert round(acc["ratio"], 2) == g["ratios"][f"R{R}"]
    # the printed basis row is not its own shape at 4-byte elements (a garble, passed through)
    assert O.pages_block_bytes(128, 16, 0)["basis"] == rows["basis"] // 2


def test_residual_sweep_store_sizes_match_fp16_rows():
    """The store grows by one fp16 K+V row per residual slot per block, and the
    3.80x ratio is dense fp16 KV at 16k over the R=8 store."""
    g = json.load(open(os.path.join(GOLDEN, "residual_sweep_16k.json")))
    R, store = np.array(g["R"], float), np.array(g["store_gb"]) * 1e9
    slope = np.polyfit(R, store, 1)[0]
    per_row = O.residual_row_bytes(g["head_dim"]) * g["n_blocks"] * g["n_layers"] * g["n_kv_heads"]
    assert g["n_blocks"] == (g["context"] - 512) // BS
    assert abs(slope / per_row - 1) < 0.01
    dense = O.dense_kv_bytes(g["context"], g["head_dim"], g["n_layers"], g["n_kv_heads"])
    for s, ratio in zip(store, g["ratio_vs_dense"]):
        assert abs(dense / s - ratio) / ratio < 0.02


# ----------------------------------------------------------------- P9 and compression invariants

@pytest.mark.parametrize("rank", [1, 4, 9, 20])
def test_eckart_young(rank):
    """Truncation error = sum of the discarded squared singular values, taken
    from an independent symmetric eigen-solve of X^T X; the joint basis rows
    are orthonormal; no random rank-r factorisation does better."""
    rng = np.random.default_rng(90 + rank)
    d = 16
    K, V = _kv(rng, BS, d, lat=5)
    blk = O.compress_block(K, V, rank, 0)
    X = np.concatenate([K[1:] - K[0], V[1:] - V[0]], axis=1)
    Wr = np.concatenate([blk.V_K, blk.V_V], axis=1)
    err = ((X - blk.U @ Wr) ** 2).sum()
    ev = np.sort(np.linalg.eigvalsh(X.T @ X))[::-1]
    np.testing.assert_allclose(err, ev[rank:].sum(), rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(Wr @ Wr.T, np.eye(rank), atol=1e-12)
    for _ in range(5):
        Q, _ = np.linalg.qr(rng.standard_normal((2 * d, rank)))
        assert ((X - (X @ Q) @ Q.T) ** 2).sum() >= err - 1e-9


def test_anchor_is_first_token_and_deltas_are_to_it():
    rng = np.random.default_rng(11)
    d = 8
    K, V = _kv(rng, BS, d)
    blk = O.compress_block(K, V, rank=2 * d, n_residual=0)
    np.testing.assert_array_equal(blk.a_k, K[0])
    np.testing.assert_array_equal(blk.a_v, V[0])
    Kh, Vh = O.reconstruct_block(blk)
    np.testing.assert_allclose(Kh, K, atol=1e-11)
    np.testing.assert_allclose(Vh, V, atol=1e-11)
    # a constant shift of the whole block only moves the anchor: the deltas are unchanged
    b1 = O.compress_block(K, V, rank=3, n_residual=0)
    b2 = O.compress_block(K + 3.0, V - 2.0, rank=3, n_residual=0)
    np.testing.assert_allclose(b2.a_k, K[0] + 3.0)
    np.testing.assert_allclose(b2.U @ b2.V_K, b1.U @ b1.V_K, atol=1e-9)
    np.testing.assert_allclose(b2.U @ b2.V_V, b1.U @ b1.V_V, atol=1e-9)


def test_residuals_pick_the_worst_reconstructed_rows():
    """A row far off the low-rank structure is kept exact; the kept rows are
    exactly the R largest key errors, ties to the lower position."""
    rng = np.random.default_rng(12)
    d = 16
    K, V = _kv(rng, BS, d, lat=2, outliers=0)
    K[77] += rng.standard_normal(d) * 3.0   # off-structure key
    K[200] += rng.standard_normal(d) * 2.0
    blk = O.compress_block(K, V, rank=4, n_residual=2)   # rank 4 spans the K and V latents
    assert list(blk.S) == [77, 200]
    np.testing.assert_array_equal(blk.K_res, K[[77, 200]])
    np.testing.assert_array_equal(blk.V_res, V[[77, 200]])
    # brute-force the selection from the reconstruction
    Kh_lr = K[0] + blk.U @ blk.V_K
    err = np.linalg.norm(K[1:] - Kh_lr, axis=1)
    for R in (0, 1, 5, 30, 255, 300):
        S = O.select_residuals(err, R)
        assert len(S) == min(R, 255)
        if 0 < len(S) < 255:
            kept = err[S - 1]
            dropped = np.delete(err, S - 1)
            assert kept.min() >= dropped.max()
    # ties go to the lower token
    assert list(O.select_residuals(np.array([1.0, 3.0, 3.0, 3.0, 0.5]), 2)) == [2, 3]


def test_router_minmax_are_channel_extremes():
    rng = np.random.default_rng(13)
    K, V = _kv(rng, BS, 8)
    blk = O.compress_block(K, V, 2, 3)
    np.testing.assert_array_equal(blk.kmin, K.min(0))
    np.testing.assert_array_equal(blk.kmax, K.max(0))


# ----------------------------------------------------------------- P10: brute force, scalar loops

def test_tiny_brute_force_loops():
    """Scalar Python loops over tokens and channels agree with the vectorised oracle."""
    rng = np.random.default_rng(14)
    d, nb, W, G, r, R, top_k = 4, 3, 9, 2, 2, 5, 2
    K, V = _kv(rng, nb * BS + W, d, lat=2, outliers=1)
    q = rng.standard_normal((G, d))
    unit = O.compress_unit(K, V, nb, r, R)
    c = 1.0 / math.sqrt(d)
    # routing by loops
    bounds = []
    for blk in unit.blocks:
        tot = 0.0
        for j in range(d):
            qb = sum(c * q[g][j] for g in range(G)) / G
            tot += max(qb * blk.kmax[j], qb * blk.kmin[j])
        bounds.append(tot)
    order = sorted(range(nb), key=lambda b: (-bounds[b], b))[:top_k]
    routed = sorted(order)
    # token list by loops
    toks = []
    for b in routed:
        blk = unit.blocks[b]
        S = set(int(x) for x in blk.S)
        for i in range(BS):
            if i == 0:
                k, v = list(blk.a_k), list(blk.a_v)
            elif i in S:
                j = list(blk.S).index(i)
                k, v = list(blk.K_res[j]), list(blk.V_res[j])
            else:
                k = [blk.a_k[t] + sum(blk.U[i - 1][a] * blk.V_K[a][t] for a in range(r)) for t in range(d)]
                v = [blk.a_v[t] + sum(blk.U[i - 1][a] * blk.V_V[a][t] for a in range(r)) for t in range(d)]
            toks.append((k, v))
    for t in range(W):
        toks.append((list(unit.win_K[t]), list(unit.win_V[t])))
    got = O.decode_unit(q, unit, top_k)
    assert list(got["idx"]) == routed
    for g in range(G):
        s = [c * sum(q[g][t] * k[t] for t in range(d)) for k, _ in toks]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        den = sum(e)
        o = [sum(e[n] * toks[n][1][t] for n in range(len(toks))) / den for t in range(d)]
        np.testing.assert_allclose(got["o"][g], o, atol=1e-12)
        assert abs(got["lse"][g] - (m + math.log(den))) < 1e-12


def test_window_only_and_empty_inputs():
    rng = np.random.default_rng(15)
    d = 8
    K, V = _kv(rng, 50, d)
    q = rng.standard_normal((1, d))
    unit = O.compress_unit(K, V, 0, 4, 4)
    got = O.decode_unit(q, unit, 3)
    o, lse = _dense(q, K, V)
    np.testing.assert_allclose(got["o"], o, atol=1e-13)
    assert got["idx"].size == 0
    with pytest.raises(ValueError):
        O.decode_unit(q, O.compress_unit(K[:0], V[:0], 0, 4, 4), 1)
    with pytest.raises(ValueError):
        O.route(np.zeros(3), -1)


@pytest.mark.parametrize("cap,T0,chunks", [(300, 0, [1, 2, 297, 1, 255, 1, 400, 3]), (256, 100, [156, 1, 600]),
                                           (512, 700, [5, 1, 1, 300, 200])])
def test_streaming_append_equals_batch_compression(cap, T0, chunks):
    """Appending tokens in arbitrary pieces leaves the same state as compressing
    the whole sequence at once: the block count follows from the window rule
    (no block until the window is full; then one per 256 tokens past the
    capacity) and every block is the batch compression of the same 256 tokens."""
    rng = np.random.default_rng(cap + T0)
    d, rank, R = 16, 3, 5
    T = T0 + sum(chunks)
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    nb0 = 0 if T0 <= cap else -(-(T0 - cap) // 256)
    unit = O.compress_unit(K[:T0], V[:T0], nb0, rank, R)
    t = T0
    for n in chunks:
        unit = O.append_tokens(unit, K[t:t + n], V[t:t + n], cap, rank, R)
        t += n
        nb = 0 if t <= cap else -(-(t - cap) // 256)
        assert len(unit.blocks) == nb and len(unit.win_K) == t - 256 * nb
        assert cap - 256 < len(unit.win_K) <= cap or nb == 0
    ref = O.compress_unit(K, V, len(unit.blocks), rank, R)
    np.testing.assert_array_equal(unit.win_K, ref.win_K)
    np.testing.assert_array_equal(unit.win_V, ref.win_V)
    for a, b in zip(unit.blocks, ref.blocks):
        np.testing.assert_array_equal(a.a_k, b.a_k)
        np.testing.assert_array_equal(a.U, b.U)
        np.testing.assert_array_equal(a.V_K, b.V_K)
        np.testing.assert_array_equal(a.S, b.S)
        np.testing.assert_array_equal(a.kmax, b.kmax)


def test_streaming_append_needs_a_full_block_of_window():
    unit = O.compress_unit(np.zeros((100, 8)), np.zeros((100, 8)), 0, 2, 1)
    with pytest.raises(ValueError):
        O.append_tokens(unit, np.ones((1, 8)), np.ones((1, 8)), 100, 2, 1)


# ----------------------------------------------------------------- group-quantised residuals

@pytest.mark.parametrize("bits", [8, 4])
def test_quantization_recovers_values_on_its_own_grid(bits):
    """Values that sit exactly on a group's grid (bias + scale * code, with the
    lowest and highest codes present) quantise to exactly that scale, bias and
    codes, and dequantise back without error."""
    rng = np.random.default_rng(70 + bits)
    top = 2 ** bits - 1
    n, d, g = 6, 128, O.RESIDUAL_QUANT_GROUP
    scale = 2.0 ** rng.integers(-8, -2, size=(n, d // g))
    bias = rng.integers(-64, 64, size=(n, d // g)) * scale
    codes = rng.integers(0, top + 1, size=(n, d))
    codes[:, 0::g] = 0
    codes[:, 1::g] = top
    X = (codes.reshape(n, d // g, g) * scale[:, :, None] + bias[:, :, None]).reshape(n, d)
    assert np.array_equal(X.astype(np.float16).astype(np.float64), X)  # exact fp16 values
    q, s, b = O.quantize_groups(X, bits)
    assert np.array_equal(q, codes)
    assert np.array_equal(s.astype(np.float64), scale) and np.array_equal(b.astype(np.float64), bias)
    assert np.array_equal(O.dequantize_groups(q, s, b), X)


@pytest.mark.parametrize("bits", [8, 4])
def test_quantization_picks_the_nearest_code(bits):
    """Brute force over every code: the chosen code's reconstruction is the
    nearest to the value on the group's stored fp16 grid (within the fp32
    rounding of the division at exact midpoints)."""
    rng = np.random.default_rng(80 + bits)
    X = (rng.standard_normal((8, 128)) * rng.uniform(0.1, 20, size=(8, 1))).astype(np.float16).astype(np.float64)
    q, s, b = O.quantize_groups(X, bits)
    g = O.RESIDUAL_QUANT_GROUP
    grid = np.arange(2 ** bits, dtype=np.float64)
    for i in range(X.shape[0]):
        for j in range(X.shape[1]):
            sv, bv = float(s[i, j // g]), float(b[i, j // g])
            err = np.abs(X[i, j] - (sv * grid + bv))
            assert err[q[i, j]] <= err.min() + 1e-6 * max(sv, 1e-30), (i, j, q[i, j], int(err.argmin()))


@pytest.mark.parametrize("bits", [8, 4])
def test_quantization_error_is_within_half_a_step(bits):
    """|x - x_hat| <= scale / 2, up to the fp16 rounding of the stored scale at the
    top of the group's range ((2^bits - 1) steps of at most 2^-11 scale each) and
    the fp16 rounding of the dequantised value (half an fp16 ulp, 2^-11 |x_hat|)."""
    rng = np.random.default_rng(90 + bits)
    X = (rng.standard_normal((64, 128)) * 4).astype(np.float16).astype(np.float64)
    X[3] *= 8.0  # an outlier row
    q, s, b = O.quantize_groups(X, bits)
    xr = O.dequantize_groups(q, s, b)
    g = O.RESIDUAL_QUANT_GROUP
    step = np.repeat(s.astype(np.float64), g, axis=1)
    rng_ = np.repeat((X.reshape(64, -1, g).max(2) - X.reshape(64, -1, g).min(2)), g, axis=1)
    assert (np.abs(X - xr) <= step / 2 + rng_ * 2.0 ** -10 + np.abs(xr) * 2.0 ** -11 + 1e-12).all()
    assert q.max() <= 2 ** bits - 1


def test_quantization_of_a_constant_group_is_exact():
    """A group whose values are all equal has scale 0, every code 0 and
    reconstructs exactly; the other group of the row is unaffected."""
    X = np.zeros((2, 128))
    X[0, :64] = 1.5
    X[0, 64:] = np.linspace(-2, 2, 64).astype(np.float16)
    X[1, :] = -3.25
    for bits in (8, 4):
        q, s, b = O.quantize_groups(X, bits)
        assert float(s[0, 0]) == 0.0 and (q[0, :64] == 0).all() and float(b[0, 0]) == 1.5
        assert (q[1] == 0).all()
        xr = O.dequantize_groups(q, s, b)
        assert np.array_equal(xr[0, :64], X[0, :64]) and np.array_equal(xr[1], X[1])
        assert float(s[0, 1]) > 0


def test_quantized_row_bytes_match_the_pages():
    """[README Innov] item 2: 16 words of codes plus 8 bytes of scale and bias per
    d128 int4 row; 3.56x (int4) and 1.9x (int8) against an fp16 row; R = 256 int4
    residuals in 44 % less memory than R = 128 fp16 ones (112.9 / 200.7 MB at 16k)."""
    gold = json.load(open(os.path.join(GOLDEN, "residual_quant.json")))
    d = gold["head_dim"]
    assert gold["group_size"] == O.RESIDUAL_QUANT_GROUP
    int4 = O.quant_residual_row_bytes(d, 4)
    int8 = O.quant_residual_row_bytes(d, 8)
    assert int4 == gold["int4_words_per_row"] * 4 + gold["scale_bias_bytes_per_row"]
    fp16 = O.residual_row_bytes(d) // 2  # one row (key or value) of fp16
    assert round(fp16 / int4, 2) == gold["compression_vs_fp16"]["int4"]
    assert round(fp16 / int8, 1) == gold["compression_vs_fp16"]["int8"]
    ratio = (256 * int4) / (128 * fp16)
    mb = gold["store_16k_mb"]
    assert abs(ratio - mb["int4_R256"] / mb["fp16_R128"]) < 5e-4
    assert round(100 * (1 - ratio)) == gold["less_memory_pct"]


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_residual_decode_brute_force(bits):
    """Decode over blocks whose residual rows are stored quantised equals a
    scalar-loop reconstruction: rows in S rebuilt element by element from their
    own codes, scale and bias (keys and values each from their own), each value
    rounded to fp16; every other row from the anchor and the low-rank factors."""
    rng = np.random.default_rng(100 + bits)
    d, nb, W, r, R = 64, 2, 20, 5, 9
    K, V = _kv(rng, nb * BS + W, d)
    K = K.astype(np.float16).astype(np.float64)
    V = V.astype(np.float16).astype(np.float64)
    q = rng.standard_normal((2, d))
    unit = O.compress_unit(K, V, nb, r, R)
    qunit = O.Unit(blocks=[O.quantize_block_residuals(b, bits) for b in unit.blocks], win_K=unit.win_K,
                   win_V=unit.win_V)
    got = O.decode_unit(q, qunit, 0)
    g = O.RESIDUAL_QUANT_GROUP
    Ks, Vs = [], []
    for blk in unit.blocks:
        kq, ks, kb = O.quantize_groups(blk.K_res, bits)
        vq, vs, vb = O.quantize_groups(blk.V_res, bits)
        for t in range(BS):
            krow, vrow = [], []
            for j in range(d):
                if t == 0:
                    kx, vx = blk.a_k[j], blk.a_v[j]
                elif t in list(blk.S):
                    i = list(blk.S).index(t)
                    kx = float(np.float16(float(ks[i, j // g]) * int(kq[i, j]) + float(kb[i, j // g])))
                    vx = float(np.float16(float(vs[i, j // g]) * int(vq[i, j]) + float(vb[i, j // g])))
                else:
                    kx = blk.a_k[j] + sum(blk.U[t - 1, k] * blk.V_K[k, j] for k in range(r))
                    vx = blk.a_v[j] + sum(blk.U[t - 1, k] * blk.V_V[k, j] for k in range(r))
                krow.append(kx)
                vrow.append(vx)
            Ks.append(krow)
            Vs.append(vrow)
    Ks = np.array(Ks + list(unit.win_K))
    Vs = np.array(Vs + list(unit.win_V))
    o, lse = _dense(q, Ks, Vs)
    np.testing.assert_allclose(got["o"], o, atol=1e-10, rtol=0)
    np.testing.assert_allclose(got["lse"], lse, atol=1e-10, rtol=0)
    assert np.abs(got["o"] - O.decode_unit(q, unit, 0)["o"]).max() > 0  # the quantisation is visible


# ----------------------------------------------------------------- block-sparse prefill

def _causal_dense(Q, K, V):
    """Textbook causal softmax attention via scipy: token t attends keys 0..t."""
    G, T, d = Q.shape
    s = np.einsum("gtd,kd->gtk", Q, K) / math.sqrt(d)
    s = np.where(np.triu(np.ones((T, T), bool), 1)[None], -np.inf, s)
    return scipy.special.softmax(s, axis=2) @ V, scipy.special.logsumexp(s, axis=2)


@pytest.mark.parametrize("T,top_k", [(700, 0), (700, 3), (512, 2), (256, 0), (37, 1), (1100, 50)])
def test_prefill_routing_every_block_is_dense_causal_attention(T, top_k):
    """top_k 0 or >= the number of earlier blocks: every query attends every key at
    or before it, i.e. dense causal softmax attention."""
    rng = np.random.default_rng(T + top_k)
    d = 16
    K, V = _kv(rng, T, d)
    Q = rng.standard_normal((3, T, d))
    got = O.prefill_unit(Q, K, V, top_k)
    o, lse = _causal_dense(Q, K, V)
    nb = -(-T // BS)
    if top_k == 0 or top_k >= nb - 1:
        np.testing.assert_allclose(got["o"], o, atol=1e-11, rtol=0)
        np.testing.assert_allclose(got["lse"], lse, atol=1e-11, rtol=0)
    else:  # the first top_k + 1 query blocks still see every earlier block
        t1 = (top_k + 1) * BS
        np.testing.assert_allclose(got["o"][:, :t1], o[:, :t1], atol=1e-11, rtol=0)


def test_prefill_brute_force_loops():
    """Scalar loops: the block-mean query, the bounds (max of the two products per
    channel over the block's own min and max), the ranking with ties to the lower
    block, each token's key set (own block causally, routed blocks whole) and its
    softmax.  Each block's first query is made atypical, so that routing on one
    token instead of the block mean would pick other blocks."""
    rng = np.random.default_rng(5)
    T, d, G, top_k = 6 * BS + 40, 8, 2, 2
    K, V = _kv(rng, T, d)
    Q = 0.3 * rng.standard_normal((G, T, d))
    for i in range(7):  # each block's queries lean one way, its first query the other way
        lean = 2.0 * rng.standard_normal(d)
        Q[:, i * BS:(i + 1) * BS, :] += lean
        Q[:, i * BS, :] = -3.0 * lean
    K[BS:2 * BS] = K[:BS]  # blocks 0 and 1 have the same box: a tie, to the lower block
    got = O.prefill_unit(Q, K, V, top_k)
    differs = False
    for i in range(7):
        t0, t1 = i * BS, min(T, (i + 1) * BS)
        qbar = [sum(Q[g, t, c] / math.sqrt(d) for g in range(G) for t in range(t0, t1)) / (G * (t1 - t0))
                for c in range(d)]
        bounds, first = [], []
        for j in range(i):
            lo = [min(K[t, c] for t in range(j * BS, (j + 1) * BS)) for c in range(d)]
            hi = [max(K[t, c] for t in range(j * BS, (j + 1) * BS)) for c in range(d)]
            bounds.append(sum(max(qbar[c] * lo[c], qbar[c] * hi[c]) for c in range(d)))
            q0 = [Q[0, t0, c] / math.sqrt(d) for c in range(d)]
            first.append(sum(max(q0[c] * lo[c], q0[c] * hi[c]) for c in range(d)))
        routed = sorted(sorted(range(i), key=lambda j: (-bounds[j], j))[:top_k]) if i > top_k else list(range(i))
        by_first = sorted(sorted(range(i), key=lambda j: (-first[j], j))[:top_k]) if i > top_k else list(range(i))
        differs |= routed != by_first
        assert list(got["routes"][i]) == routed
        for t in range(t0, t1, 61):
            keys = [k for j in routed for k in range(j * BS, (j + 1) * BS)] + list(range(t0, t + 1))
            for g in range(G):
                sc = [sum(Q[g, t, c] * K[k, c] for c in range(d)) / math.sqrt(d) for k in keys]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                o = [sum(e[n] * V[k, c] for n, k in enumerate(keys)) / sum(e) for c in range(d)]
                np.testing.assert_allclose(got["o"][g, t], o, atol=1e-10, rtol=0)
                assert abs(got["lse"][g, t] - (m + math.log(sum(e)))) < 1e-10
    assert differs, "the case does not tell the block mean from the first query"


def test_prefill_bound_is_an_upper_bound_on_every_key():
    rng = np.random.default_rng(6)
    T, d = 5 * BS, 32
    K, _ = _kv(rng, T, d)
    Q = rng.standard_normal((6, T, d))
    routes = O.prefill_routes(Q, K, 2)
    for i, (_, bounds) in enumerate(routes):
        qbar = (Q[:, i * BS:(i + 1) * BS] / math.sqrt(d)).mean(axis=(0, 1))
        for j in range(i):
            assert bounds[j] >= (K[j * BS:(j + 1) * BS] @ qbar).max() - 1e-12


def test_prefill_blockwise_merge_equals_the_single_softmax():
    """Per query block, a partial per attended key block (routed blocks whole, the own
    block causally) merged by the split log-sum-exp gives the one-softmax result."""
    rng = np.random.default_rng(7)
    T, d, top_k = 4 * BS + 100, 16, 2
    K, V = _kv(rng, T, d)
    Q = rng.standard_normal((2, T, d))
    got = O.prefill_unit(Q, K, V, top_k)
    for i, idx in enumerate(got["routes"]):
        t0, t1 = i * BS, min(T, (i + 1) * BS)
        for t in range(t0, t1, 29):
            parts = []
            for j in list(idx) + [i]:
                k1 = (j + 1) * BS if j != i else t + 1
                s = (Q[:, t, :] / math.sqrt(d)) @ K[j * BS:k1].T
                m = s.max(axis=1)
                e = np.exp(s - m[:, None])
                parts.append((m, e.sum(axis=1), e @ V[j * BS:k1]))
            o, lse = O.lse_merge(parts)
            np.testing.assert_allclose(got["o"][:, t], o, atol=1e-12, rtol=0)
            np.testing.assert_allclose(got["lse"][:, t], lse, atol=1e-12, rtol=0)


@pytest.mark.parametrize("n,top_k", [(1, 4), (8, 4), (64, 16), (256, 16), (5, 0)])
def test_prefill_cost_is_linear_in_length(n, top_k):
    """[README Core] "Sub-Quadratic Prefill": O(L^2) down to O(L * K).  For T = 256 n the
    scored pairs are n causal triangles plus 256^2 per routed block, sum_i min(i, K)."""
    T = n * BS
    k_of = lambda i: i if (top_k == 0 or top_k >= i) else top_k
    closed = n * BS * (BS + 1) // 2 + BS * BS * sum(k_of(i) for i in range(n))
    assert O.prefill_pairs(T, top_k) == closed
    if top_k and n >= 256:  # doubling the length doubles the cost once n >> K
        ratio = O.prefill_pairs(2 * T, top_k) / O.prefill_pairs(T, top_k)
        assert 1.95 < ratio < 2.05
    if top_k == 0:
        assert O.prefill_pairs(T, 0) == T * (T + 1) // 2  # dense causal


# ----------------------------------------------------------------- un-rotated pool (RoPE at read)
# [README Knobs] DKV_ROTATED_POOL=0 stores keys before RoPE and rotates them to their
# absolute positions at read.  The pins below rotate with complex arithmetic of their
# own (pair j as the complex number x_j + i x_{j + dims/2}, multiplied by
# exp(i pos base^(-2j/dims))), not with the oracle's rotation.

def _rope_complex(X, pos, dims, base):
    X = np.asarray(X, dtype=np.float64)
    out = X.copy()
    if dims == 0:
        return out
    h = dims // 2
    inv_freq = 1.0 / np.power(float(base), np.arange(0, dims, 2, dtype=np.float64) / dims)
    z = (X[:, :h] + 1j * X[:, h:dims]) * np.exp(1j * np.outer(np.asarray(pos, dtype=np.float64), inv_freq))
    out[:, :h], out[:, h:dims] = z.real, z.imag
    return out


@pytest.mark.parametrize("d,dims,base", [(16, 16, 10000.0), (32, 8, 500.0), (64, 64, 1e6), (32, 0, 1e4)])
def test_rope_is_a_complex_rotation_of_channel_pairs(d, dims, base):
    """Each pair (j, j + dims/2) turns by pos * base^(-2j/dims); channels >= dims stay."""
    rng = np.random.default_rng(dims + d)
    X = rng.standard_normal((40, d))
    pos = rng.integers(0, 70000, 40)
    got = O.apply_rope(X, pos, O.Rope(dims, base))
    # angles up to 7e4 rad carry fp64 rounding of ~1e-11 rad whichever way the frequency is written
    np.testing.assert_allclose(got, _rope_complex(X, pos, dims, base), atol=2e-10, rtol=0)
    np.testing.assert_array_equal(got[:, dims:], X[:, dims:])
    np.testing.assert_allclose(O.apply_rope(X, np.zeros(40, dtype=np.int64), O.Rope(dims, base)), X, atol=0)


def test_rope_scores_depend_on_relative_position_only():
    """(R_m q) . (R_n k) = (R_{m+s} q) . (R_{n+s} k) = q . (R_{n-m} k): RoPE's defining property."""
    rng = np.random.default_rng(77)
    rope = O.Rope(32, 10000.0)
    q, k = rng.standard_normal((1, 32)), rng.standard_normal((1, 32))
    for m, n, s in ((5, 900, 1000), (0, 3, 65000), (700, 2, 12345)):
        a = (O.apply_rope(q, [m], rope) * O.apply_rope(k, [n], rope)).sum()
        b = (O.apply_rope(q, [m + s], rope) * O.apply_rope(k, [n + s], rope)).sum()
        c = (q * O.apply_rope(k, [n - m], rope)).sum()
        assert abs(a - b) < 1e-9 and abs(a - c) < 1e-9


def _rope_unit_case(rng, d, nb, W, rank, R, dims, base=10000.0, exact_rank=None):
    K, V = _kv(rng, nb * BS + W, d)
    if exact_rank is not None:  # every block's K|V deltas to its anchor of rank exact_rank
        for b in range(nb):
            L = rng.standard_normal((BS - 1, exact_rank))
            Wk, Wv = rng.standard_normal((2, exact_rank, d))
            K[b * BS + 1:(b + 1) * BS] = K[b * BS] + L @ Wk
            V[b * BS + 1:(b + 1) * BS] = V[b * BS] + L @ Wv
    rope = O.Rope(dims, base)
    return K, V, rope, O.compress_unit(K, V, nb, rank, R, rope=rope)


@pytest.mark.parametrize("d,nb,W,dims", [(16, 3, 40, 16), (8, 2, 0, 8), (32, 2, 7, 16)])
def test_unrotated_pool_full_rank_equals_dense_rope_attention(d, nb, W, dims):
    """r = min(255, 2d), R = 0, every block routed: softmax of q against every key
    rotated to its own position (block b token i at 256 b + i, window token w at
    256 NB + w), values unrotated."""
    rng = np.random.default_rng(90 + d)
    K, V, rope, unit = _rope_unit_case(rng, d, nb, W, min(255, 2 * d), 0, dims)
    q = rng.standard_normal((3, d))
    Kr = _rope_complex(K, np.arange(K.shape[0]), dims, rope.base)
    o, lse = _dense(q, Kr, V)
    got = O.decode_unit(q, unit, 0)
    np.testing.assert_allclose(got["o"], o, atol=1e-10, rtol=0)
    np.testing.assert_allclose(got["lse"], lse, atol=1e-10, rtol=0)


def test_unrotated_pool_is_exact_on_low_rank_keys_before_rope():
    """Blocks whose K|V deltas before RoPE have rank r: the un-rotated pool at rank r
    is lossless, while compressing the rotated keys at the same rank is not (RoPE
    turns every token by its own angle, which raises the rank of the deltas)."""
    rng = np.random.default_rng(5)
    d, nb, W, r = 16, 2, 10, 3
    K, V, rope, unit = _rope_unit_case(rng, d, nb, W, r, 0, d, base=100.0, exact_rank=r)
    q = rng.standard_normal((2, d))
    Kr = _rope_complex(K, np.arange(K.shape[0]), d, rope.base)
    o, _ = _dense(q, Kr, V)
    np.testing.assert_allclose(O.decode_unit(q, unit, 0)["o"], o, atol=1e-9, rtol=0)
    rotated = O.compress_unit(Kr, V, nb, r, 0)
    assert np.abs(O.decode_unit(q, rotated, 0)["o"] - o).max() > 1e-4


def test_unrotated_residual_key_round_trip():
    """A residual key read back from the pool and rotated to its absolute position
    reproduces the rotated key that lived there (the README's un-rotated pool
    round trip); with partial RoPE a position off by one moves only the rotated
    channels."""
    rng = np.random.default_rng(6)
    d, nb, dims = 32, 3, 8
    K, V, rope, unit = _rope_unit_case(rng, d, nb, 5, 2, 12, dims)
    Kr = _rope_complex(K, np.arange(K.shape[0]), dims, rope.base)
    for b, blk in enumerate(unit.blocks):
        pos = b * BS + blk.S
        np.testing.assert_allclose(O.apply_rope(blk.K_res, pos, rope), Kr[pos], atol=1e-12, rtol=0)
        off = O.apply_rope(blk.K_res, pos + 1, rope) - Kr[pos]
        assert np.abs(off[:, :dims]).max() > 1e-3
        np.testing.assert_array_equal(off[:, dims:], 0.0)


def test_unrotated_router_box_bounds_every_rotated_key():
    """The box is the channel extremes of the block's exact keys at their positions,
    so bound_b >= qbar . k for each of them."""
    rng = np.random.default_rng(8)
    d, nb = 16, 4
    K, V, rope, unit = _rope_unit_case(rng, d, nb, 0, 2, 3, d)
    Kr = _rope_complex(K, np.arange(K.shape[0]), d, rope.base)
    q = rng.standard_normal((4, d))
    qbar = (q / math.sqrt(d)).mean(axis=0)
    bounds = O.router_bounds(q, np.stack([b.kmin for b in unit.blocks]), np.stack([b.kmax for b in unit.blocks]))
    for b, blk in enumerate(unit.blocks):
        np.testing.assert_allclose(blk.kmin, Kr[b * BS:(b + 1) * BS].min(axis=0), atol=1e-12, rtol=0)
        np.testing.assert_allclose(blk.kmax, Kr[b * BS:(b + 1) * BS].max(axis=0), atol=1e-12, rtol=0)
        assert bounds[b] >= (Kr[b * BS:(b + 1) * BS] @ qbar).max() - 1e-12


def test_unrotated_streaming_append_equals_batch_compression():
    """Appending into an un-rotated pool: the window's oldest tokens keep their
    positions when they become a block, so the result equals compressing the whole
    sequence at once."""
    rng = np.random.default_rng(9)
    d, cap = 16, 300
    K, V = _kv(rng, 1100, d)
    rope = O.Rope(16, 10000.0)
    unit = O.compress_unit(K[:0], V[:0], 0, 3, 5, rope=rope)
    t = 0
    for n in (1, 299, 1, 256, 300, 243):
        unit = O.append_tokens(unit, K[t:t + n], V[t:t + n], cap, 3, 5)
        t += n
    nb = len(unit.blocks)
    ref = O.compress_unit(K[:t], V[:t], nb, 3, 5, rope=rope)
    for a, b in zip(unit.blocks, ref.blocks):
        np.testing.assert_allclose(a.kmin, b.kmin, atol=1e-12, rtol=0)
        np.testing.assert_allclose(a.kmax, b.kmax, atol=1e-12, rtol=0)
    q = rng.standard_normal((2, d))
    np.testing.assert_allclose(O.decode_unit(q, unit, 2)["o"], O.decode_unit(q, ref, 2)["o"], atol=1e-12, rtol=0)


def test_unrotated_pool_brute_force_loops():
    """Tiny case in scalar Python: rotate every routed key with math.cos / math.sin at
    its position, one softmax, against decode_unit."""
    rng = np.random.default_rng(11)
    d, nb, W, dims, base = 8, 3, 5, 4, 50.0
    K, V, rope, unit = _rope_unit_case(rng, d, nb, W, 2, 4, dims, base=base)
    q = rng.standard_normal((2, d))
    got = O.decode_unit(q, unit, 2)
    keys, vals = [], []
    for b in got["idx"]:
        Kh, Vh = O.reconstruct_block(unit.blocks[b])
        for i in range(BS):
            keys.append((b * BS + i, list(Kh[i])))
            vals.append(list(Vh[i]))
    for w in range(W):
        keys.append((nb * BS + w, list(K[nb * BS + w])))
        vals.append(list(V[nb * BS + w]))
    h = dims // 2
    for g in range(2):
        scores = []
        for pos, k in keys:
            kr = list(k)
            for j in range(h):
                a = pos * base ** (-2.0 * j / dims)
                kr[j] = k[j] * math.cos(a) - k[j + h] * math.sin(a)
                kr[j + h] = k[j + h] * math.cos(a) + k[j] * math.sin(a)
            scores.append(sum(q[g][c] * kr[c] for c in range(d)) / math.sqrt(d))
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        l = sum(e)
        o = [sum(e[t] * vals[t][c] for t in range(len(e))) / l for c in range(d)]
        np.testing.assert_allclose(got["o"][g], o, atol=1e-11, rtol=0)
        assert abs(got["lse"][g] - (m + math.log(l))) < 1e-11


def test_unrotated_pool_refuses_the_factored_scorer_and_zero_dims_is_the_rotated_pool():
    rng = np.random.default_rng(12)
    d = 16
    K, V = _kv(rng, 2 * BS + 9, d)
    q = rng.standard_normal((2, d))
    with pytest.raises(ValueError):
        O.decode_unit_factored(q, O.compress_unit(K, V, 2, 3, 4, rope=O.Rope(16, 1e4)), 1)
    plain = O.decode_unit(q, O.compress_unit(K, V, 2, 3, 4), 1)
    zero = O.decode_unit(q, O.compress_unit(K, V, 2, 3, 4, rope=O.Rope(0, 1e4)), 1)
    np.testing.assert_allclose(zero["o"], plain["o"], atol=1e-13, rtol=0)
