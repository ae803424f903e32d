"""Planted mistakes in the oracle (CPU only).

Each case swaps one function of the fp64 oracle for a copy with one plausible
slip (a dropped term, a wrong sign, index or tie order, a transposed or swapped
operand, a missing rescale) and runs the pins of tests/test_oracle_pins.py
against it: at least one pin must fail.  A slip that no pin catches would mean
the pins leave that part of the oracle unchecked.  The mistakes are planted in
the oracle only, on the CPU; nothing here touches the GPU path.
"""
import math

import numpy as np
import pytest

from oracle import dkv_oracle as O
from tests import test_oracle_pins as P

BS = O.BLOCK_SIZE


def _pin_calls():
    """Every pin of test_oracle_pins with each of its parameter sets."""
    calls = []
    for name in sorted(n for n in dir(P) if n.startswith("test_")):
        f = getattr(P, name)
        params = [m for m in getattr(f, "pytestmark", []) if m.name == "parametrize"]
        if not params:
            calls.append((name, f, {}))
            continue
        assert len(params) == 1, name
        argnames, values = params[0].args[0], params[0].args[1]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for v in values:
            v = tuple(v) if len(argnames) > 1 else (v,)
            calls.append((name, f, dict(zip(argnames, v))))
    return calls


def _first_failing_pin(monkeypatch, fn_name, mutant):
    """The first pin whose assertion fails with the mutant in place, and the
    other errors met on the way (an error is not a catch: it may be the
    mutant's own fault)."""
    monkeypatch.setattr(O, fn_name, mutant)
    errors = []
    for name, f, kw in _pin_calls():
        try:
            f(**kw)
        except (AssertionError, pytest.fail.Exception):
            return name, errors
        except Exception as e:
            errors.append(f"{name}{kw}: {type(e).__name__}: {e}")
    return None, errors


# ----------------------------------------------------------------------------- mutants

_orig = {n: getattr(O, n) for n in ("router_bounds", "route", "select_residuals", "compress_block",
                                    "reconstruct_block", "softmax_attention", "lse_merge", "block_partial",
                                    "decode_unit", "append_tokens", "effective_top_k", "compress_unit",
                                    "decode_unit_factored", "_part", "pages_block_bytes", "residual_row_bytes",
                                    "dense_kv_bytes", "quantize_groups", "dequantize_groups",
                                    "quantize_block_residuals", "quant_residual_row_bytes", "prefill_routes",
                                    "prefill_unit", "prefill_pairs", "apply_rope", "rope_angles", "rope_key_box")}


def _bounds_without_kmin(q, kmin, kmax):
    q = np.asarray(q, dtype=np.float64)
    qbar = (q / math.sqrt(q.shape[1])).mean(axis=0)
    return (qbar[None, :] * np.asarray(kmax, dtype=np.float64)).sum(axis=1)


def _bounds_first_head_only(q, kmin, kmax):
    return _orig["router_bounds"](np.asarray(q)[:1], kmin, kmax)


def _bounds_unscaled(q, kmin, kmax):
    q = np.asarray(q, dtype=np.float64)
    return _orig["router_bounds"](q * math.sqrt(q.shape[1]), kmin, kmax)


def _route_ties_to_higher(bounds, top_k):
    k = O.effective_top_k(top_k, bounds.shape[0])
    order = sorted(range(bounds.shape[0]), key=lambda b: (-float(bounds[b]), -b))[:k]
    return np.array(sorted(order), dtype=np.int64)


def _route_in_rank_order(bounds, top_k):
    k = O.effective_top_k(top_k, bounds.shape[0])
    return np.array(sorted(range(bounds.shape[0]), key=lambda b: (-float(bounds[b]), b))[:k], dtype=np.int64)


def _residuals_best_rows(err, n_residual):
    R = max(0, min(int(n_residual), err.shape[0]))
    return np.array(sorted(i + 1 for i in sorted(range(err.shape[0]), key=lambda i: (float(err[i]), i))[:R]),
                    dtype=np.int64)


def _residuals_ties_to_higher(err, n_residual):
    R = max(0, min(int(n_residual), err.shape[0]))
    return np.array(sorted(i + 1 for i in sorted(range(err.shape[0]), key=lambda i: (-float(err[i]), -i))[:R]),
                    dtype=np.int64)


def _compress(Kb, Vb, rank, n_residual, *, fold_sigma=True, delta_to_mean=False, swap_halves=False,
              minmax_over_deltas=False, error_on_values=False):
    """compress_block with one switchable slip."""
    Kb = np.asarray(Kb, dtype=np.float64)
    Vb = np.asarray(Vb, dtype=np.float64)
    d = Kb.shape[1]
    a_k, a_v = Kb[0].copy(), Vb[0].copy()
    ref_k, ref_v = (Kb[1:].mean(0), Vb[1:].mean(0)) if delta_to_mean else (a_k, a_v)
    dK, dV = Kb[1:] - ref_k, Vb[1:] - ref_v
    U_hat, sigma, Wt = np.linalg.svd(np.concatenate([dK, dV], axis=1), full_matrices=False)
    r = max(0, min(int(rank), sigma.shape[0]))
    U = U_hat[:, :r] * sigma[:r] if fold_sigma else U_hat[:, :r].copy()
    V_K, V_V = Wt[:r, :d].copy(), Wt[:r, d:].copy()
    if swap_halves:
        V_K, V_V = V_V, V_K
    err = np.sqrt((((dV - U @ V_V) if error_on_values else (dK - U @ V_K)) ** 2).sum(axis=1))
    S = O.select_residuals(err, n_residual)
    keys = Kb[1:] - a_k if minmax_over_deltas else Kb
    return O.Block(a_k=a_k, a_v=a_v, U=U, V_K=V_K, V_V=V_V, S=S, K_res=Kb[S].copy(), V_res=Vb[S].copy(),
                   kmin=keys.min(axis=0), kmax=keys.max(axis=0), sigma=sigma, err=err)


def _reconstruct(blk, *, substitute=True, shift=0):
    d = blk.a_k.shape[0]
    Kh, Vh = np.empty((BS, d)), np.empty((BS, d))
    Kh[0], Vh[0] = blk.a_k, blk.a_v
    Kh[1:] = blk.a_k + blk.U @ blk.V_K
    Vh[1:] = blk.a_v + blk.U @ blk.V_V
    if substitute and blk.S.size:
        Kh[blk.S - shift] = blk.K_res
        Vh[blk.S - shift] = blk.V_res
    return Kh, Vh


def _softmax_unscaled(q, K, V):
    q = np.asarray(q, dtype=np.float64)
    return _orig["softmax_attention"](q * math.sqrt(q.shape[1]), K, V)


def _merge_without_rescale(parts):
    ms = np.stack([p[0] for p in parts])
    mstar = ms.max(axis=0)
    w = np.exp(ms - mstar[None, :])
    lstar = sum(p[1] for p in parts)
    acc = sum(wj[:, None] * p[2] for wj, p in zip(w, parts))
    return acc / lstar[:, None], mstar + np.log(lstar)


def _merge_lse_without_max(parts):
    o, lse = _orig["lse_merge"](parts)
    return o, lse - np.stack([p[0] for p in parts]).max(axis=0)


def _partial(q, blk, *, anchor=True, anchor_value=True, z_sign=1.0):
    """block_partial with one switchable slip."""
    q = np.asarray(q, dtype=np.float64)
    qt = q / math.sqrt(q.shape[1])
    z = qt @ blk.V_K.T
    base = qt @ blk.a_k
    lowrank = np.ones(BS, dtype=bool)
    lowrank[blk.S] = False
    lr = np.nonzero(lowrank[1:])[0]
    s_lr = base[:, None] + z_sign * (z @ blk.U[lr].T)
    s_res = qt @ blk.K_res.T
    s_anchor = base[:, None] if anchor else np.full_like(base[:, None], -np.inf)
    m = np.concatenate([s_anchor, s_lr, s_res], axis=1).max(axis=1)
    p_a, p_lr, p_res = (np.exp(x - m[:, None]) for x in (s_anchor, s_lr, s_res))
    pa = p_a[:, 0] + p_lr.sum(axis=1)
    acc = (pa if anchor_value else p_lr.sum(axis=1))[:, None] * blk.a_v[None, :] + (p_lr @ blk.U[lr]) @ blk.V_V \
        + p_res @ blk.V_res
    return m, pa + p_res.sum(axis=1), acc


def _decode_without_window(q, unit, top_k):
    return _orig["decode_unit"](q, O.Unit(blocks=unit.blocks, win_K=unit.win_K[:0], win_V=unit.win_V[:0]), top_k)


def _append_newest_first(unit, K_new, V_new, window_capacity, rank, n_residual):
    blocks = list(unit.blocks)
    win_K = [row for row in np.asarray(unit.win_K, dtype=np.float64)]
    win_V = [row for row in np.asarray(unit.win_V, dtype=np.float64)]
    for k, v in zip(np.asarray(K_new, dtype=np.float64), np.asarray(V_new, dtype=np.float64)):
        if len(win_K) == window_capacity:
            if len(win_K) < BS:
                raise ValueError("window capacity below one block")
            blocks.append(O.compress_block(np.array(win_K[-BS:]), np.array(win_V[-BS:]), rank, n_residual))
            win_K, win_V = win_K[:-BS], win_V[:-BS]
        win_K.append(k)
        win_V.append(v)
    d = np.asarray(unit.win_K).shape[-1]
    return O.Unit(blocks=blocks, win_K=np.array(win_K).reshape(-1, d), win_V=np.array(win_V).reshape(-1, d))


def _window_one_token_late(K, V, n_blocks, rank, n_residual):
    unit = _orig["compress_unit"](K, V, n_blocks, rank, n_residual)
    return O.Unit(blocks=unit.blocks, win_K=unit.win_K[1:], win_V=unit.win_V[1:])


def _factored_window_chunks_overlap(q, unit, top_k, window_chunk=256):
    W = unit.win_K.shape[0]
    if W <= 1:
        return _orig["decode_unit_factored"](q, unit, top_k, window_chunk)
    step = max(1, window_chunk - 1)  # consecutive chunks share a token
    q = np.asarray(q, dtype=np.float64)
    qt = q / math.sqrt(q.shape[1])
    nb = len(unit.blocks)
    bounds = O.router_bounds(q, np.stack([b.kmin for b in unit.blocks]), np.stack([b.kmax for b in unit.blocks])) \
        if nb else np.zeros(0)
    idx = O.route(bounds, top_k) if nb else np.zeros(0, dtype=np.int64)
    parts = [O.block_partial(q, unit.blocks[b]) for b in idx]
    for t0 in range(0, W, step):
        parts.append(O._part(qt @ unit.win_K[t0:t0 + window_chunk].T, unit.win_V[t0:t0 + window_chunk]))
    o, lse = O.lse_merge(parts)
    return {"o": o, "lse": lse, "idx": idx, "bounds": bounds}


def _part_with_mean_shift(s, V):
    m = s.mean(axis=1)  # any shift cancels in o, but l and m must describe the same exponentials
    e = np.exp(s - s.max(axis=1)[:, None])
    return m, e.sum(axis=1), e @ V


def _residual_positions_zero_based(err, n_residual):
    return _orig["select_residuals"](err, n_residual) - 1


def _bytes_u_with_256_rows(d, u_rank, R, elem_bytes=4, basis_bytes=None, meta_bytes=8):
    acc = _orig["pages_block_bytes"](d, u_rank, R, elem_bytes, basis_bytes, meta_bytes)
    extra = u_rank * elem_bytes
    return dict(acc, U=acc["U"] + extra, core=acc["core"] + extra, block=acc["block"] + extra,
                ratio=acc["dense"] / (acc["block"] + extra))


def _residual_row_key_only(d, elem_bytes=2):
    return d * elem_bytes


def _dense_bytes_one_layer(context, d, n_layers, n_kv_heads, elem_bytes=2):
    return _orig["dense_kv_bytes"](context, d, 1, n_kv_heads, elem_bytes)


def _top_k_all_but_one(top_k, n_blocks):
    k = _orig["effective_top_k"](top_k, n_blocks)
    return max(0, n_blocks - 1) if k == n_blocks else k


def _partial_residuals_offset_by_anchor(q, blk):
    m, l, acc = _orig["block_partial"](q, blk)
    if blk.S.size == 0:
        return m, l, acc
    q = np.asarray(q, dtype=np.float64)
    qt = q / math.sqrt(q.shape[1])
    # score the exact rows as if they were deltas: q.(a_k + k_j)
    shifted = O.Block(**{**blk.__dict__, "K_res": blk.K_res + blk.a_k[None, :]})
    return _orig["block_partial"](q, shifted)


def _top_k_zero_is_none(top_k, n_blocks):
    if top_k < 0:
        raise ValueError("top_k must be >= 0")
    return min(int(top_k), n_blocks)


def _quantize(X, bits, group=64, rounding=np.rint, levels=None, bias_fn=None, interleave=False):
    """quantize_groups with one slip (rounding, step count, bias or group shape)."""
    X = np.asarray(X, dtype=np.float32)
    n, d = X.shape
    Xg = X.reshape(n, group, d // group).transpose(0, 2, 1) if interleave else X.reshape(n, d // group, group)
    lo, hi = Xg.min(axis=2), Xg.max(axis=2)
    lv = np.float32(levels if levels is not None else 2 ** bits - 1)
    scale = ((hi - lo) / lv).astype(np.float16)
    bias = (bias_fn(Xg) if bias_fn else lo).astype(np.float16)
    sv = scale.astype(np.float32)[:, :, None]
    bv = bias.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = rounding((Xg - bv) / sv)
    q = np.clip(np.where(sv == 0, 0.0, q), 0, 2 ** bits - 1)
    if interleave:
        q = q.transpose(0, 2, 1)
    return q.reshape(n, d).astype(np.uint8), scale, bias


def _dequantize_scale_bias_swapped(codes, scale, bias, group=64):
    return _orig["dequantize_groups"](codes, bias, scale, group)


def _quant_block_kv_swapped(blk, bits):
    import dataclasses
    if blk.S.size == 0:
        return dataclasses.replace(blk)
    return dataclasses.replace(blk, K_res=O.dequantize_groups(*O.quantize_groups(blk.V_res, bits)),
                               V_res=O.dequantize_groups(*O.quantize_groups(blk.K_res, bits)))


def _quant_block_keys_only(blk, bits):
    import dataclasses
    if blk.S.size == 0:
        return dataclasses.replace(blk)
    return dataclasses.replace(blk, K_res=O.dequantize_groups(*O.quantize_groups(blk.K_res, bits)))


def _prefill_routes(Q, K, top_k, mean=True, use_min=True, later=False, zero_is_none=False):
    """prefill_routes with one slip."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    G, T, d = Q.shape
    nb = -(-T // BS)
    out = []
    for i in range(nb):
        t0, t1 = i * BS, min(T, (i + 1) * BS)
        qbar = (Q[:, t0:t1, :] / math.sqrt(d)).mean(axis=(0, 1)) if mean else Q[0, t0] / math.sqrt(d)
        cand = [j for j in range(nb) if j != i] if later else list(range(i))
        b = {}
        for j in cand:
            blk = K[j * BS:min(T, (j + 1) * BS)]
            b[j] = (np.maximum(qbar * blk.max(axis=0), qbar * blk.min(axis=0)) if use_min else qbar * blk.max(axis=0)).sum()
        k = len(cand) if (top_k >= len(cand) or (top_k == 0 and not zero_is_none)) else int(top_k)
        order = sorted(cand, key=lambda j: (-float(b[j]), j))[:k]
        out.append((np.array(sorted(order), dtype=np.int64), np.array([b.get(j, 0.0) for j in range(i)])))
    return out


def _prefill_unit(Q, K, V, top_k, causal_shift=0, own=True):
    """prefill_unit with one slip (the causal mask one token off, or the own block left out)."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    G, T, d = Q.shape
    routes = O.prefill_routes(Q, K, top_k)
    o = np.zeros((G, T, d))
    lse = np.zeros((G, T))
    for i, (idx, _) in enumerate(routes):
        t0, t1 = i * BS, min(T, (i + 1) * BS)
        parts = [np.arange(j * BS, (j + 1) * BS) for j in idx]
        if own or not parts:
            parts.append(np.arange(t0, t1))
        keys = np.concatenate(parts).astype(np.int64)
        s = np.einsum("gtd,kd->gtk", Q[:, t0:t1, :], K[keys]) / math.sqrt(d)
        mask = (keys[None, :] >= t0) & (keys[None, :] > np.arange(t0, t1)[:, None] + causal_shift)
        s = np.where(mask[None], -np.inf, s)
        m = s.max(axis=2, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=2, keepdims=True)
        o[:, t0:t1, :] = np.einsum("gtk,kd->gtd", e, V[keys]) / l
        lse[:, t0:t1] = (m + np.log(l))[:, :, 0]
    return {"o": o, "lse": lse, "routes": [r for r, _ in routes], "bounds": [b for _, b in routes]}


def _prefill_pairs_full_own_block(T, top_k):
    nb = -(-T // BS)
    return sum((min(T, (i + 1) * BS) - i * BS) ** 2 + (min(T, (i + 1) * BS) - i * BS) *
               (i if (top_k == 0 or top_k >= i) else top_k) * BS for i in range(nb))


def _rope(X, pos, rope, pairs="half", sin_sign=1.0, exponent=2.0, all_channels=False):
    X = np.asarray(X, dtype=np.float64)
    out = X.copy()
    dims = X.shape[1] if all_channels else rope.dims
    if dims == 0 or X.shape[0] == 0:
        return out
    h = dims // 2
    theta = float(rope.base) ** (-exponent * np.arange(h) / dims)
    a = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]
    c, sn = np.cos(a), sin_sign * np.sin(a)
    if pairs == "half":
        i, j = np.arange(h), np.arange(h) + h
    else:  # adjacent channels (2j, 2j + 1)
        i, j = 2 * np.arange(h), 2 * np.arange(h) + 1
    out[:, i] = X[:, i] * c - X[:, j] * sn
    out[:, j] = X[:, j] * c + X[:, i] * sn
    return out


def _decode_rope_positions(q, unit, top_k, block_pos=True, window_base=True, rotate_values=False):
    """decode_unit with a slip in where the keys sit (or in what is rotated)."""
    if unit.rope is None:
        return _orig["decode_unit"](q, unit, top_k)
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[1]
    nb = len(unit.blocks)
    bounds = O.router_bounds(q, np.stack([b.kmin for b in unit.blocks]), np.stack([b.kmax for b in unit.blocks])) \
        if nb else np.zeros(0)
    idx = O.route(bounds, top_k) if nb else np.zeros(0, dtype=np.int64)
    Ks, Vs = [], []
    for b in idx:
        Kh, Vh = O.reconstruct_block(unit.blocks[b])
        pos = np.arange(BS) + (b * BS if block_pos else 0)
        Ks.append(O.apply_rope(Kh, pos, unit.rope))
        Vs.append(O.apply_rope(Vh, pos, unit.rope) if rotate_values else Vh)
    W = unit.win_K.shape[0]
    Ks.append(O.apply_rope(unit.win_K, np.arange(W) + (nb * BS if window_base else 0), unit.rope))
    Vs.append(unit.win_V)
    o, lse = O.softmax_attention(q, np.concatenate(Ks), np.concatenate(Vs))
    return {"o": o, "lse": lse, "idx": idx, "bounds": bounds}


def _append_rope_box_at_block_zero(unit, K_new, V_new, window_capacity, rank, n_residual):
    out = _orig["append_tokens"](unit, K_new, V_new, window_capacity, rank, n_residual)
    if unit.rope is None:
        return out
    # recompute the boxes of the blocks this call cut as if each sat at block 0
    blocks = list(out.blocks)
    for b in range(len(unit.blocks), len(blocks)):
        Kh, _ = O.reconstruct_block(blocks[b])
        Kr = O.apply_rope(Kh, np.arange(BS), unit.rope)
        blocks[b] = O.Block(**{**blocks[b].__dict__, "kmin": Kr.min(axis=0), "kmax": Kr.max(axis=0)})
    return O.Unit(blocks=blocks, win_K=out.win_K, win_V=out.win_V, rope=out.rope)


MUTANTS = {
    "RoPE pairs adjacent channels": ("apply_rope", lambda X, pos, rope: _rope(X, pos, rope, pairs="adjacent")),
    "RoPE turns the wrong way": ("apply_rope", lambda X, pos, rope: _rope(X, pos, rope, sin_sign=-1.0)),
    "RoPE frequencies base^(-j/dims)": ("apply_rope", lambda X, pos, rope: _rope(X, pos, rope, exponent=1.0)),
    "partial RoPE rotates every channel": ("apply_rope", lambda X, pos, rope: _rope(X, pos, rope, all_channels=True)),
    "RoPE angles one position late": ("rope_angles", lambda pos, rope: _orig["rope_angles"](np.asarray(pos) + 1, rope)),
    "un-rotated box over the keys before RoPE": ("rope_key_box",
                                                 lambda Kb, b, rope: (np.asarray(Kb).min(axis=0), np.asarray(Kb).max(axis=0))),
    "un-rotated box at block 0's positions": ("rope_key_box", lambda Kb, b, rope: _orig["rope_key_box"](Kb, 0, rope)),
    "un-rotated blocks all at positions 0..255": ("decode_unit",
                                                  lambda q, u, k: _decode_rope_positions(q, u, k, block_pos=False)),
    "un-rotated window positions from 0": ("decode_unit",
                                           lambda q, u, k: _decode_rope_positions(q, u, k, window_base=False)),
    "un-rotated pool rotates the values too": ("decode_unit",
                                               lambda q, u, k: _decode_rope_positions(q, u, k, rotate_values=True)),
    "un-rotated append boxes at block 0": ("append_tokens", _append_rope_box_at_block_zero),
    "prefill routes by the block's first query": ("prefill_routes", lambda Q, K, k: _prefill_routes(Q, K, k, mean=False)),
    "prefill bound drops the kmin branch": ("prefill_routes", lambda Q, K, k: _prefill_routes(Q, K, k, use_min=False)),
    "prefill routes later blocks too": ("prefill_routes", lambda Q, K, k: _prefill_routes(Q, K, k, later=True)),
    "prefill top-K 0 routes no block": ("prefill_routes", lambda Q, K, k: _prefill_routes(Q, K, k, zero_is_none=True)),
    "prefill causal mask one token late": ("prefill_unit", lambda Q, K, V, k: _prefill_unit(Q, K, V, k, causal_shift=1)),
    "prefill leaves out the own block": ("prefill_unit", lambda Q, K, V, k: _prefill_unit(Q, K, V, k, own=False)),
    "prefill cost counts the whole own block": ("prefill_pairs", _prefill_pairs_full_own_block),

    "quantisation rounds down": ("quantize_groups", lambda X, bits, group=64: _quantize(X, bits, group, rounding=np.floor)),
    "quantisation step over 2^bits levels": ("quantize_groups",
                                             lambda X, bits, group=64: _quantize(X, bits, group, levels=2 ** bits)),
    "quantisation bias at the group mean": ("quantize_groups", lambda X, bits, group=64: _quantize(
        X, bits, group, bias_fn=lambda Xg: Xg.mean(axis=2))),
    "quantisation groups strided across the row": ("quantize_groups",
                                                   lambda X, bits, group=64: _quantize(X, bits, group, interleave=True)),
    "dequantisation swaps scale and bias": ("dequantize_groups", _dequantize_scale_bias_swapped),
    "quantised residual keys and values swapped": ("quantize_block_residuals", _quant_block_kv_swapped),
    "quantised residuals leave the values exact": ("quantize_block_residuals", _quant_block_keys_only),
    "quantised row bytes without scale and bias": ("quant_residual_row_bytes", lambda d, bits, group=64: d * bits // 8),

    "router bound drops the kmin branch": ("router_bounds", _bounds_without_kmin),
    "router bound uses one head, not the group mean": ("router_bounds", _bounds_first_head_only),
    "router bound misses the 1/sqrt(d) scale": ("router_bounds", _bounds_unscaled),
    "routing ties go to the higher block": ("route", _route_ties_to_higher),
    "routed indices left in rank order": ("route", _route_in_rank_order),
    "residuals keep the best rows": ("select_residuals", _residuals_best_rows),
    "residual ties go to the higher token": ("select_residuals", _residuals_ties_to_higher),
    "singular values not folded into U": ("compress_block", lambda *a, **k: _compress(*a, **k, fold_sigma=False)),
    "deltas taken to the block mean": ("compress_block", lambda *a, **k: _compress(*a, **k, delta_to_mean=True)),
    "V_K and V_V swapped": ("compress_block", lambda *a, **k: _compress(*a, **k, swap_halves=True)),
    "key box over the deltas": ("compress_block", lambda *a, **k: _compress(*a, **k, minmax_over_deltas=True)),
    "residual error measured on values": ("compress_block", lambda *a, **k: _compress(*a, **k, error_on_values=True)),
    "residual rows not substituted": ("reconstruct_block", lambda b: _reconstruct(b, substitute=False)),
    "residual rows substituted one row early": ("reconstruct_block", lambda b: _reconstruct(b, shift=1)),
    "softmax misses the 1/sqrt(d) scale": ("softmax_attention", _softmax_unscaled),
    "merge sums l without rescaling": ("lse_merge", _merge_without_rescale),
    "merged lse drops the maximum": ("lse_merge", _merge_lse_without_max),
    "factored scores drop the anchor": ("block_partial", lambda q, b: _partial(q, b, anchor=False)),
    "factored value drops the anchor's weight": ("block_partial", lambda q, b: _partial(q, b, anchor_value=False)),
    "factored scores subtract U z": ("block_partial", lambda q, b: _partial(q, b, z_sign=-1.0)),
    "decode skips the window": ("decode_unit", _decode_without_window),
    "append compresses the newest tokens": ("append_tokens", _append_newest_first),
    "top-K 0 routes no block": ("effective_top_k", _top_k_zero_is_none),
    "top-K >= NB routes all but one block": ("effective_top_k", _top_k_all_but_one),
    "window starts one token late": ("compress_unit", _window_one_token_late),
    "factored window chunks overlap by a token": ("decode_unit_factored", _factored_window_chunks_overlap),
    "partial's maximum is not its shift": ("_part", _part_with_mean_shift),
    "residual positions zero-based": ("select_residuals", _residual_positions_zero_based),
    "factored residual scores offset by the anchor": ("block_partial", _partial_residuals_offset_by_anchor),
    "page table: U with 256 rows": ("pages_block_bytes", _bytes_u_with_256_rows),
    "residual row counts the key only": ("residual_row_bytes", _residual_row_key_only),
    "dense bytes of one layer": ("dense_kv_bytes", _dense_bytes_one_layer),
}


@pytest.mark.parametrize("slip", sorted(MUTANTS))
def test_pins_catch_a_planted_slip(slip, monkeypatch):
    fn_name, mutant = MUTANTS[slip]
    caught_by, errors = _first_failing_pin(monkeypatch, fn_name, mutant)
    assert caught_by is not None, f"no pin fails when the oracle's {fn_name} has the slip: {slip}; errors: {errors[:3]}"


def test_the_unmutated_oracle_passes_every_pin(monkeypatch):
    """The harness itself: with the oracle as it is, no pin fails."""
    assert _first_failing_pin(monkeypatch, "route", _orig["route"]) == (None, [])
