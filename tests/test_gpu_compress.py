"""GPU block compression (dkv_compress_layout) against the fp64 oracle.

Exact parts (anchors, key min/max, residual rows, window) must be bit-exact.
The low-rank part is compared through what the truncated SVD fixes: the
Eckart-Young error (the oracle's discarded singular values), orthonormal
basis rows, and a residual set that is the R worst-reconstructed rows of the
GPU's own factors and agrees with the oracle's set outside a narrow band
around the R-th error.  A layout round trip (dkv_import_factors, then the
host unpacker) pins the packing itself bit-exactly.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H
from tests import layout_unpack as LU

pytestmark = pytest.mark.gpu

# Residual-set agreement.  Where the rank cut has a spectral gap the GPU must
# keep the oracle's rows except those whose oracle error is within RES_BAND of
# the oracle's R-th largest.  Everywhere, the GPU's choice must be nearly as
# good by the oracle's own objective: the key error energy left on the
# non-residual rows, sum_{i not in S} e_i^2 with the oracle's e, may exceed the
# oracle's optimum by at most RES_LOSS (relative).  When the cut falls inside a
# near-degenerate stretch of the spectrum (sigma_r / sigma_{r+1} < GAP) the
# truncated subspace itself is not unique, so per-row errors may differ there.
RES_BAND = 0.05
RES_LOSS = 0.02
GAP = 1.1


def _gpu_cache(w, layer, K, V, layout=dkv.DKV_LAYOUT_FRAGMENT):
    r = w.rank(layer)
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          layout=layout)
    ws = torch.zeros(max(256, dkv.dkv_decode_workspace_bytes(desc, w.top_k)), dtype=torch.uint8, device="cuda")
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), workspace=ws)
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK, f"device error word {word:#x}"
    return desc, cache


def _check_block(g, ob, Kb, Vb, r, R, stats):
    f64 = np.float64
    np.testing.assert_array_equal(g["a_k"], Kb[0])
    np.testing.assert_array_equal(g["a_v"], Vb[0])
    np.testing.assert_array_equal(g["kmin"], Kb.min(0))
    np.testing.assert_array_equal(g["kmax"], Kb.max(0))
    assert (g["U_row0"] == 0).all() and g["res_pad_zero"]
    S = g["S"]
    nres = min(R, 255)
    assert len(S) == R and (S[:nres] >= 1).all() and (S[:nres] <= 255).all() and (np.diff(S[:nres]) > 0).all()
    np.testing.assert_array_equal(g["K_res"][:nres], Kb[S[:nres]])
    np.testing.assert_array_equal(g["V_res"][:nres], Vb[S[:nres]])
    m = np.zeros(256, bool)
    m[S[:nres]] = True
    np.testing.assert_array_equal(g["mask"], m)
    X = np.concatenate([Kb[1:].astype(f64) - Kb[0], Vb[1:].astype(f64) - Vb[0]], axis=1)
    d = Kb.shape[1]
    if r > 0:
        Wg = np.concatenate([g["V_K"], g["V_V"]], axis=1).astype(f64)
        Ug = g["U"].astype(f64)
        E_gpu = ((X - Ug @ Wg) ** 2).sum()
        E_opt = float((ob.sigma[r:] ** 2).sum())
        Wo = np.concatenate([ob.V_K, ob.V_V], axis=1)
        E_rnd = ((X - ob.U.astype(np.float16).astype(f64) @ Wo.astype(np.float16).astype(f64)) ** 2).sum()
        # Where the cut has a spectral gap the GPU's iteration converges and may
        # exceed the optimum by 0.1 % plus what fp16 storage costs.  In a flat
        # stretch of the spectrum any subspace of the near-equal directions is
        # almost optimal and convergence is slow; there 1 % is allowed.
        gap_ok = r >= len(ob.sigma) or ob.sigma[r - 1] > GAP * ob.sigma[r]
        allowance = 3 * max(E_rnd - E_opt, 0.0) + (1e-3 if gap_ok else 1e-2) * E_opt + 1e-6 * (X ** 2).sum()
        stats["ey"].append((E_gpu - E_opt) / max(E_opt, 1e-30))
        assert E_gpu - E_opt <= allowance, f"Eckart-Young: E_gpu {E_gpu}, E_opt {E_opt}, fp16 rounding {E_rnd}"
        assert np.abs(Wg @ Wg.T - np.eye(r)).max() < 4e-3
        e_gpu = np.sqrt(((X[:, :d] - Ug @ g["V_K"].astype(f64)) ** 2).sum(1))
        slack = 2.0 ** -9 * np.sqrt((Ug ** 2).sum(1)).max()
    else:
        e_gpu = np.sqrt((X[:, :d] ** 2).sum(1))
        slack = 0.0
    # all rows reconstructed to rounding level (r >= rank of X): any choice is exact
    degenerate = np.sort(ob.err)[::-1][max(nres - 1, 0)] <= 1e-4 * np.sqrt((X[:, :d] ** 2).mean())
    if 0 < nres < 255 and not degenerate:
        kept = e_gpu[S[:nres] - 1]
        dropped = np.delete(e_gpu, S[:nres] - 1)
        assert kept.min() >= dropped.max() - slack, "GPU residual set is not the worst-reconstructed rows"
        diff = set(S[:nres].tolist()) ^ set(ob.S.tolist())
        thr = np.sort(ob.err)[::-1][nres - 1]
        stats["res_diff"].append(len(diff))
        loss = lambda keep: float((np.delete(ob.err, np.asarray(keep) - 1) ** 2).sum())
        l_opt = loss(ob.S)
        excess = (loss(S[:nres]) - l_opt) / max(l_opt, 1e-30)
        stats["res_loss"].append(excess)
        assert excess <= RES_LOSS, f"residual choice loses {excess:.3%} of the oracle's objective"
        gapped = r == 0 or r >= len(ob.sigma) or ob.sigma[r - 1] > GAP * ob.sigma[r]
        for t in diff:
            rel = abs(ob.err[t - 1] - thr) / thr
            stats["res_rel"].append(rel)
            if gapped:
                assert rel <= RES_BAND, f"row {t}: oracle error {ob.err[t - 1]} vs R-th {thr}"


def _run(w, layer, bh_check, decode=True, layout=dkv.DKV_LAYOUT_FRAGMENT):
    K, V = synth.layer_kv(w, layer)
    desc, cache = _gpu_cache(w, layer, K, V, layout)
    host = cache.cpu().numpy()
    r, R = w.rank(layer), w.n_residual
    stats = {"ey": [], "res_diff": [], "res_rel": [], "res_loss": []}
    q = synth.queries(w, layer)
    if decode:
        out, lse, routed = dkv.dkv_decode_attend(desc, torch.from_numpy(q).cuda(), cache, w.top_k)
        out, routed = out.cpu().numpy(), (routed.cpu().numpy() if routed is not None else None)
    G = w.group
    for (b, h) in bh_check:
        u = b * w.n_kv_heads + h
        ounit = H.oracle_unit_blockwise(K[b, h], V[b, h], w.n_blocks, r, R)
        for blk in range(w.n_blocks):
            g = LU.unpack_block(host, desc, u, blk)
            _check_block(g, ounit.blocks[blk], K[b, h, blk * 256:(blk + 1) * 256],
                         V[b, h, blk * 256:(blk + 1) * 256], r, R, stats)
        wk, wv = LU.unpack_window(host, desc, u)
        np.testing.assert_array_equal(wk, K[b, h, w.n_blocks * 256:])
        np.testing.assert_array_equal(wv, V[b, h, w.n_blocks * 256:])
        if decode:
            qg = q[b, h * G:(h + 1) * G].astype(np.float64)
            ref = O.decode_unit(qg, ounit, w.top_k)
            ref16 = O.decode_unit(qg, H.round_unit(ounit), w.top_k)
            if routed is not None:
                H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
            # end to end: both sides compress on their own; the bound adds what fp16
            # storage of the factors costs (measured on the oracle's own factors)
            storage = np.abs(ref16["o"] - ref["o"]).max()
            err = np.abs(out[b, h * G:(h + 1) * G] - ref["o"]).max()
            stats.setdefault("e2e", []).append((err, storage))
            assert err <= H.ATOL_OUT + 4 * storage, f"end-to-end {err} vs storage {storage}"
    return stats


LAYOUTS = [dkv.DKV_LAYOUT_FRAGMENT, dkv.DKV_LAYOUT_TC]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_roundtrip_is_bit_exact(layout):
    w = synth.WORKLOADS["8k"]
    units = H.oracle_units(w, 0, [(0, 0), (0, 1)])
    arrs = H.factor_arrays(units, 128, 32, 40, w.window)
    desc = dkv.dkv_layout(1, 12, 2, 128, w.n_blocks, w.window, 32, 40, layout=layout)
    host = dkv.dkv_import_factors(desc, H.to_device(arrs)).cpu().numpy()
    for u in range(2):
        for b in range(w.n_blocks):
            g = LU.unpack_block(host, desc, u, b)
            for k in ("a_k", "a_v", "U", "V_K", "V_V", "K_res", "V_res", "kmin", "kmax"):
                np.testing.assert_array_equal(g[k], arrs[k][u, b], err_msg=k)
            np.testing.assert_array_equal(g["S"], arrs["res_pos"][u, b])
        wk, wv = LU.unpack_window(host, desc, u)
        np.testing.assert_array_equal(wk, arrs["win_K"][u])
        np.testing.assert_array_equal(wv, arrs["win_V"][u])


def test_compress_tiny():
    w = synth.WORKLOADS["tiny"]
    s = _run(w, 0, [(0, 0)])
    print("tiny", {k: (np.max(v) if len(v) else None) for k, v in s.items() if k != "e2e"}, s.get("e2e"))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_compress_8k(layout):
    w = synth.WORKLOADS["8k"]
    s = _run(w, 0, [(0, 0), (0, 1)], layout=layout)
    print("8k", {k: (np.max(v) if len(v) else None) for k, v in s.items() if k != "e2e"}, s.get("e2e"))


def test_compress_32k_sampled():
    w = synth.WORKLOADS["32k"]
    s = _run(w, 0, [(0, 0), (3, 1)])
    print("32k", {k: (np.max(v) if len(v) else None) for k, v in s.items() if k != "e2e"}, s.get("e2e"))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("layer", [0, 10, 27])
def test_compress_64k_sampled(layer, layout):
    w = synth.WORKLOADS["64k"]
    s = _run(w, layer, [(5, 1)], layout=layout)
    print("64k", layer, {k: (np.max(v) if len(v) else None) for k, v in s.items() if k != "e2e"}, s.get("e2e"))


@pytest.mark.parametrize("kw", [dict(r=0), dict(R=0), dict(R=255), dict(r=64, d=128), dict(r=128, d=64),
                                dict(r=24, R=5, W=17), dict(nb=0, W=40)])
def test_compress_edge(kw):
    base = dict(d=64, G=6, nb=3, W=100, r=16, R=24)
    base.update(kw)
    w = synth.Workload("edge", 1, base["G"], 1, base["d"], base["nb"], base["W"], (base["r"],), base["R"], 2, 4,
                       False, 11)
    _run(w, 0, [(0, 0)])


@pytest.mark.parametrize("kw", [dict(r=1, R=1, W=17), dict(r=48, R=128, W=300), dict(nb=0, W=129)])
def test_compress_edge_tensor_core_layout(kw):
    base = dict(G=6, nb=3, W=100, r=16, R=24)
    base.update(kw)
    w = synth.Workload("edge", 1, base["G"], 1, 128, base["nb"], base["W"], (base["r"],), base["R"], 2, 4,
                       False, 11)
    _run(w, 0, [(0, 0)], layout=dkv.DKV_LAYOUT_TC)
