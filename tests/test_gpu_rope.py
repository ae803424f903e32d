"""GPU parity of the un-rotated pool (keys stored before RoPE, rotated to their
absolute positions at read) against the fp64 oracle.

Caches are filled from oracle factors (dkv_import_factors) or compressed on the
GPU; the oracle decodes by its plain definition (every attended key rebuilt,
rotated to 256 b + i or 256 NB + w, one softmax).  Outputs and lse within 2e-3;
routed blocks exact outside the 1e-4 tie band (the boxes are fp32 on the GPU,
fp64 in the oracle).
"""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H
from tests import layout_unpack as LU

pytestmark = pytest.mark.gpu


def _import_case(w, layer, top_ks, rope, distinct=None):
    r = w.rank(layer)
    bh = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    todo = bh if distinct is None else bh[:distinct]
    base = H.oracle_units(w, layer, todo, rope=rope)
    units = [base[i % len(base)] for i in range(len(bh))]
    rounded = [H.round_unit(u) for u in base]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          rope_dims=rope.dims, rope_base=rope.base)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, w.head_dim, r, w.n_residual, w.window)))
    q = synth.queries(w, layer)
    qd = torch.from_numpy(q).cuda()
    ws = torch.zeros(max(dkv.dkv_decode_workspace_bytes(desc, k) for k in top_ks), dtype=torch.uint8, device="cuda")
    G = w.group
    n_tie = 0
    for top_k in top_ks:
        out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, top_k, workspace=ws)
        out_ns, _, _ = dkv.dkv_decode_attend(desc, qd, cache, top_k, routed=False, workspace=ws)
        torch.cuda.synchronize()
        st, word = dkv.dkv_get_error(ws)
        assert st == dkv.DKV_OK and word == 0, f"device error word {word:#x}"
        out, lse, out_ns = out.cpu().numpy(), lse.cpu().numpy(), out_ns.cpu().numpy()
        routed = routed.cpu().numpy() if routed is not None else None
        for i, (b, h) in enumerate(bh):
            qg = q[b, h * G:(h + 1) * G].astype(np.float64)
            ref = O.decode_unit(qg, rounded[i % len(rounded)], top_k)
            if routed is not None:
                H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
                if set(routed[b, h]) != set(ref["idx"]):
                    n_tie += 1
                    continue
            for o_ in (out, out_ns):
                err = np.abs(o_[b, h * G:(h + 1) * G] - ref["o"]).max()
                assert err <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k}: max |o - o_ref| = {err}"
            errl = np.abs(lse[b, h * G:(h + 1) * G] - ref["lse"]).max()
            assert errl <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k}: max |lse - lse_ref| = {errl}"
    assert n_tie <= max(1, len(bh) * len(top_ks) // 20)


@pytest.mark.parametrize("dims,base", [(64, 10000.0), (32, 500.0)])
def test_tiny_unrotated(dims, base):
    w = synth.WORKLOADS["tiny"]
    _import_case(w, 0, [0, 1, 2, 3], O.Rope(dims, base))


@pytest.mark.parametrize("dims,base", [(128, 1e6), (64, 10000.0), (32, 10000.0)])
def test_8k_unrotated(dims, base):
    w = synth.WORKLOADS["8k"]
    _import_case(w, 0, [w.top_k, 0], O.Rope(dims, base))


@pytest.mark.parametrize("kw", [
    dict(batch=1, n_q_heads=8, n_kv_heads=1, head_dim=128, n_blocks=5, window=37, ranks=(24,), n_residual=5),
    dict(batch=2, n_q_heads=4, n_kv_heads=1, head_dim=64, n_blocks=3, window=9, ranks=(16,), n_residual=3),
    dict(batch=1, n_q_heads=2, n_kv_heads=2, head_dim=128, n_blocks=2, window=0, ranks=(0,), n_residual=0),
    dict(batch=1, n_q_heads=6, n_kv_heads=1, head_dim=128, n_blocks=4, window=256, ranks=(48,), n_residual=128),
])
def test_edge_shapes_unrotated(kw):
    """Ragged windows and residual stages (half groups), rank 0, no window, R = 128."""
    w = synth.Workload("edge", kw["batch"], kw["n_q_heads"], kw["n_kv_heads"], kw["head_dim"], kw["n_blocks"],
                       kw["window"], kw["ranks"], kw["n_residual"], 2, 4, True, 777 + kw["n_blocks"])
    _import_case(w, 0, [0, 1, 2], O.Rope(kw["head_dim"], 10000.0))


def test_64k_unrotated_sampled_units():
    """The 64k layer shape (batch 16, 252 blocks, window 1024, R 128, top-K 16) in the
    launch configuration of the benchmark; two oracle units replicated over the batch."""
    w = synth.WORKLOADS["64k"]
    _import_case(w, 10, [w.top_k], O.Rope(128, 1e6), distinct=2)


def test_rope_tables_hold_the_angles():
    """Page and in-page entries are (cos, sin) of 256 p theta_j and i theta_j."""
    desc = dkv.dkv_layout(1, 2, 1, 128, 3, 100, 8, 4, block_capacity=40, window_capacity=300, rope_dims=64,
                          rope_base=1e6)
    K = torch.randn(1, 1, 3 * 256 + 100, 128, device="cuda").half()
    raw = dkv.dkv_compress_layout(desc, K, K).cpu().numpy()
    page, inpage = LU.unpack_rope_tables(raw, desc)
    theta = 1e6 ** (-2.0 * np.arange(32) / 64)
    assert page.shape[0] == -(-(40 * 256 + 300) // 256)
    a = 256.0 * np.arange(page.shape[0])[:, None] * theta[None, :]
    np.testing.assert_allclose(page[..., 0], np.cos(a), atol=1e-7, rtol=0)
    np.testing.assert_allclose(page[..., 1], np.sin(a), atol=1e-7, rtol=0)
    a = np.arange(256)[:, None] * theta[None, :]
    np.testing.assert_allclose(inpage[..., 0], np.cos(a), atol=1e-7, rtol=0)
    np.testing.assert_allclose(inpage[..., 1], np.sin(a), atol=1e-7, rtol=0)


def _unit_from_cache(raw, desc, u, rope):
    f = lambda x: np.asarray(x, dtype=np.float64)
    blocks = []
    for b in range(desc.n_blocks):
        g = LU.unpack_block(raw, desc, u, b)
        blocks.append(O.Block(a_k=f(g["a_k"]), a_v=f(g["a_v"]), U=f(g["U"]), V_K=f(g["V_K"]), V_V=f(g["V_V"]),
                              S=g["S"], K_res=f(g["K_res"]), V_res=f(g["V_res"]), kmin=f(g["kmin"]),
                              kmax=f(g["kmax"])))
    wk, wv = LU.unpack_window(raw, desc, u)
    return O.Unit(blocks=blocks, win_K=f(wk), win_V=f(wv), rope=rope)


@pytest.mark.parametrize("name,layer,units,dims,base", [
    ("8k", 0, None, 128, 1e6), ("32k", 0, [0, 5], 64, 10000.0), ("64k", 0, [3], 128, 1e6)])
def test_gpu_compressed_unrotated_pool(name, layer, units, dims, base):
    """GPU compression of keys before RoPE: each block's fp32 box is the oracle's box of
    the exact keys rotated to their positions, and the decode of the GPU's own cache
    matches the oracle reading that cache."""
    w = synth.WORKLOADS[name]
    r = w.rank(layer)
    rope = O.Rope(dims, base)
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          rope_dims=dims, rope_base=base)
    K, V = synth.layer_kv_torch(w, layer, torch.device("cuda"))
    cache = dkv.dkv_compress_layout(desc, K, V)
    Kh = K.cpu().numpy()
    del K, V
    raw = cache.cpu().numpy()
    q = synth.queries(w, layer)
    qd = torch.from_numpy(q).cuda()
    out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, w.top_k)
    out, lse, routed = out.cpu().numpy(), lse.cpu().numpy(), routed.cpu().numpy()
    G = w.group
    todo = list(range(w.batch * w.n_kv_heads)) if units is None else units
    for u in todo:
        b, h = divmod(u, w.n_kv_heads)
        unit = _unit_from_cache(raw, desc, u, rope)
        for j in (0, w.n_blocks // 2, w.n_blocks - 1):
            kmin, kmax = O.rope_key_box(Kh[b, h, 256 * j:256 * (j + 1)], j, rope)
            np.testing.assert_allclose(unit.blocks[j].kmin, kmin, atol=2e-5 * (1 + np.abs(kmin).max()), rtol=0)
            np.testing.assert_allclose(unit.blocks[j].kmax, kmax, atol=2e-5 * (1 + np.abs(kmax).max()), rtol=0)
        ref = O.decode_unit(q[b, h * G:(h + 1) * G].astype(np.float64), unit, w.top_k)
        H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
        if set(routed[b, h]) != set(ref["idx"]):
            continue
        assert np.abs(out[b, h * G:(h + 1) * G] - ref["o"]).max() <= H.ATOL_OUT
        assert np.abs(lse[b, h * G:(h + 1) * G] - ref["lse"]).max() <= H.ATOL_OUT


def test_unrotated_and_rotated_pools_differ_where_they_should():
    """rope_dims 0 and a rope_dims > 0 cache of the same tokens give different outputs
    (the rotation is applied), and the un-rotated decode equals the oracle's."""
    w = synth.WORKLOADS["tiny"]
    units = H.oracle_units(w, 0, [(0, 0)], parallel=False)
    runits = H.oracle_units(w, 0, [(0, 0)], parallel=False, rope=O.Rope(64, 10000.0))
    q = synth.queries(w, 0)
    qd = torch.from_numpy(q).cuda()
    outs = []
    for us, kw in ((units, {}), (runits, dict(rope_dims=64, rope_base=10000.0))):
        desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, w.rank(0),
                              w.n_residual, **kw)
        cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(us, w.head_dim, w.rank(0), w.n_residual,
                                                                         w.window)))
        outs.append(dkv.dkv_decode_attend(desc, qd, cache, 0)[0].cpu().numpy())
    assert np.abs(outs[0] - outs[1]).max() > 1e-2
    ref = O.decode_unit(q[0, :1].astype(np.float64), H.round_unit(runits[0]), 0)
    assert np.abs(outs[1][0, :1] - ref["o"]).max() <= H.ATOL_OUT
