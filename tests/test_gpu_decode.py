"""GPU parity of dkv_decode_attend against the fp64 oracle (through the C ABI).

The oracle compresses each unit in fp64; its factors are rounded to fp16 (the
stored operands), imported into the packed cache with dkv_import_factors, and
both sides decode the same fp16 operands: the oracle in fp64 by definition
(materialised tokens, one softmax), the GPU with its kernels.  Routed block
indices must match exactly except inside the 1e-4 tie band of the K-th
bound; outputs and log-sum-exp must agree within 2e-3 (max abs).
"""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _run_case(w: synth.Workload, layer: int, top_ks, distinct: int | None = None, units_override=None,
              layout: int = dkv.DKV_LAYOUT_FRAGMENT):
    """Import oracle factors for every unit of `w` (optionally replicating `distinct`
    oracle-compressed units across the batch), decode on the GPU, compare all units.
    `layout` picks the cache byte order and with it the decode kernel (mma.sync or tcgen05)."""
    r = w.rank(layer)
    bh = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    n_units = len(bh)
    if units_override is not None:
        base_units = units_override
    else:
        todo = bh if distinct is None else bh[:distinct]
        base_units = H.oracle_units(w, layer, todo)
    units = [base_units[i % len(base_units)] for i in range(n_units)]
    rounded = [H.round_unit(u) for u in base_units]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          layout=layout)
    arrs = H.factor_arrays(units, w.head_dim, r, w.n_residual, w.window)
    cache = dkv.dkv_import_factors(desc, H.to_device(arrs))
    q = synth.queries(w, layer)
    qd = torch.from_numpy(q).cuda()
    G = w.group
    worst = 0.0
    n_tie = 0
    ws = torch.zeros(max(dkv.dkv_decode_workspace_bytes(desc, k) for k in top_ks), dtype=torch.uint8, device="cuda")
    for top_k in top_ks:
        out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, top_k, workspace=ws)
        # without a copy of the indices the router puts each block in its rank's slot
        # (another block order, the same blocks): the path the benchmark times
        out_ns, lse_ns, _ = dkv.dkv_decode_attend(desc, qd, cache, top_k, routed=False, workspace=ws)
        torch.cuda.synchronize()
        # no bounded wait gave up, not even one that only delays the exit (outputs stay right then)
        st, word = dkv.dkv_get_error(ws)
        assert st == dkv.DKV_OK and word == 0, f"top_k {top_k}: device error word {word:#x}"
        out, lse = out.cpu().numpy(), lse.cpu().numpy()
        out_ns, lse_ns = out_ns.cpu().numpy(), lse_ns.cpu().numpy()
        routed = routed.cpu().numpy() if routed is not None else None
        for i, (b, h) in enumerate(bh):
            qg = q[b, h * G:(h + 1) * G].astype(np.float64)
            ref = O.decode_unit(qg, rounded[i % len(rounded)], top_k)
            if routed is not None:
                H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
                if set(routed[b, h]) != set(ref["idx"]):
                    n_tie += 1
                    continue
            for o_, l_, path in ((out, lse, "ascending"), (out_ns, lse_ns, "rank slots")):
                err = np.abs(o_[b, h * G:(h + 1) * G] - ref["o"]).max()
                errl = np.abs(l_[b, h * G:(h + 1) * G] - ref["lse"]).max()
                worst = max(worst, err, errl)
                assert err <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k} ({path}): max |o - o_ref| = {err}"
                assert errl <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k} ({path}): max |lse - lse_ref| = {errl}"
    assert n_tie <= max(1, n_units * len(top_ks) // 20)
    return worst


def test_tiny():
    w = synth.WORKLOADS["tiny"]
    _run_case(w, 0, [w.top_k, 0, 1, 3])


TC = dkv.DKV_LAYOUT_TC
LAYOUTS = [dkv.DKV_LAYOUT_FRAGMENT, TC]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_8k(layout):
    w = synth.WORKLOADS["8k"]
    _run_case(w, 0, [w.top_k, 0], layout=layout)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_32k(layout):
    w = synth.WORKLOADS["32k"]
    _run_case(w, 0, [w.top_k], layout=layout)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("layer", [0, 10, 27])
def test_64k_full_launch_sampled_units(layer, layout):
    """Full 64k launch (batch 16, 32 units, R=128, W=1024) with the layer's rank;
    two oracle-compressed units are replicated over the batch (queries differ per
    unit), and every unit is checked against the oracle."""
    w = synth.WORKLOADS["64k"]
    _run_case(w, layer, [w.top_k], distinct=2, layout=layout)


def test_sweep16k_full_launch_sampled_units():
    w = synth.WORKLOADS["sweep16k"]
    _run_case(w, 0, list(synth.SWEEP_TOP_K), distinct=4)


# ---------------------------------------------------------------- edge cases on small shapes

def _small(d=64, G=6, nb=3, W=100, r=16, R=24, B=1, Hkv=1, seed=7, latent=4):
    return synth.Workload("edge", B, G * Hkv, Hkv, d, nb, W, (r,), R, 2, latent, False, seed)


@pytest.mark.parametrize("kw", [
    dict(), dict(r=0), dict(R=0), dict(R=255), dict(r=8, R=8), dict(r=24, R=40), dict(W=0), dict(nb=0, W=300),
    dict(W=17), dict(W=1), dict(G=1), dict(G=8), dict(G=3), dict(d=128), dict(d=128, r=48, R=128, W=1024),
    dict(d=128, r=104, R=5), dict(d=64, r=128, R=0), dict(B=2, Hkv=2, nb=5),
    dict(nb=1, W=65536),  # the largest window the layout accepts
])
def test_edge_shapes(kw):
    w = _small(**kw)
    tks = [0, 1, 2, w.n_blocks + 3] if w.n_blocks else [0, 4]
    _run_case(w, 0, tks)


@pytest.mark.parametrize("kw", [
    dict(), dict(r=8, R=8), dict(r=1, R=1), dict(r=48, R=128, W=1024), dict(W=0), dict(nb=0, W=300),
    dict(W=17), dict(W=1), dict(W=129), dict(G=1), dict(G=8), dict(G=3), dict(B=2, Hkv=2, nb=5),
    dict(r=40, R=100, W=700, nb=9),
])
def test_edge_shapes_tensor_core_layout(kw):
    """The tcgen05 decode kernel: head_dim 128; ragged windows across its 128-token
    groups, every group size, one-row residual sets, a rank that fills one plane."""
    w = _small(**dict(dict(d=128), **kw))
    tks = [0, 1, 2, w.n_blocks + 3] if w.n_blocks else [0, 4]
    _run_case(w, 0, tks, layout=TC)


def test_full_rank_matches_dense_attention():
    """d=64, r = 2d = 128 (full rank of the joint deltas), R = 0, all blocks
    routed: the GPU output equals dense softmax attention over the exact K, V
    up to the fp16 storage of U and the basis."""
    w = _small(d=64, r=128, R=0, nb=2, W=64)
    K, V = synth.unit_kv(w, 0, 0, 0)
    unit = O.compress_unit(K, V, w.n_blocks, 128, 0)
    q = synth.queries(w, 0)
    _run_case(w, 0, [0], units_override=[unit])
    qg = q[0].astype(np.float64)
    o_dense, _ = O.softmax_attention(qg, K.astype(np.float64), V.astype(np.float64))
    o_fp16 = O.decode_unit(qg, H.round_unit(unit), 0)["o"]
    desc = dkv.dkv_layout(1, w.n_q_heads, 1, 64, w.n_blocks, w.window, 128, 0)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays([unit], 64, 128, 0, w.window)))
    out, _, _ = dkv.dkv_decode_attend(desc, torch.from_numpy(q).cuda(), cache, 0)
    storage = np.abs(o_fp16 - o_dense).max()  # what fp16 storage of the factors alone costs
    assert np.abs(out.cpu().numpy()[0] - o_dense).max() <= 2 * storage + H.ATOL_OUT


def test_errors_are_reported_not_launched():
    w = _small()
    desc = dkv.dkv_layout(1, 6, 1, 64, 3, 100, 16, 24)
    q = torch.zeros(1, 6, 64, dtype=torch.float16, device="cuda")
    cache = torch.zeros(desc.total_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_decode_attend(desc, q, cache, -1)
    assert e.value.status == dkv.DKV_ERR_ARG
    small_ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_decode_attend(desc, q, cache, 2, workspace=small_ws)
    assert e.value.status == dkv.DKV_ERR_WORKSPACE
    # misaligned output pointer
    out = torch.empty(1 * 6 * 64 + 1, dtype=torch.float32, device="cuda")[1:].view(1, 6, 64)
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_decode_attend(desc, q, cache, 2, out=out)
    assert e.value.status == dkv.DKV_ERR_ALIGN


def test_bad_residual_positions_raise_index_error():
    w = _small()
    units = H.oracle_units(w, 0, [(0, 0)], parallel=False)
    arrs = H.factor_arrays(units, 64, 16, 24, 100)
    arrs["res_pos"][0, 1, 3] = arrs["res_pos"][0, 1, 2]  # not strictly ascending
    desc = dkv.dkv_layout(1, 6, 1, 64, 3, 100, 16, 24)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dkv.dkv_import_factors(desc, H.to_device(arrs), workspace=ws)
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_ERR_DEVICE and word & dkv.DKV_DEVERR_INDEX
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK and word == 0


def test_decode_is_deterministic_and_stream_ordered():
    w = synth.WORKLOADS["8k"]
    units = H.oracle_units(w, 0, [(0, 0), (0, 1)])
    desc = dkv.dkv_layout(1, 12, 2, 128, w.n_blocks, w.window, 32, 40)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, 128, 32, 40, w.window)))
    q = torch.from_numpy(synth.queries(w, 0)).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = [dkv.dkv_decode_attend(desc, q, cache, 8)[0].clone() for _ in range(3)]
    s.synchronize()
    for x in a[1:]:
        assert torch.equal(x, a[0])


@pytest.mark.parametrize("layout", LAYOUTS)
def test_stage_calls_equal_the_fused_call_and_reuse_the_workspace(layout):
    """route -> blocks (partials only) -> combine equals dkv_decode_attend (routing
    and merge in the attention grid); one workspace serves many calls of
    different top-K values, since every call leaves its arrival counters at zero."""
    w = synth.WORKLOADS["8k"]
    units = H.oracle_units(w, 0, [(0, 0), (0, 1)])
    desc = dkv.dkv_layout(1, 12, 2, 128, w.n_blocks, w.window, 32, 40, layout=layout)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, 128, 32, 40, w.window)))
    q = torch.from_numpy(synth.queries(w, 0)).cuda()
    ws = torch.zeros(dkv.dkv_decode_workspace_bytes(desc, 0), dtype=torch.uint8, device="cuda")
    for top_k in (8, 3, 0, 8, 30, 1):
        fused, fl, fr = dkv.dkv_decode_attend(desc, q, cache, top_k, workspace=ws)
        k_eff = w.n_blocks if top_k in (0, w.n_blocks) else top_k
        routed = torch.empty(1, 2, k_eff, dtype=torch.int32, device="cuda")
        dkv.dkv_decode_route(desc, q, cache, top_k, ws, routed=routed)
        dkv.dkv_decode_blocks(desc, q, cache, top_k, ws)
        out = torch.empty_like(fused)
        lse = torch.empty_like(fl)
        dkv.dkv_decode_combine(desc, top_k, out, ws, lse=lse)
        torch.cuda.synchronize()
        assert torch.equal(routed, fr)
        # the one-grid call merges the partial records in another order than the combine
        # kernel: fp32 reassociation over n records moves a result by at most about
        # n * 2^-24 of its magnitude (n = 96 here)
        assert torch.allclose(out, fused, rtol=1e-5, atol=1e-5)
        assert torch.allclose(lse, fl, rtol=1e-5, atol=1e-5)
        # the stage route without a copy of the indices writes the rank slots instead
        dkv.dkv_decode_route(desc, q, cache, top_k, ws)
        dkv.dkv_decode_blocks(desc, q, cache, top_k, ws)
        dkv.dkv_decode_combine(desc, top_k, out, ws, lse=lse)
        torch.cuda.synchronize()
        assert torch.allclose(out, fused, rtol=1e-5, atol=1e-5)
        assert torch.allclose(lse, fl, rtol=1e-5, atol=1e-5)
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK and word == 0
