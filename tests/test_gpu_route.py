"""Routing on the GPU against the oracle's router ("Decode router bounds" of
the Differential-KV README's per-block memory table; DKV_TOPK_BLOCKS and
DKV_CB_GQA_ROUTE, README "Key Environment Knobs"), at block counts the other
parity tests do not reach (1000, 1100 and the 2048-block limit: 125, 138 and
256 blocks for each CTA of the router's 8-CTA cluster).

The cache comes from the GPU compressor (the router rows are the exact fp16
key minima and maxima, so both sides bound the same keys).  Routed indices
must equal the oracle's except inside the 1e-4 tie band of the K-th bound;
dkv_decode_attend and the stage call dkv_decode_route must agree bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_blocks, top_ks", [(1000, [1, 7, 300, 999]), (1100, [5, 600]), (2048, [1, 16, 2047])])
def test_routing_at_large_block_counts(n_blocks, top_ks):
    d, G, B, Hkv = 64, 6, 1, 2
    w = synth.Workload("route", B, G * Hkv, Hkv, d, n_blocks, 16, (8,), 8, 2, 4, False, 11)
    desc = dkv.dkv_layout(B, G * Hkv, Hkv, d, n_blocks, 16, 8, 8)
    K, V = synth.layer_kv(w, 0)
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    q = synth.queries(w, 0)
    qd = torch.from_numpy(q).cuda()
    for top_k in top_ks:
        assert dkv.dkv_decode_launches(desc, top_k) == 3  # router, attention, combine
        _, _, routed = dkv.dkv_decode_attend(desc, qd, cache, top_k)
        ws = torch.zeros(dkv.dkv_decode_workspace_bytes(desc, top_k), dtype=torch.uint8, device="cuda")
        staged = torch.empty(B, Hkv, O.effective_top_k(top_k, n_blocks), dtype=torch.int32, device="cuda")
        dkv.dkv_decode_route(desc, qd, cache, top_k, ws, routed=staged)
        torch.cuda.synchronize()
        assert torch.equal(routed, staged), f"top_k {top_k}: dkv_decode_attend and dkv_decode_route differ"
        routed = routed.cpu().numpy()
        for b in range(B):
            for h in range(Hkv):
                Kb = K[b, h, :n_blocks * 256].astype(np.float64).reshape(n_blocks, 256, d)
                bounds = O.router_bounds(q[b, h * G:(h + 1) * G], Kb.min(axis=1), Kb.max(axis=1))
                H.check_routing(routed[b, h], O.route(bounds, top_k), bounds)
    assert dkv.dkv_decode_launches(desc, 0) == 2  # every block routed: no router grid


def test_equal_bounds_route_the_lowest_blocks_in_both_paths():
    """Every block of a unit gets block 0's key box, so all router bounds are equal
    and (score desc, index asc) routes blocks 0 .. K-1.  Both router outputs must
    decode exactly those blocks: the ascending list written when the caller asks
    for the indices, and the rank slots written without a copy.  A rank shared by
    two blocks would leave a slot of a fresh (zeroed) list at block 0, which would
    then count twice."""
    w = synth.WORKLOADS["8k"]
    G = w.group
    units = []
    for un in H.oracle_units(w, 0, [(0, 0), (0, 1)]):
        b0 = un.blocks[0]
        blocks = [dataclasses.replace(b, kmin=b0.kmin.copy(), kmax=b0.kmax.copy()) for b in un.blocks]
        units.append(O.Unit(blocks=blocks, win_K=un.win_K, win_V=un.win_V))
    rounded = [H.round_unit(u) for u in units]
    desc = dkv.dkv_layout(1, w.n_q_heads, 2, 128, w.n_blocks, w.window, 32, 40)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, 128, 32, 40, w.window)))
    q = synth.queries(w, 0)
    qd = torch.from_numpy(q).cuda()
    for top_k in (1, 5, 8, 17):
        k_eff = O.effective_top_k(top_k, w.n_blocks)
        fresh = lambda: torch.zeros(dkv.dkv_decode_workspace_bytes(desc, top_k), dtype=torch.uint8, device="cuda")
        out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, top_k, workspace=fresh())
        out_ns, lse_ns, _ = dkv.dkv_decode_attend(desc, qd, cache, top_k, routed=False, workspace=fresh())
        torch.cuda.synchronize()
        for h in range(2):
            ref = O.decode_unit(q[0, h * G:(h + 1) * G].astype(np.float64), rounded[h], top_k)
            assert list(ref["idx"]) == list(range(k_eff))
            assert routed[0, h].tolist() == list(range(k_eff))
            for o_, l_, path in ((out, lse, "ascending"), (out_ns, lse_ns, "rank slots")):
                err = np.abs(o_[0, h * G:(h + 1) * G].cpu().numpy() - ref["o"]).max()
                errl = np.abs(l_[0, h * G:(h + 1) * G].cpu().numpy() - ref["lse"]).max()
                assert err <= H.ATOL_OUT, f"top_k {top_k} head {h} ({path}): max |o - o_ref| = {err}"
                assert errl <= H.ATOL_OUT, f"top_k {top_k} head {h} ({path}): max |lse - lse_ref| = {errl}"
