"""Routing on the GPU against the oracle's router ("Decode router bounds" of
the Differential-KV README's per-block memory table; DKV_TOPK_BLOCKS and
DKV_CB_GQA_ROUTE, README "Key Environment Knobs"), at block counts the other
parity tests do not reach (1000 and 1100 blocks: 125 and 138 blocks for each
CTA of the router's 8-CTA cluster).

The cache comes from the GPU compressor (the router rows are the exact fp16
key minima and maxima, so both sides bound the same keys).  Routed indices
must equal the oracle's except inside the 1e-4 tie band of the K-th bound;
dkv_decode_attend and the stage call dkv_decode_route must agree bit for bit.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_blocks, top_ks", [(1000, [1, 7, 300, 999]), (1100, [5, 600])])
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
