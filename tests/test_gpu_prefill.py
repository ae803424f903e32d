"""GPU parity of block-sparse prefill (dkv_prefill_attend) against the fp64 oracle.

Both sides take the same fp16 q, K, V.  Routed blocks must match the oracle's
exactly, except blocks whose oracle bound lies within 1e-4 of the K-th bound
(the block-mean query is an fp32 sum on the GPU, an fp64 one in the oracle);
outputs and lse within 2e-3 for every query block whose routed set matches.
"""
import math

import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu
BS = O.BLOCK_SIZE


def _inputs(B, Hq, Hkv, d, T, seed):
    nb = T // BS
    w = synth.Workload("prefill", B, Hq, Hkv, d, nb, T - nb * BS, (8,), 8, 2, 16, True, seed)
    K, V = synth.layer_kv(w, 0)
    q = np.random.default_rng(seed).standard_normal((B, Hq, T, d)).astype(np.float16)
    return q, K, V


def _check_routes(gpu_routed, ref_routes, ref_bounds, top_k):
    """Per query block: the GPU's routed list against the oracle's (tie band); returns
    the query blocks whose sets agree."""
    agree = []
    for i, (ref, bounds) in enumerate(zip(ref_routes, ref_bounds)):
        got = [int(x) for x in gpu_routed[i] if x >= 0]
        assert got == sorted(got) and len(set(got)) == len(got)
        assert len(got) == len(ref), (i, got, list(ref))
        if set(got) == set(int(x) for x in ref):
            agree.append(i)
            continue
        kth = np.sort(bounds)[::-1][len(ref) - 1]
        for j in set(got) ^ set(int(x) for x in ref):
            assert abs(bounds[j] - kth) <= H.TIE_BAND, f"block {i}: routed {j} (bound {bounds[j]}, K-th {kth})"
    return agree


@pytest.mark.parametrize("B,Hq,Hkv,d,T,top_k", [
    (1, 6, 1, 64, 37, 1), (1, 6, 1, 64, 256, 1), (1, 6, 1, 64, 700, 1), (1, 6, 1, 64, 1100, 2),
    (2, 4, 2, 64, 1300, 0), (1, 12, 2, 128, 2148, 3), (1, 1, 1, 128, 1536, 2), (1, 8, 1, 128, 800, 4),
    (1, 12, 2, 128, 4096, 4)])
def test_prefill_matches_the_oracle(B, Hq, Hkv, d, T, top_k):
    q, K, V = _inputs(B, Hq, Hkv, d, T, 100 + T + top_k)
    out, lse, routed = dkv.dkv_prefill_attend(torch.from_numpy(q).cuda(), torch.from_numpy(K).cuda(),
                                              torch.from_numpy(V).cuda(), top_k)
    out, lse, routed = out.cpu().numpy(), lse.cpu().numpy(), routed.cpu().numpy()
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            ref = O.prefill_unit(q[b, h * G:(h + 1) * G].astype(np.float64), K[b, h], V[b, h], top_k)
            agree = _check_routes(routed[b, h], ref["routes"], ref["bounds"], top_k)
            for i in agree:
                t0, t1 = i * BS, min(T, (i + 1) * BS)
                err = np.abs(out[b, h * G:(h + 1) * G, t0:t1] - ref["o"][:, t0:t1]).max()
                errl = np.abs(lse[b, h * G:(h + 1) * G, t0:t1] - ref["lse"][:, t0:t1]).max()
                assert err <= H.ATOL_OUT, f"unit {(b, h)} block {i}: max |o - o_ref| = {err}"
                assert errl <= H.ATOL_OUT, f"unit {(b, h)} block {i}: max |lse - lse_ref| = {errl}"
            assert len(agree) >= len(ref["routes"]) - 1


def test_prefill_32k_sampled_tokens():
    """The Qwen2.5-1.5B-shaped layer at 32k (12 q / 2 KV heads, d 128, top-K 16): routes of
    every query block, outputs of sampled tokens (the oracle's routes and one softmax per token)."""
    B, Hq, Hkv, d, T, top_k = 1, 12, 2, 128, 32768, 16
    q, K, V = _inputs(B, Hq, Hkv, d, T, 32)
    out, lse, routed = dkv.dkv_prefill_attend(torch.from_numpy(q).cuda(), torch.from_numpy(K).cuda(),
                                              torch.from_numpy(V).cuda(), top_k)
    out, lse, routed = out.cpu().numpy(), lse.cpu().numpy(), routed.cpu().numpy()
    G = Hq // Hkv
    rng = np.random.default_rng(3)
    for h in range(Hkv):
        Qh = q[0, h * G:(h + 1) * G].astype(np.float64)
        routes = O.prefill_routes(Qh, K[0, h], top_k)
        agree = _check_routes(routed[0, h], [r for r, _ in routes], [b for _, b in routes], top_k)
        for t in sorted(set(rng.integers(0, T, 24).tolist()) | {0, 255, 256, T - 1}):
            i = t // BS
            if i not in agree:
                continue
            keys = np.concatenate([np.arange(j * BS, (j + 1) * BS) for j in routes[i][0]] + [np.arange(i * BS, t + 1)])
            o, l = O.softmax_attention(Qh[:, t, :], K[0, h, keys].astype(np.float64), V[0, h, keys].astype(np.float64))
            assert np.abs(out[0, h * G:(h + 1) * G, t] - o).max() <= H.ATOL_OUT, (h, t)
            assert np.abs(lse[0, h * G:(h + 1) * G, t] - l).max() <= H.ATOL_OUT, (h, t)


def test_prefill_validation():
    x = torch.zeros(1, 6, 300, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_prefill_attend(x, x[:, :1], x[:, :1], -1)
    assert e.value.status == dkv.DKV_ERR_ARG
    y = torch.zeros(1, 6, 300, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_prefill_attend(y, y[:, :1], y[:, :1], 1)
    assert e.value.status == dkv.DKV_ERR_UNSUPPORTED
