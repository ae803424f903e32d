"""Dense fp16 decode attention (dkv_dense_decode) against the oracle's plain
softmax attention over the same fp16 K, V, q.

The dense kernel is the bytes/throughput reference of the compressed path
(the dense full-KV baselines of the DKV Zenodo abstract).  Outputs must match
the fp64 definition within the decode tolerance (fp16 operands, fp32
accumulation); lse within 1e-3 (natural log).
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _check(q, K, V, out, lse, units):
    B, Hkv, T, d = K.shape
    G = q.shape[1] // Hkv
    worst = 0.0
    for b, h in units:
        ref_o, ref_l = O.softmax_attention(q[b, h * G:(h + 1) * G], K[b, h], V[b, h])
        err = np.abs(out[b, h * G:(h + 1) * G] - ref_o).max()
        worst = max(worst, err)
        assert err <= H.ATOL_OUT, f"unit ({b}, {h}): max |out - oracle| = {err}"
        np.testing.assert_allclose(lse[b, h * G:(h + 1) * G], ref_l, atol=1e-3, rtol=0)
    return worst


def _random_case(seed, B, Hq, Hkv, d, T):
    rng = np.random.default_rng(seed)
    K = (rng.standard_normal((B, Hkv, T, d)) * 2.0).astype(np.float16)
    V = rng.standard_normal((B, Hkv, T, d)).astype(np.float16)
    # a few outlier rows, as in the synthetic cache
    rows = rng.random((B, Hkv, T)) < 0.01
    K[rows] *= np.float16(8)
    V[rows] *= np.float16(8)
    q = rng.standard_normal((B, Hq, d)).astype(np.float16)
    return q, K, V


@pytest.mark.parametrize("B,Hq,Hkv,d,T", [
    (1, 1, 1, 64, 1),          # a single token
    (1, 1, 1, 64, 7),          # ragged, below one tile
    (1, 6, 1, 128, 64),        # exactly one tile
    (2, 12, 2, 128, 100),      # ragged tail
    (1, 8, 1, 128, 1000),      # G = 8, several chunks
    (1, 3, 1, 64, 4096),       # d = 64, odd group
    (3, 4, 4, 128, 777),       # G = 1, several units
])
def test_dense_matches_softmax_attention(B, Hq, Hkv, d, T):
    q, K, V = _random_case(B * 1000 + T, B, Hq, Hkv, d, T)
    out, lse = dkv.dkv_dense_decode(torch.from_numpy(q).cuda(), torch.from_numpy(K).cuda(),
                                    torch.from_numpy(V).cuda())
    _check(q, K, V, out.cpu().numpy(), lse.cpu().numpy(), [(b, h) for b in range(B) for h in range(Hkv)])


def test_dense_sweep16k_full_launch_sampled_units():
    """The 16k sweep's dense reference shape (batch 64, 12q/2kv, d 128, T 16384),
    inputs drawn on the device by the synthetic generator; sampled units checked."""
    w = synth.WORKLOADS["sweep16k"]
    K, V = synth.layer_kv_torch(w, 0, "cuda")
    q = torch.from_numpy(synth.queries(w, 0)).cuda()
    out, lse = dkv.dkv_dense_decode(q, K, V)
    units = [(0, 0), (31, 1), (63, 1)]
    Kh = np.stack([K[b, h].cpu().numpy() for b, h in units])
    Vh = np.stack([V[b, h].cpu().numpy() for b, h in units])
    qh, oh, lh = q.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    G = w.group
    for i, (b, h) in enumerate(units):
        ref_o, ref_l = O.softmax_attention(qh[b, h * G:(h + 1) * G], Kh[i], Vh[i])
        err = np.abs(oh[b, h * G:(h + 1) * G] - ref_o).max()
        assert err <= H.ATOL_OUT, f"unit ({b}, {h}): {err}"
        np.testing.assert_allclose(lh[b, h * G:(h + 1) * G], ref_l, atol=1e-3, rtol=0)


def test_dense_equals_full_rank_compressed_path():
    """The compressed path with every row exact (R = 255) and every block routed
    attends exactly the same tokens: both must agree with each other too."""
    w = synth.WORKLOADS["8k"].with_(batch=1)
    K, V = synth.layer_kv(w, 0)
    q = synth.queries(w, 0)
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, 8, 255)
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    o_c, l_c, _ = dkv.dkv_decode_attend(desc, torch.from_numpy(q).cuda(), cache, 0)
    o_d, l_d = dkv.dkv_dense_decode(torch.from_numpy(q).cuda(), torch.from_numpy(K).cuda(),
                                    torch.from_numpy(V).cuda())
    assert (o_c - o_d).abs().max().item() <= 2 * H.ATOL_OUT
    assert (l_c - l_d).abs().max().item() <= 2e-3


def test_dense_rejects_bad_arguments():
    q = torch.zeros(1, 3, 64, dtype=torch.float16, device="cuda")
    K = torch.zeros(1, 2, 16, 64, dtype=torch.float16, device="cuda")  # 3 q heads over 2 kv heads
    with pytest.raises(dkv.DkvError):
        dkv.dkv_dense_decode(q, K, K)
    q = torch.zeros(1, 2, 96, dtype=torch.float16, device="cuda")
    K = torch.zeros(1, 1, 16, 96, dtype=torch.float16, device="cuda")  # head_dim 96
    with pytest.raises(dkv.DkvError):
        dkv.dkv_dense_decode(q, K, K)
