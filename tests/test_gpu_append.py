"""Streaming append (dkv_append) on the GPU.

The window rule fixes the whole state: after appending tokens in any pieces,
the cache must hold byte for byte what dkv_compress_layout writes for the whole
token sequence with the final (n_blocks, window) and the same capacities (the
GPU compressor is deterministic and each block depends only on its own 256
tokens).  Decoding the appended cache is checked against the oracle's own
streaming append (which pins to the oracle's batch compression on CPU).
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _tokens(B, Hq, Hkv, d, T, r, R, seed):
    nb = T // 256
    w = synth.Workload("append", B, Hq, Hkv, d, nb, T - nb * 256, (r,), R, 2, 16, True, seed)
    K, V = synth.layer_kv(w, 0)
    return K, V, synth.queries(w, 0)


def _expected_counts(T, cap_w):
    nb = 0 if T <= cap_w else -(-(T - cap_w) // 256)
    return nb, T - 256 * nb


@pytest.mark.parametrize("d,r,R,cap_b,cap_w,T0,chunks", [
    (128, 24, 40, 6, 600, 856, [1, 7, 36, 1, 300, 256, 5]),     # starts with one block and a full window
    (128, 16, 128, 5, 512, 0, [1, 255, 256, 1, 700]),           # starts empty; R = 128
    (64, 8, 16, 4, 300, 300, [1, 1, 254, 300]),                 # d = 64, window starts full
    (128, 48, 5, 3, 256, 100, [156, 1, 255, 3]),                # capacity of exactly one block
])
def test_append_equals_batch_compression(d, r, R, cap_b, cap_w, T0, chunks):
    _append_vs_batch(d, r, R, cap_b, cap_w, T0, chunks, 0)


@pytest.mark.parametrize("d,r,R,cap_b,cap_w,T0,chunks,rope_dims", [
    (128, 24, 40, 6, 600, 856, [1, 7, 36, 1, 300, 256, 5], 128),   # keys before RoPE, every channel rotated
    (128, 16, 128, 5, 512, 0, [1, 255, 256, 1, 700], 64),           # starts empty: the first append writes the tables
    (64, 8, 16, 4, 300, 300, [1, 1, 254, 300], 32),                  # partial RoPE at d = 64
])
def test_append_into_an_unrotated_pool_equals_batch_compression(d, r, R, cap_b, cap_w, T0, chunks, rope_dims):
    """The same byte identity for an un-rotated pool: its blocks' boxes are taken over the
    keys rotated to the positions the tokens keep when they leave the window."""
    _append_vs_batch(d, r, R, cap_b, cap_w, T0, chunks, 0, rope_dims)


@pytest.mark.parametrize("bits", [8, 4])
def test_append_with_quantised_residuals_equals_batch_compression(bits):
    """The same byte identity when the residual rows are stored group-quantised."""
    _append_vs_batch(128, 24, 40, 6, 600, 856, [1, 7, 36, 1, 300, 256, 5], bits)
    _append_vs_batch(64, 8, 16, 4, 300, 300, [1, 1, 254, 300], bits)


def _append_vs_batch(d, r, R, cap_b, cap_w, T0, chunks, bits, rope_dims=0):
    B, Hq, Hkv = 2, 6, 2
    rope = dict(rope_dims=rope_dims, rope_base=10000.0 if rope_dims else 0.0)
    T = T0 + sum(chunks)
    K, V, _ = _tokens(B, Hq, Hkv, d, T, r, R, 321 + T)
    Kd, Vd = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    nb0, w0 = _expected_counts(T0, cap_w)
    desc = dkv.dkv_layout(B, Hq, Hkv, d, nb0, w0, r, R, block_capacity=cap_b, window_capacity=cap_w,
                          residual_bits=bits, **rope)
    ws = torch.zeros(max(dkv.dkv_append_workspace_bytes(desc), dkv.dkv_compress_workspace_bytes(desc), 256),
                     dtype=torch.uint8, device="cuda")
    cache = torch.empty(desc.total_bytes, dtype=torch.uint8, device="cuda")
    if T0:
        dkv.dkv_compress_layout(desc, Kd[:, :, :T0].contiguous(), Vd[:, :, :T0].contiguous(), cache=cache,
                                workspace=ws)
    else:
        cache.zero_()
    t = T0
    for n in chunks:
        dkv.dkv_append(desc, Kd[:, :, t:t + n].contiguous(), Vd[:, :, t:t + n].contiguous(), cache, workspace=ws)
        t += n
        assert (desc.n_blocks, desc.window) == _expected_counts(t, cap_w)
    torch.cuda.synchronize()
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK, f"device error word {word:#x}"
    ref_desc = dkv.dkv_layout(B, Hq, Hkv, d, desc.n_blocks, desc.window, r, R, block_capacity=cap_b,
                              window_capacity=cap_w, residual_bits=bits, **rope)
    assert bytes(ref_desc) == bytes(desc)
    ref = dkv.dkv_compress_layout(ref_desc, Kd, Vd, workspace=ws)
    torch.cuda.synchronize()
    diff = (cache != ref).nonzero()
    assert diff.numel() == 0, f"{diff.numel()} bytes differ, first at {diff[0].item()}"


def test_append_then_decode_matches_the_oracle_stream():
    """Decode parity on an appended cache: the oracle runs its own streaming
    append over the same tokens, then decodes by the plain definition."""
    B, Hq, Hkv, d, r, R, cap_b, cap_w = 1, 12, 2, 128, 32, 40, 4, 640
    T0, chunks = 300, [1, 339, 1, 400, 3]
    T = T0 + sum(chunks)
    K, V, q = _tokens(B, Hq, Hkv, d, T, r, R, 99)
    Kd, Vd = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    desc = dkv.dkv_layout(B, Hq, Hkv, d, 0, T0, r, R, block_capacity=cap_b, window_capacity=cap_w)
    cache = dkv.dkv_compress_layout(desc, Kd[:, :, :T0].contiguous(), Vd[:, :, :T0].contiguous())
    units = [O.compress_unit(K[0, h, :T0], V[0, h, :T0], 0, r, R) for h in range(Hkv)]
    t = T0
    for n in chunks:
        dkv.dkv_append(desc, Kd[:, :, t:t + n].contiguous(), Vd[:, :, t:t + n].contiguous(), cache)
        units = [O.append_tokens(units[h], K[0, h, t:t + n], V[0, h, t:t + n], cap_w, r, R) for h in range(Hkv)]
        t += n
    assert desc.n_blocks == len(units[0].blocks) == 2 and desc.window == len(units[0].win_K)
    G = Hq // Hkv
    for top_k in (1, 0):
        out, lse, routed = dkv.dkv_decode_attend(desc, torch.from_numpy(q).cuda(), cache, top_k)
        out, lse = out.cpu().numpy(), lse.cpu().numpy()
        for h in range(Hkv):
            ref = O.decode_unit(q[0, h * G:(h + 1) * G].astype(np.float64), units[h], top_k)
            # both sides compress on their own: allow what fp16 storage of the factors costs
            ref16 = O.decode_unit(q[0, h * G:(h + 1) * G].astype(np.float64), H.round_unit(units[h]), top_k)
            storage = np.abs(ref16["o"] - ref["o"]).max()
            if routed is not None and top_k == 1:
                H.check_routing(routed.cpu().numpy()[0, h], ref["idx"], ref["bounds"])
            err = np.abs(out[0, h * G:(h + 1) * G] - ref["o"]).max()
            assert err <= H.ATOL_OUT + 4 * storage, f"head {h} top_k {top_k}: {err} (storage {storage})"


def test_append_rejects_what_does_not_fit():
    desc = dkv.dkv_layout(1, 6, 1, 64, 1, 300, 8, 4, block_capacity=1, window_capacity=300)
    cache = torch.zeros(desc.total_bytes, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 1, 1, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_append(desc, x, x, cache)  # the full window would need a second block
    assert e.value.status == dkv.DKV_ERR_UNSUPPORTED
    assert (desc.n_blocks, desc.window) == (1, 300)
