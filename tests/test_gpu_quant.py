"""GPU parity of group-quantised residual rows (residual_bits 8 and 4).

The README's "Physical 4-Bit Group-Quantized Residual Buffers" ("Core
Innovations", item 2) stores each exact residual key row and value row as
codes with an fp16 scale and bias per 64 channels, dequantised in registers
at decode.  Checks:

* the codes, scales and biases the GPU writes (from imported factors, and
  from its own compression) equal the oracle's quantisation of the same fp16
  rows bit for bit (the code is an integer decision both sides take in fp32);
* the decode over quantised residuals matches the oracle decoding the same
  quantised rows (dequantised in fp64) within 2e-3, routed indices exact
  outside the 1e-4 tie band.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H
from tests import layout_unpack as LU

pytestmark = pytest.mark.gpu


def _quant_unit(u: O.Unit, bits: int) -> O.Unit:
    return O.Unit(blocks=[O.quantize_block_residuals(b, bits) for b in u.blocks], win_K=u.win_K, win_V=u.win_V)


def _check_codes(raw, desc, unit_index, blk_index, rows_k, rows_v, bits):
    got = LU.unpack_block(raw, desc, unit_index, blk_index)
    for name, rows in (("K", rows_k), ("V", rows_v)):
        c, s, b = O.quantize_groups(rows, bits)
        assert np.array_equal(got[name + "_codes"], c), f"{name} codes differ in block {blk_index}"
        assert np.array_equal(got[name + "_scale"].view(np.uint16), s.view(np.uint16)), f"{name} scales differ"
        assert np.array_equal(got[name + "_bias"].view(np.uint16), b.view(np.uint16)), f"{name} biases differ"


def _run(w, layer, top_ks, bits, distinct=None):
    r = w.rank(layer)
    bh = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    todo = bh if distinct is None else bh[:distinct]
    base = H.oracle_units(w, layer, todo)
    units = [base[i % len(base)] for i in range(len(bh))]
    rounded = [H.round_unit(u) for u in base]
    qref = [_quant_unit(u, bits) for u in rounded]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          residual_bits=bits)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, w.head_dim, r, w.n_residual, w.window)))
    raw = cache.cpu().numpy()
    if w.n_residual and w.n_blocks:
        for i in range(min(2, len(rounded))):
            for b in sorted({0, w.n_blocks - 1}):
                blk = rounded[i].blocks[b]
                _check_codes(raw, desc, i, b, blk.K_res, blk.V_res, bits)
    q = synth.queries(w, layer)
    qd = torch.from_numpy(q).cuda()
    G = w.group
    n_tie = 0
    for top_k in top_ks:
        for want_routed in (True, False):
            out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, top_k, routed=want_routed)
            out, lse = out.cpu().numpy(), lse.cpu().numpy()
            routed = routed.cpu().numpy() if routed is not None else None
            for i, (b, h) in enumerate(bh):
                ref = O.decode_unit(q[b, h * G:(h + 1) * G].astype(np.float64), qref[i % len(qref)], top_k)
                if routed is not None:
                    H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
                    if set(routed[b, h]) != set(ref["idx"]):
                        n_tie += 1
                        continue
                err = np.abs(out[b, h * G:(h + 1) * G] - ref["o"]).max()
                errl = np.abs(lse[b, h * G:(h + 1) * G] - ref["lse"]).max()
                assert err <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k} bits {bits}: max |o - o_ref| = {err}"
                assert errl <= H.ATOL_OUT, f"unit {(b, h)} top_k {top_k} bits {bits}: max |lse - lse_ref| = {errl}"
    assert n_tie <= max(1, len(bh) * len(top_ks) // 20)


@pytest.mark.parametrize("bits", [8, 4])
def test_tiny(bits):
    w = synth.WORKLOADS["tiny"]
    _run(w, 0, [w.top_k, 0, 1, 3], bits)


@pytest.mark.parametrize("bits", [8, 4])
def test_8k(bits):
    w = synth.WORKLOADS["8k"]
    _run(w, 0, [w.top_k, 0], bits)


def test_32k_int8():
    w = synth.WORKLOADS["32k"]
    _run(w, 0, [w.top_k], 8)


@pytest.mark.parametrize("bits", [8, 4])
def test_64k_full_launch_sampled_units(bits):
    """The 64k launch (32 units, R = 128 in two 64-row stages) at the rank-48 layer."""
    w = synth.WORKLOADS["64k"]
    _run(w, 10, [w.top_k], bits, distinct=2)


def _small(d=64, G=6, nb=3, W=100, r=16, R=24, B=1, Hkv=1, seed=11):
    return synth.Workload("qedge", B, G * Hkv, Hkv, d, nb, W, (r,), R, 2, 4, False, seed)


@pytest.mark.parametrize("kw", [
    dict(R=0), dict(R=255), dict(R=5), dict(R=17), dict(W=0), dict(d=128, r=48, R=128, W=1024), dict(G=1),
    dict(G=8), dict(r=0), dict(B=2, Hkv=2, nb=5)])
@pytest.mark.parametrize("bits", [8, 4])
def test_edge_shapes(kw, bits):
    w = _small(**kw)
    _run(w, 0, [0, 1, w.n_blocks + 3], bits)


@pytest.mark.parametrize("name,layer,bits", [("tiny", 0, 8), ("tiny", 0, 4), ("8k", 0, 8), ("8k", 0, 4),
                                             ("64k", 10, 8)])
def test_compression_writes_the_oracle_codes(name, layer, bits):
    """GPU compression with quantised residuals: the rows it keeps (its own residual
    selection) are quantised exactly as the oracle quantises those same fp16 rows,
    and decoding that cache matches the oracle decoding the GPU's own factors."""
    w = synth.WORKLOADS[name]
    if name == "64k":
        w = w.with_(batch=1)
    r = w.rank(layer)
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          residual_bits=bits)
    K, V = synth.layer_kv(w, layer)
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    torch.cuda.synchronize()
    raw = cache.cpu().numpy()
    for u in range(min(2, w.units_per_layer)):
        b_, h_ = divmod(u, w.n_kv_heads)
        for blk in sorted({0, w.n_blocks // 2, w.n_blocks - 1}):
            got = LU.unpack_block(raw, desc, u, blk)
            S = got["S"]
            src_k = K[b_, h_, blk * 256 + S].astype(np.float64)
            src_v = V[b_, h_, blk * 256 + S].astype(np.float64)
            _check_codes(raw, desc, u, blk, src_k, src_v, bits)
