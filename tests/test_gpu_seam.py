"""The compress -> decode seam at the decode tolerance.

The cache the benchmark runs is compressed on the GPU.  Here the oracle reads
that very cache: every block's factors are unpacked from the packed bytes
(tests/layout_unpack.py, its own index arithmetic), the oracle decodes them by
the plain definition in fp64, and the GPU's decode of the same cache must
match within 2e-3 (routed indices exact outside the 1e-4 tie band).  Both
sides then use identical fp16 operands, so no allowance for the two
compressors' different (equally valid) SVD bases is needed.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H
from tests import layout_unpack as LU

pytestmark = pytest.mark.gpu


def _unit_from_cache(raw, desc, u):
    blocks = []
    f = lambda x: np.asarray(x, dtype=np.float64)
    for b in range(desc.n_blocks):
        g = LU.unpack_block(raw, desc, u, b)
        blocks.append(O.Block(a_k=f(g["a_k"]), a_v=f(g["a_v"]), U=f(g["U"]), V_K=f(g["V_K"]), V_V=f(g["V_V"]),
                              S=g["S"], K_res=f(g["K_res"]), V_res=f(g["V_res"]), kmin=f(g["kmin"]),
                              kmax=f(g["kmax"])))
    wk, wv = LU.unpack_window(raw, desc, u)
    return O.Unit(blocks=blocks, win_K=f(wk), win_V=f(wv))


@pytest.mark.parametrize("name,layer,units,bits", [
    ("tiny", 0, None, 0), ("8k", 0, None, 0), ("8k", 0, None, 8), ("32k", 0, [0, 5], 0),
    ("64k", 0, [0, 31], 0), ("64k", 10, [7], 0), ("64k", 27, [20], 0), ("sweep16k", 0, [0, 77, 127], 0)])
def test_gpu_compressed_cache_decodes_like_the_oracle_reading_it(name, layer, units, bits):
    w = synth.WORKLOADS[name]
    r = w.rank(layer)
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, r, w.n_residual,
                          residual_bits=bits)
    K, V = synth.layer_kv_torch(w, layer, torch.device("cuda"))
    cache = dkv.dkv_compress_layout(desc, K, V)
    del K, V
    q = synth.queries(w, layer)
    top_ks = list(synth.SWEEP_TOP_K) if name == "sweep16k" else [w.top_k]
    raw = cache.cpu().numpy()
    G = w.group
    todo = list(range(w.units_per_layer)) if units is None else units
    oracle_units = {u: _unit_from_cache(raw, desc, u) for u in todo}
    for top_k in top_ks:
        out, lse, routed = dkv.dkv_decode_attend(desc, torch.from_numpy(q).cuda(), cache, top_k)
        out, lse, routed = out.cpu().numpy(), lse.cpu().numpy(), routed.cpu().numpy()
        for u in todo:
            b, h = divmod(u, w.n_kv_heads)
            ref = O.decode_unit(q[b, h * G:(h + 1) * G].astype(np.float64), oracle_units[u], top_k)
            H.check_routing(routed[b, h], ref["idx"], ref["bounds"])
            if set(routed[b, h]) != set(ref["idx"]):
                continue  # a tie inside the band: the two sides attend different (equally valid) sets
            err = np.abs(out[b, h * G:(h + 1) * G] - ref["o"]).max()
            errl = np.abs(lse[b, h * G:(h + 1) * G] - ref["lse"]).max()
            assert err <= H.ATOL_OUT, f"{name} unit {u} top_k {top_k}: max |o - o_ref| = {err}"
            assert errl <= H.ATOL_OUT, f"{name} unit {u} top_k {top_k}: max |lse - lse_ref| = {errl}"
