"""dkv_debug_set_launch(0): the decode grids go in plain stream order instead of as
programmatic dependents of the grid before them (the benchmark times consecutive
attention grids that way).  Only the launch order changes, so the results must
equal those of the default launches bit for bit, through the fused call and the
stage calls, in both cache layouts.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,layout", [("tiny", dkv.DKV_LAYOUT_FRAGMENT), ("8k", dkv.DKV_LAYOUT_FRAGMENT),
                                         ("8k", dkv.DKV_LAYOUT_TC)])
def test_plain_stream_order_gives_the_same_results(name, layout):
    w = synth.WORKLOADS[name]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, w.rank(0),
                          w.n_residual, layout=layout)
    K, V = synth.layer_kv(w, 0)
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    q = torch.from_numpy(np.random.default_rng(9).standard_normal((w.batch, w.n_q_heads, w.head_dim))
                         .astype(np.float16)).cuda()
    ws = torch.zeros(dkv.dkv_decode_workspace_bytes(desc, w.top_k), dtype=torch.uint8, device="cuda")

    def stages():
        # without a caller's copy of the indices the router fills the attention grid's list
        # in rank order, so the stage calls sum in another order than the fused call above
        out = torch.full((w.batch, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
        lse = torch.full((w.batch, w.n_q_heads), float("nan"), device="cuda")
        dkv.dkv_decode_route(desc, q, cache, w.top_k, ws)
        dkv.dkv_decode_blocks(desc, q, cache, w.top_k, ws)
        dkv.dkv_decode_combine(desc, w.top_k, out, ws, lse=lse)
        torch.cuda.synchronize()
        return out, lse

    ref_out, ref_lse, ref_routed = dkv.dkv_decode_attend(desc, q, cache, w.top_k)
    ref_s_out, ref_s_lse = stages()
    try:
        dkv.dkv_debug_set_launch(False)
        out, lse, routed = dkv.dkv_decode_attend(desc, q, cache, w.top_k)
        s_out, s_lse = stages()
    finally:
        dkv.dkv_debug_set_launch(True)
    assert dkv.dkv_get_error(ws)[0] == dkv.DKV_OK
    # the same kernels on the same plan in a fixed summation order
    assert torch.equal(routed, ref_routed)
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)
    assert torch.equal(s_out, ref_s_out)
    assert torch.equal(s_lse, ref_s_lse)
