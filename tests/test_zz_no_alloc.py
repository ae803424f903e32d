"""dkv_decode_attend_noalloc: the decode call for callers that cannot allocate
device memory (fixed-pool runtimes, plugins without an allocator, loops that
must not synchronise the device through cudaMalloc).  Its scratch comes from
a fixed area inside the library, so its results must equal those of
dkv_decode_attend with a caller-provided workspace, call after call.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth

pytestmark = pytest.mark.gpu


def _noalloc(desc, q, cache, top_k, out, lse, routed, stream):
    return dkv.lib().dkv_decode_attend_noalloc(ctypes.byref(desc), q.data_ptr(), cache.data_ptr(), int(top_k),
                                               out.data_ptr(), lse.data_ptr(), routed.data_ptr(),
                                               ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("name,layout", [("tiny", dkv.DKV_LAYOUT_FRAGMENT), ("8k", dkv.DKV_LAYOUT_FRAGMENT),
                                         ("8k", dkv.DKV_LAYOUT_TC)])
def test_noalloc_matches_decode_attend_on_consecutive_calls(name, layout):
    w = synth.WORKLOADS[name]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, w.rank(0),
                          w.n_residual, layout=layout)
    K, V = synth.layer_kv(w, 0)
    cache = dkv.dkv_compress_layout(desc, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(5)
    for call in range(2):  # two calls in a row share the library's scratch area
        q = torch.from_numpy(rng.standard_normal((w.batch, w.n_q_heads, w.head_dim)).astype(np.float16)).cuda()
        ref_out, ref_lse, ref_routed = dkv.dkv_decode_attend(desc, q, cache, w.top_k)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        routed = torch.full_like(ref_routed, -1)
        st = _noalloc(desc, q, cache, w.top_k, out, lse, routed, stream)
        assert st == dkv.DKV_OK, dkv.dkv_status_string(st)
        torch.cuda.synchronize()
        # both calls run the same kernels on the same plan, in a fixed summation order:
        # any difference means the shared scratch carried something over
        assert torch.equal(routed, ref_routed), f"call {call}: routed blocks differ"
        assert torch.equal(out, ref_out), f"call {call}: outputs differ"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs"


def test_noalloc_rejects_a_scratch_need_beyond_its_area():
    w = synth.WORKLOADS["sweep16k"]  # at batch 2048: 4096 units of partial records, ~17 MB of scratch
    desc = dkv.dkv_layout(2048, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, 32, 40)
    assert dkv.dkv_decode_workspace_bytes(desc, 0) > (8 << 20)
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    st = dkv.lib().dkv_decode_attend_noalloc(ctypes.byref(desc), t.data_ptr(), t.data_ptr(), 0, t.data_ptr(), None,
                                             None, None)
    assert st == dkv.DKV_ERR_WORKSPACE
