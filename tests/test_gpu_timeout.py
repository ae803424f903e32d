"""The bounded-wait failure path, provoked on the host side.

dkv_debug_set_limits makes every attention CTA's producer stop issuing after a
few chunks and shortens the bounded waits.  The consumer warps then wait for
chunks that are never issued (nothing is in flight: the producer drains what
it did issue), their waits give up, the kernel raises DKV_DEVERR_TIMEOUT and
the host reads it with dkv_get_error.  The context stays usable: the next call
on the same workspace decodes like a fresh one.  No GPU fault is involved.
"""
import numpy as np
import pytest
import torch

from compressed_kv_cache_dkv_gb300 import dkv, synth
from oracle import dkv_oracle as O
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stop_after", [0, 1])
def test_timeout_is_reported_and_the_workspace_stays_usable(stop_after):
    w = synth.WORKLOADS["8k"]
    units = H.oracle_units(w, 0, [(0, 0), (0, 1)])
    desc = dkv.dkv_layout(1, 12, 2, 128, w.n_blocks, w.window, 32, 40)
    cache = dkv.dkv_import_factors(desc, H.to_device(H.factor_arrays(units, 128, 32, 40, w.window)))
    q = synth.queries(w, 0)
    qd = torch.from_numpy(q).cuda()
    ws = torch.zeros(dkv.dkv_decode_workspace_bytes(desc, w.top_k), dtype=torch.uint8, device="cuda")
    try:
        dkv.dkv_debug_set_limits(stop_after, 64)  # 64 polls of at most ~20 us: a wait gives up within ~1.3 ms
        dkv.dkv_decode_attend(desc, qd, cache, w.top_k, workspace=ws)
        st, word = dkv.dkv_get_error(ws)
    finally:
        dkv.dkv_debug_set_limits(-1, 0)
    assert st == dkv.DKV_ERR_TIMEOUT and word & dkv.DKV_DEVERR_TIMEOUT, (st, word)
    # the same workspace, default limits: a correct decode and a clean error word
    out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, w.top_k, workspace=ws)
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK and word == 0
    out = out.cpu().numpy()
    for h in range(2):
        ref = O.decode_unit(q[0, 6 * h:6 * h + 6].astype(np.float64), H.round_unit(units[h]), w.top_k)
        H.check_routing(routed.cpu().numpy()[0, h], ref["idx"], ref["bounds"])
        assert np.abs(out[0, 6 * h:6 * h + 6] - ref["o"]).max() <= H.ATOL_OUT


@pytest.mark.parametrize("stop_after", [3, 6])
def test_timeout_in_the_middle_of_long_ranges(stop_after):
    """128 units (the 16k sweep's shape): about two ranges per unit, dozens of chunks
    each, so the producers stop in the middle of their lists.  Afterwards the same
    workspace gives bit for bit what a fresh one gives."""
    w = synth.WORKLOADS["sweep16k"]
    desc = dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window, 32, 40)
    K, V = synth.layer_kv_torch(w, 0, torch.device("cuda"))
    cache = dkv.dkv_compress_layout(desc, K, V)
    del K, V
    qd = torch.from_numpy(synth.queries(w, 0)).cuda()
    ws = torch.zeros(dkv.dkv_decode_workspace_bytes(desc, 16), dtype=torch.uint8, device="cuda")
    try:
        dkv.dkv_debug_set_limits(stop_after, 64)
        dkv.dkv_decode_attend(desc, qd, cache, 16, workspace=ws)
        st, word = dkv.dkv_get_error(ws)
    finally:
        dkv.dkv_debug_set_limits(-1, 0)
    assert st == dkv.DKV_ERR_TIMEOUT and word & dkv.DKV_DEVERR_TIMEOUT, (st, word)
    out, lse, routed = dkv.dkv_decode_attend(desc, qd, cache, 16, workspace=ws)
    st, word = dkv.dkv_get_error(ws)
    assert st == dkv.DKV_OK and word == 0
    fresh = torch.zeros_like(ws)
    out2, lse2, routed2 = dkv.dkv_decode_attend(desc, qd, cache, 16, workspace=fresh)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2) and torch.equal(routed, routed2)
