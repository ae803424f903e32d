"""Host side of dkv_prefill_attend (no GPU): argument checks that return before any
launch, the routed-slot count and the workspace size.  The arguments are plain
integers standing for device addresses; every call here is refused before the
library would touch them.
"""
import pytest

from compressed_kv_cache_dkv_gb300 import dkv

A = 1 << 20  # a 16-byte aligned stand-in address


def _call(batch, hq, hkv, d, T, top_k, ws_bytes=1 << 40, q=A, K=A, V=A, out=A, lse=None, routed=None, ws=A):
    return dkv.lib().dkv_prefill_attend(batch, hq, hkv, d, T, top_k, q, K, V, out, lse, routed, ws, ws_bytes, None)


@pytest.mark.parametrize("args,status", [
    ((0, 12, 2, 128, 4096, 16), dkv.DKV_ERR_ARG),          # no batch
    ((1, 12, 2, 128, 0, 16), dkv.DKV_ERR_ARG),             # empty prompt
    ((1, 12, 2, 128, 4096, -1), dkv.DKV_ERR_ARG),          # negative top-K
    ((1, 12, 5, 128, 4096, 16), dkv.DKV_ERR_SHAPE),        # query heads not a multiple of KV heads
    ((1, 12, 2, 96, 4096, 16), dkv.DKV_ERR_UNSUPPORTED),   # head_dim 96
    ((1, 18, 2, 128, 4096, 16), dkv.DKV_ERR_UNSUPPORTED),  # GQA group of 9
    ((1, 12, 2, 128, 1025 * 256 + 1, 16), dkv.DKV_ERR_UNSUPPORTED),  # past the longest prompt
])
def test_prefill_rejects_bad_shapes(args, status):
    assert _call(*args) == status


def test_prefill_rejects_missing_and_misaligned_buffers():
    assert _call(1, 12, 2, 128, 4096, 16, q=None) == dkv.DKV_ERR_ARG
    assert _call(1, 12, 2, 128, 4096, 16, ws=None) == dkv.DKV_ERR_ARG
    assert _call(1, 12, 2, 128, 4096, 16, K=A + 8) == dkv.DKV_ERR_ALIGN
    assert _call(1, 12, 2, 128, 4096, 16, lse=A + 4) == dkv.DKV_ERR_ALIGN
    assert _call(1, 12, 2, 128, 4096, 16, routed=A + 2) == dkv.DKV_ERR_ALIGN


def test_prefill_rejects_a_short_workspace():
    need = dkv.dkv_prefill_workspace_bytes(2, 12, 2, 64, 1000, 3)
    assert need > 0
    assert _call(2, 12, 2, 64, 1000, 3, ws_bytes=need - 1) == dkv.DKV_ERR_WORKSPACE


@pytest.mark.parametrize("T,top_k,slots", [
    (1, 0, 1), (256, 4, 1), (257, 4, 1), (1000, 0, 3), (1000, 2, 2), (1000, 3, 3), (1000, 9, 3),
    (32768, 16, 16), (32768, 0, 127), (32768, 127, 127), (32768, 200, 127),
])
def test_prefill_routed_slots(T, top_k, slots):
    """ceil(T / 256) - 1 earlier blocks at most (one slot even for a single block); top-K 0
    or at least that many means every earlier block."""
    assert dkv.dkv_prefill_routed_slots(T, top_k) == slots


@pytest.mark.parametrize("B,hkv,d,T,top_k", [(1, 2, 128, 32768, 16), (2, 4, 64, 1000, 3), (3, 1, 128, 300, 0)])
def test_prefill_workspace_bytes(B, hkv, d, T, top_k):
    """Header, then per (unit, block) the fp32 key box (2d) and mean query (d), then the
    routed lists, each section starting on a 256-byte boundary."""
    up = lambda x: -(-x // 256) * 256
    nb = -(-T // 256)
    units = B * hkv
    k_eff = dkv.dkv_prefill_routed_slots(T, top_k)
    header = 256
    off_qbar = up(header + units * nb * 2 * d * 4)
    off_routed = up(off_qbar + units * nb * d * 4)
    assert dkv.dkv_prefill_workspace_bytes(B, 6 * hkv, hkv, d, T, top_k) == off_routed + units * nb * k_eff * 4
    assert dkv.dkv_prefill_workspace_bytes(B, 6 * hkv, hkv, 96, T, top_k) == 0
