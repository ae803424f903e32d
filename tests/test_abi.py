"""The C-ABI library: loads, exports every symbol include/dkv.h declares, and
validates descriptors and arguments on the host (no GPU needed here)."""
import ctypes
import os
import re

import pytest

from compressed_kv_cache_dkv_gb300 import dkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dkv_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = dkv.lib()
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dkv.EXPORTED)
    assert lib.dkv_version() == 5


def test_status_strings():
    for st in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert dkv.dkv_status_string(st)
    assert dkv.dkv_status_string(-99) == "unknown status"


def test_layout_validation():
    ok = dict(batch=1, n_q_heads=12, n_kv_heads=2, head_dim=128, n_blocks=30, window=512, rank=32, n_residual=40)
    dkv.dkv_layout(**ok)
    bad = [
        (dict(batch=0), dkv.DKV_ERR_ARG), (dict(rank=-1), dkv.DKV_ERR_ARG), (dict(n_blocks=-1), dkv.DKV_ERR_ARG),
        (dict(n_q_heads=13), dkv.DKV_ERR_SHAPE), (dict(n_blocks=0, window=0), dkv.DKV_ERR_SHAPE),
        (dict(head_dim=96), dkv.DKV_ERR_UNSUPPORTED), (dict(rank=129), dkv.DKV_ERR_UNSUPPORTED),
        (dict(n_residual=256), dkv.DKV_ERR_UNSUPPORTED), (dict(n_q_heads=18), dkv.DKV_ERR_UNSUPPORTED),
        (dict(block_size=128), dkv.DKV_ERR_UNSUPPORTED), (dict(layout=2), dkv.DKV_ERR_ARG),
        (dict(layout=-1), dkv.DKV_ERR_ARG),
        # the tensor-core layout: head_dim 128, 1 <= rank <= 48, 1 <= R <= 128
        (dict(layout=1, head_dim=64), dkv.DKV_ERR_UNSUPPORTED), (dict(layout=1, rank=49), dkv.DKV_ERR_UNSUPPORTED),
        (dict(layout=1, rank=0), dkv.DKV_ERR_UNSUPPORTED), (dict(layout=1, n_residual=0), dkv.DKV_ERR_UNSUPPORTED),
        (dict(layout=1, n_residual=129), dkv.DKV_ERR_UNSUPPORTED),
        # group-quantised residual rows: 8 or 4 bits, fragment layout only
        (dict(residual_bits=2), dkv.DKV_ERR_ARG), (dict(residual_bits=16), dkv.DKV_ERR_ARG),
        (dict(residual_bits=-8), dkv.DKV_ERR_ARG), (dict(layout=1, residual_bits=8), dkv.DKV_ERR_UNSUPPORTED),
        # the un-rotated pool: rope_dims a multiple of 32 up to head_dim, base > 1, fragment layout,
        # fp16 residual rows, rank up to 64
        (dict(rope_dims=-32, rope_base=1e4), dkv.DKV_ERR_ARG), (dict(rope_dims=160, rope_base=1e4), dkv.DKV_ERR_ARG),
        (dict(rope_dims=64, rope_base=1.0), dkv.DKV_ERR_ARG), (dict(rope_dims=64, rope_base=float("inf")), dkv.DKV_ERR_ARG),
        (dict(rope_dims=64, rope_base=float("nan")), dkv.DKV_ERR_ARG),
        (dict(rope_dims=48, rope_base=1e4), dkv.DKV_ERR_UNSUPPORTED),
        (dict(rope_dims=64, rope_base=1e4, layout=1), dkv.DKV_ERR_UNSUPPORTED),
        (dict(rope_dims=64, rope_base=1e4, residual_bits=8), dkv.DKV_ERR_UNSUPPORTED),
        (dict(rope_dims=64, rope_base=1e4, rank=65), dkv.DKV_ERR_UNSUPPORTED),
    ]
    for change, status in bad:
        kw = dict(ok, **change)
        with pytest.raises(dkv.DkvError) as e:
            dkv.dkv_layout(**kw)
        assert e.value.status == status, change


@pytest.mark.parametrize("d,nb,W,r,R,layout", [
    (128, 30, 512, 32, 40, 0), (128, 252, 1024, 48, 128, 0), (64, 3, 256, 8, 16, 0), (128, 5, 17, 24, 5, 0),
    (64, 0, 100, 0, 0, 0), (128, 30, 512, 32, 40, 1), (128, 252, 1024, 48, 128, 1), (128, 5, 17, 24, 5, 1),
    (128, 2, 300, 1, 1, 1)])
def test_layout_bytes(d, nb, W, r, R, layout):
    """Both layouts hold the same sections in the same number of bytes, 16-byte aligned."""
    desc = dkv.dkv_layout(2, 6, 2, d, nb, W, r, R, layout=layout)
    assert desc.layout == layout
    r8, R8, W16 = -(-r // 8) * 8, -(-R // 8) * 8, -(-W // 16) * 16
    hot = 4 * d + 32 + 2 * r8 * d + 512 * r8 + 4 * R8 * d + 2 * r8 * d
    assert desc.block_bytes == hot
    assert desc.block_stride % 128 == 0 and desc.block_stride >= hot
    for off in (desc.blk_off_mask, desc.blk_off_vk, desc.blk_off_u, desc.blk_off_res, desc.blk_off_vv,
                desc.off_blocks, desc.off_cold, desc.off_window, desc.unit_stride):
        assert off % 16 == 0
    assert desc.unit_stride >= nb * (4 * d + desc.block_stride) + W16 * 4 * d
    assert desc.total_bytes == desc.unit_stride * 2 * 2
    assert dkv.dkv_layout_bytes(desc) == desc.total_bytes
    # sections do not overlap: [start, end) of each inside the block record
    sec = sorted([(desc.blk_off_mask, 32), (desc.blk_off_vk, 2 * r8 * d), (desc.blk_off_u, 512 * r8),
                  (desc.blk_off_res, 4 * R8 * d), (desc.blk_off_vv, 2 * r8 * d)])
    for (a, na), (b, _) in zip(sec, sec[1:]):
        assert a + na <= b
    assert sec[-1][0] + sec[-1][1] <= desc.block_bytes


def test_calls_validate_before_touching_the_device():
    """Bad arguments return an error code without any CUDA work."""
    desc = dkv.dkv_layout(1, 6, 1, 64, 3, 100, 16, 24)
    L = dkv.lib()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert L.dkv_decode_attend(ctypes.byref(desc), None, fake, 2, fake, None, None, fake, 1 << 20, None) == dkv.DKV_ERR_ARG
    assert L.dkv_decode_attend(ctypes.byref(desc), fake, fake, -3, fake, None, None, fake, 1 << 20, None) == dkv.DKV_ERR_ARG
    assert L.dkv_decode_attend(ctypes.byref(desc), odd, fake, 2, fake, None, None, fake, 1 << 20, None) == dkv.DKV_ERR_ALIGN
    assert L.dkv_decode_attend(ctypes.byref(desc), fake, fake, 2, fake, None, None, fake, 16, None) == dkv.DKV_ERR_WORKSPACE
    edited = dkv.dkv_desc.from_buffer_copy(desc)
    edited.rank = 24     # descriptor changed after dkv_layout()
    assert L.dkv_decode_attend(ctypes.byref(edited), fake, fake, 2, fake, None, None, fake, 1 << 20, None) == dkv.DKV_ERR_SHAPE
    assert L.dkv_compress_layout(ctypes.byref(desc), None, fake, fake, fake, 1 << 20, None) == dkv.DKV_ERR_ARG
    assert L.dkv_dense_decode(1, 6, 4, 64, 10, fake, fake, fake, fake, None, fake, 1 << 20, None) == dkv.DKV_ERR_SHAPE
    assert L.dkv_dense_decode(1, 6, 1, 80, 10, fake, fake, fake, fake, None, fake, 1 << 20, None) == dkv.DKV_ERR_UNSUPPORTED
    assert dkv.dkv_decode_workspace_bytes(desc, -1) == 0
    assert dkv.dkv_decode_workspace_bytes(desc, 2) > 0


def test_capacity_fields_fix_the_offsets():
    """With capacities set, the byte layout stays the same whatever the live counts."""
    base = dict(batch=2, n_q_heads=12, n_kv_heads=2, head_dim=128, rank=32, n_residual=40,
                block_capacity=40, window_capacity=700)
    ref = dkv.dkv_layout(n_blocks=40, window=700, **base)
    for nb, w in ((0, 1), (3, 0), (17, 699), (40, 700), (0, 0)):
        desc = dkv.dkv_layout(n_blocks=nb, window=w, **base)
        for f in ("off_router", "off_blocks", "off_cold", "off_window", "block_stride", "unit_stride", "total_bytes"):
            assert getattr(desc, f) == getattr(ref, f), f
        assert desc.window_pad == -(-w // 16) * 16
    # no capacity: the live counts are the capacity
    plain = dkv.dkv_layout(2, 12, 2, 128, 40, 700, 32, 40)
    assert plain.total_bytes == ref.total_bytes
    bad = [(dict(n_blocks=41, window=1), dkv.DKV_ERR_SHAPE), (dict(n_blocks=1, window=701), dkv.DKV_ERR_SHAPE),
           (dict(n_blocks=1, window=1, block_capacity=-1), dkv.DKV_ERR_ARG),
           (dict(n_blocks=1, window=1, block_capacity=2049), dkv.DKV_ERR_UNSUPPORTED),
           (dict(n_blocks=1, window=1, window_capacity=65537), dkv.DKV_ERR_UNSUPPORTED),
           (dict(n_blocks=0, window=0, window_capacity=0, block_capacity=0), dkv.DKV_ERR_SHAPE)]
    for change, status in bad:
        with pytest.raises(dkv.DkvError) as e:
            dkv.dkv_layout(**dict(base, **change))
        assert e.value.status == status, change


def test_append_validates_before_touching_the_device():
    """dkv_append plans the whole append on the host: too little room, a bad
    count, misaligned pointers, a small workspace or the tensor-core layout are
    reported with nothing launched (the fake pointers are never dereferenced)."""
    L = dkv.lib()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    big = 1 << 30

    def call(desc, n_new, k=fake, ws=big):
        before = bytes(desc)
        st = L.dkv_append(ctypes.byref(desc), k, fake, n_new, fake, fake, ws, None)
        assert bytes(desc) == before  # the descriptor only advances on success
        return st

    d = dkv.dkv_layout(1, 6, 1, 64, 1, 300, 8, 4, block_capacity=2, window_capacity=300)
    assert call(d, -1) == dkv.DKV_ERR_ARG
    assert call(d, 1, k=odd) == dkv.DKV_ERR_ALIGN
    assert call(d, 1, ws=16) == dkv.DKV_ERR_WORKSPACE
    # 300 + 256 + 1 tokens would need a third block
    assert call(d, 2 * 256 + 1) == dkv.DKV_ERR_UNSUPPORTED
    st0 = bytes(d)
    assert L.dkv_append(ctypes.byref(d), fake, fake, 0, fake, fake, big, None) == dkv.DKV_OK  # nothing to do
    assert bytes(d) == st0
    # a window capacity below one block cannot slide
    small = dkv.dkv_layout(1, 6, 1, 64, 0, 200, 8, 4, block_capacity=4, window_capacity=200)
    assert call(small, 1) == dkv.DKV_ERR_UNSUPPORTED
    tc = dkv.dkv_layout(1, 6, 1, 128, 1, 300, 8, 4, layout=dkv.DKV_LAYOUT_TC, block_capacity=4, window_capacity=512)
    assert call(tc, 1) == dkv.DKV_ERR_UNSUPPORTED
    assert dkv.dkv_append_workspace_bytes(d) >= 256 + 2 * 256 * 64 * 2


def test_decode_launch_counts():
    """dkv_decode_launches (host only): router, attention and combine; no router grid
    when nothing is routed or, for the fragment layout, when every block is."""
    frag = dkv.dkv_layout(2, 12, 2, 128, 30, 512, 32, 40)
    assert [dkv.dkv_decode_launches(frag, k) for k in (8, 1, 29)] == [3, 3, 3]
    assert [dkv.dkv_decode_launches(frag, k) for k in (30, 31, 0)] == [2, 2, 2]  # every block routed
    assert dkv.dkv_decode_launches(frag, -1) == 0                                # invalid top_k
    empty = dkv.dkv_layout(2, 12, 2, 128, 0, 512, 32, 40)
    assert [dkv.dkv_decode_launches(empty, k) for k in (0, 4)] == [2, 2]
    tc = dkv.dkv_layout(2, 12, 2, 128, 30, 512, 32, 40, layout=dkv.DKV_LAYOUT_TC)
    assert [dkv.dkv_decode_launches(tc, k) for k in (8, 0, 30)] == [3, 3, 3]  # the tc path always routes
    tc_empty = dkv.dkv_layout(2, 12, 2, 128, 0, 512, 32, 40, layout=dkv.DKV_LAYOUT_TC)
    assert [dkv.dkv_decode_launches(tc_empty, k) for k in (0, 4)] == [2, 2]


@pytest.mark.parametrize("d,R,bits", [(128, 40, 8), (128, 128, 4), (64, 16, 8), (64, 5, 4), (128, 255, 8), (128, 0, 4)])
def test_quantised_residual_layout_bytes(d, R, bits):
    """A group-quantised residual store holds R rounded up to 16 rows in 16-token groups
    of K and V codes plus one fp16 scale and bias per 64 channels of every row; the
    other sections are those of the fp16 layout."""
    desc = dkv.dkv_layout(2, 6, 2, d, 7, 100, 24, R, residual_bits=bits)
    plain = dkv.dkv_layout(2, 6, 2, d, 7, 100, 24, R)
    R16 = -(-R // 16) * 16
    assert desc.res_pad == R16 and desc.residual_bits == bits
    group = 2 * 16 * d * bits // 8 + 4 * 16 * 2 * (d // 64)
    assert desc.blk_off_vv - desc.blk_off_res == R16 // 16 * group
    assert desc.block_bytes - desc.blk_off_vv == plain.block_bytes - plain.blk_off_vv
    assert desc.blk_off_res == plain.blk_off_res
    for off in (desc.blk_off_vv, desc.block_stride, desc.off_window, desc.unit_stride):
        assert off % 16 == 0
    assert desc.block_bytes < plain.block_bytes or R == 0


@pytest.mark.parametrize("d,dims,cap_b,cap_w", [(128, 128, 30, 512), (128, 32, 252, 1024), (64, 64, 3, 300),
                                                (64, 32, 0, 100)])
def test_unrotated_pool_layout_bytes(d, dims, cap_b, cap_w):
    """An un-rotated pool stores fp32 router boxes (8d bytes a block) and ends with the
    RoPE tables: a (cos, sin) fp32 pair per RoPE channel pair for every 256-token page
    the capacities reach and for each of the 256 in-page offsets; the block records and
    the window are those of the rotated pool."""
    kw = dict(block_capacity=cap_b, window_capacity=cap_w)
    desc = dkv.dkv_layout(2, 6, 2, d, min(cap_b, 2), min(cap_w, 50), 24, 40, rope_dims=dims, rope_base=1e6, **kw)
    plain = dkv.dkv_layout(2, 6, 2, d, min(cap_b, 2), min(cap_w, 50), 24, 40, **kw)
    assert desc.rope_dims == dims and desc.rope_base == 1e6
    assert desc.block_bytes == plain.block_bytes and desc.blk_off_res == plain.blk_off_res
    assert desc.off_blocks == -(-cap_b * 8 * d // 128) * 128
    assert desc.off_window - desc.off_blocks == plain.off_window - plain.off_blocks
    pages = max(1, -(-(cap_b * 256 + cap_w) // 256))
    assert desc.off_rope == desc.unit_stride * desc.n_units and desc.off_rope % 16 == 0
    assert desc.total_bytes == desc.off_rope + (pages + 256) * (dims // 2) * 8
    assert plain.off_rope == 0 and plain.total_bytes == plain.unit_stride * plain.n_units
