"""Thin ctypes binding of libdkv (include/dkv.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of libdkv.so.  PyTorch supplies device memory and the current CUDA
stream.  The functions keep the C names; tensors are passed where the C ABI
takes device pointers, and outputs the caller does not supply are allocated
with torch on the inputs' device.

There is no CPU fallback: when libdkv.so is missing every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdkv.so")

DKV_OK = 0
DKV_ERR_ARG = -1
DKV_ERR_SHAPE = -2
DKV_ERR_ALIGN = -3
DKV_ERR_UNSUPPORTED = -4
DKV_ERR_CUDA = -5
DKV_ERR_TIMEOUT = -6
DKV_ERR_WORKSPACE = -7
DKV_ERR_DEVICE = -8
DKV_DEVERR_TIMEOUT = 0x1
DKV_DEVERR_INDEX = 0x2
DKV_DEVERR_RANGE = 0x4
BLOCK_SIZE = 256
DKV_LAYOUT_FRAGMENT = 0
DKV_LAYOUT_TC = 1

EXPORTED = (
    "dkv_version", "dkv_status_string", "dkv_layout", "dkv_layout_bytes",
    "dkv_compress_workspace_bytes", "dkv_compress_layout", "dkv_import_factors",
    "dkv_decode_workspace_bytes", "dkv_decode_launches", "dkv_decode_attend", "dkv_decode_route", "dkv_decode_blocks",
    "dkv_decode_combine",
    "dkv_dense_workspace_bytes", "dkv_dense_decode", "dkv_get_error", "dkv_decode_attend_noalloc",
    "dkv_append_workspace_bytes", "dkv_append", "dkv_debug_set_limits", "dkv_debug_set_launch", "dkv_prefill_routed_slots",
    "dkv_prefill_workspace_bytes", "dkv_prefill_attend",
)


class DkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {dkv_status_string(status)} ({status})")
        self.status = status


class dkv_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_q_heads", "n_kv_heads", "head_dim", "block_size", "n_blocks", "window", "rank",
        "n_residual", "layout", "block_capacity", "window_capacity", "residual_bits", "rope_dims")] + [
        ("rope_base", ctypes.c_float)] + [(n, ctypes.c_int32) for n in ("rank_pad", "res_pad", "window_pad",
                                                                         "n_units")] + [
        (n, ctypes.c_uint64) for n in (
            "blk_off_mask", "blk_off_vk", "blk_off_u", "blk_off_res", "blk_off_vv", "block_bytes",
            "off_router", "off_blocks", "off_cold", "off_window", "block_stride", "unit_stride", "total_bytes",
            "off_rope")]

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


class dkv_factors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "a_k", "a_v", "U", "V_K", "V_V", "res_pos", "K_res", "V_res", "kmin", "kmax", "win_K", "win_V")]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libdkv.so (built by ``build.py`` / ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdkv.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        pdesc = ctypes.POINTER(dkv_desc)
        L.dkv_version.restype = ctypes.c_int
        L.dkv_status_string.restype = ctypes.c_char_p
        L.dkv_status_string.argtypes = [ctypes.c_int]
        L.dkv_layout.argtypes = [pdesc]
        L.dkv_layout_bytes.restype = sz
        L.dkv_layout_bytes.argtypes = [pdesc]
        L.dkv_compress_workspace_bytes.restype = sz
        L.dkv_compress_workspace_bytes.argtypes = [pdesc]
        L.dkv_compress_layout.argtypes = [pdesc, vp, vp, vp, vp, sz, vp]
        L.dkv_import_factors.argtypes = [pdesc, ctypes.POINTER(dkv_factors), vp, vp, vp]
        L.dkv_decode_workspace_bytes.restype = sz
        L.dkv_decode_workspace_bytes.argtypes = [pdesc, i32]
        L.dkv_decode_launches.restype = i32
        L.dkv_decode_launches.argtypes = [pdesc, i32]
        L.dkv_decode_attend.argtypes = [pdesc, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.dkv_decode_route.argtypes = [pdesc, vp, vp, i32, vp, vp, sz, vp]
        L.dkv_decode_blocks.argtypes = [pdesc, vp, vp, i32, vp, vp, vp, sz, vp]
        L.dkv_decode_combine.argtypes = [pdesc, i32, vp, vp, vp, sz, vp]
        L.dkv_dense_workspace_bytes.restype = sz
        L.dkv_dense_workspace_bytes.argtypes = [i32] * 5
        L.dkv_dense_decode.argtypes = [i32] * 5 + [vp] * 6 + [sz, vp]
        L.dkv_get_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.dkv_decode_attend_noalloc.argtypes = [pdesc, vp, vp, i32, vp, vp, vp, vp]
        L.dkv_append_workspace_bytes.restype = sz
        L.dkv_append_workspace_bytes.argtypes = [pdesc]
        L.dkv_append.argtypes = [pdesc, vp, vp, i32, vp, vp, sz, vp]
        L.dkv_debug_set_limits.argtypes = [i32, ctypes.c_uint32]
        L.dkv_debug_set_launch.argtypes = [i32]
        L.dkv_prefill_routed_slots.restype = i32
        L.dkv_prefill_routed_slots.argtypes = [i32, i32]
        L.dkv_prefill_workspace_bytes.restype = sz
        L.dkv_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        L.dkv_prefill_attend.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        _lib = L
    return _lib


def dkv_status_string(status: int) -> str:
    return lib().dkv_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != DKV_OK:
        raise DkvError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dkv_layout(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, n_blocks: int, window: int,
               rank: int, n_residual: int, block_size: int = BLOCK_SIZE,
               layout: int | None = None, block_capacity: int = 0, window_capacity: int = 0,
               residual_bits: int = 0, rope_dims: int = 0, rope_base: float = 0.0) -> dkv_desc:
    """Fill a descriptor.  `layout` is DKV_LAYOUT_FRAGMENT (mma.sync decode kernel, the
    default) or DKV_LAYOUT_TC (tcgen05 decode kernel; head_dim 128, rank <= 48, 1 <= R <= 128).
    `block_capacity` / `window_capacity` reserve room for dkv_append (0: the live counts).
    `residual_bits` 0 keeps residual rows fp16; 8 or 4 stores them group-quantised.
    `rope_dims` > 0 makes an un-rotated pool: keys are given and stored before RoPE and the
    decode rotates them to their absolute positions (RoPE base `rope_base`)."""
    d = dkv_desc(batch=batch, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                 block_size=block_size, n_blocks=n_blocks, window=window, rank=rank, n_residual=n_residual,
                 layout=DKV_LAYOUT_FRAGMENT if layout is None else layout,
                 block_capacity=block_capacity, window_capacity=window_capacity, residual_bits=residual_bits,
                 rope_dims=rope_dims, rope_base=rope_base)
    _check(lib().dkv_layout(ctypes.byref(d)), "dkv_layout")
    return d


def dkv_layout_supported(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, n_blocks: int, window: int,
                         rank: int, n_residual: int, layout: int) -> bool:
    """True when dkv_layout accepts these sizes under `layout`."""
    try:
        dkv_layout(batch, n_q_heads, n_kv_heads, head_dim, n_blocks, window, rank, n_residual, layout=layout)
    except DkvError:
        return False
    return True


def dkv_layout_bytes(d: dkv_desc) -> int:
    return int(lib().dkv_layout_bytes(ctypes.byref(d)))


def _ws(nbytes: int, device, workspace):
    if workspace is not None:
        return workspace
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def dkv_compress_workspace_bytes(d: dkv_desc) -> int:
    return int(lib().dkv_compress_workspace_bytes(ctypes.byref(d)))


def dkv_compress_layout(d: dkv_desc, K: torch.Tensor, V: torch.Tensor, cache: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """K, V: fp16 [B, Hkv, T, d] on the GPU -> packed cache (uint8 [total_bytes])."""
    if cache is None:
        cache = torch.empty(d.total_bytes, dtype=torch.uint8, device=K.device)
    need = int(lib().dkv_compress_workspace_bytes(ctypes.byref(d)))
    workspace = _ws(need, K.device, workspace)
    _check(lib().dkv_compress_layout(ctypes.byref(d), _ptr(K), _ptr(V), _ptr(cache), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "dkv_compress_layout")
    return cache


def dkv_append_workspace_bytes(d: dkv_desc) -> int:
    return int(lib().dkv_append_workspace_bytes(ctypes.byref(d)))


def dkv_append(d: dkv_desc, K_new: torch.Tensor, V_new: torch.Tensor, cache: torch.Tensor,
               workspace: torch.Tensor | None = None, stream=None) -> dkv_desc:
    """Append K_new, V_new (fp16 [B, Hkv, n_new, d] on the GPU) to the cache; advances d in place."""
    if K_new.shape != V_new.shape or K_new.dim() != 4:
        raise DkvError(DKV_ERR_SHAPE, "dkv_append")
    K_new, V_new = K_new.contiguous(), V_new.contiguous()
    workspace = _ws(dkv_append_workspace_bytes(d), K_new.device, workspace)
    _check(lib().dkv_append(ctypes.byref(d), _ptr(K_new), _ptr(V_new), int(K_new.shape[2]), _ptr(cache),
                            _ptr(workspace), workspace.numel(), _stream(stream)), "dkv_append")
    return d


def dkv_import_factors(d: dkv_desc, f: dict, cache: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """f: dict of device tensors named like the dkv_factors fields (fp16, res_pos int32)."""
    dev = next(v.device for v in f.values() if v is not None)
    if cache is None:
        cache = torch.empty(d.total_bytes, dtype=torch.uint8, device=dev)
    workspace = _ws(256, dev, workspace)
    fac = dkv_factors(**{k: _ptr(f.get(k)) for k, _ in dkv_factors._fields_})
    _check(lib().dkv_import_factors(ctypes.byref(d), ctypes.byref(fac), _ptr(cache), _ptr(workspace),
                                    _stream(stream)), "dkv_import_factors")
    return cache


def dkv_decode_workspace_bytes(d: dkv_desc, top_k: int) -> int:
    return int(lib().dkv_decode_workspace_bytes(ctypes.byref(d), int(top_k)))


def dkv_decode_launches(d: dkv_desc, top_k: int) -> int:
    """Kernel launches one dkv_decode_attend call makes on the current device (1: one grid)."""
    return int(lib().dkv_decode_launches(ctypes.byref(d), int(top_k)))


def dkv_decode_attend(d: dkv_desc, q: torch.Tensor, cache: torch.Tensor, top_k: int,
                      out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = True,
                      routed: torch.Tensor | bool | None = True, workspace: torch.Tensor | None = None,
                      stream=None):
    """q fp16 [B, Hq, d] -> (out fp32 [B, Hq, d], lse fp32 [B, Hq] or None, routed int32 [B, Hkv, K_eff] or None)."""
    dev = q.device
    k_eff = d.n_blocks if (top_k == 0 or top_k >= d.n_blocks) else top_k
    if out is None:
        out = torch.empty(d.batch, d.n_q_heads, d.head_dim, dtype=torch.float32, device=dev)
    if lse is True:
        lse = torch.empty(d.batch, d.n_q_heads, dtype=torch.float32, device=dev)
    elif lse is False:
        lse = None
    if routed is True:
        routed = torch.empty(d.batch, d.n_kv_heads, max(k_eff, 0), dtype=torch.int32, device=dev) if k_eff > 0 else None
    elif routed is False:
        routed = None
    if workspace is None:
        workspace = _ws(dkv_decode_workspace_bytes(d, top_k), dev, None)
    _check(lib().dkv_decode_attend(ctypes.byref(d), _ptr(q), _ptr(cache), int(top_k), _ptr(out), _ptr(lse),
                                   _ptr(routed), _ptr(workspace), workspace.numel(), _stream(stream)),
           "dkv_decode_attend")
    return out, lse, routed


def dkv_decode_route(d: dkv_desc, q, cache, top_k: int, workspace, routed=None, stream=None) -> None:
    _check(lib().dkv_decode_route(ctypes.byref(d), _ptr(q), _ptr(cache), int(top_k), _ptr(routed), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "dkv_decode_route")


def dkv_decode_blocks(d: dkv_desc, q, cache, top_k: int, workspace, out=None, lse=None, stream=None) -> None:
    _check(lib().dkv_decode_blocks(ctypes.byref(d), _ptr(q), _ptr(cache), int(top_k), _ptr(out), _ptr(lse),
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "dkv_decode_blocks")


def dkv_decode_combine(d: dkv_desc, top_k: int, out, workspace, lse=None, stream=None) -> None:
    _check(lib().dkv_decode_combine(ctypes.byref(d), int(top_k), _ptr(out), _ptr(lse), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "dkv_decode_combine")


def dkv_dense_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, T) -> int:
    return int(lib().dkv_dense_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, T))


def dkv_dense_decode(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, out: torch.Tensor | None = None,
                     lse: torch.Tensor | bool | None = True, workspace: torch.Tensor | None = None, stream=None):
    """Dense decode attention over uncompressed K, V fp16 [B, Hkv, T, d]; q fp16 [B, Hq, d]."""
    B, Hkv, T, dh = K.shape
    Hq = q.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty(B, Hq, dh, dtype=torch.float32, device=dev)
    if lse is True:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    elif lse is False:
        lse = None
    if workspace is None:
        workspace = _ws(dkv_dense_workspace_bytes(B, Hq, Hkv, dh, T), dev, None)
    _check(lib().dkv_dense_decode(B, Hq, Hkv, dh, T, _ptr(q), _ptr(K), _ptr(V), _ptr(out), _ptr(lse),
                                  _ptr(workspace), workspace.numel(), _stream(stream)), "dkv_dense_decode")
    return out, lse


def dkv_prefill_routed_slots(T: int, top_k: int) -> int:
    """Slots per query block of dkv_prefill_attend's routed-index output (0 on bad arguments)."""
    return int(lib().dkv_prefill_routed_slots(int(T), int(top_k)))


def dkv_prefill_workspace_bytes(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, T: int,
                                top_k: int) -> int:
    """Workspace bytes dkv_prefill_attend needs for these sizes (0 on bad arguments)."""
    return int(lib().dkv_prefill_workspace_bytes(int(batch), int(n_q_heads), int(n_kv_heads), int(head_dim), int(T),
                                                 int(top_k)))


def dkv_prefill_attend(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, top_k: int, out: torch.Tensor | None = None,
                       lse: torch.Tensor | bool = True, routed: torch.Tensor | bool = True,
                       workspace: torch.Tensor | None = None, stream=None):
    """Block-sparse prefill: q fp16 [B, Hq, T, d], K, V fp16 [B, Hkv, T, d] on the GPU ->
    (out fp32 [B, Hq, T, d], lse fp32 [B, Hq, T] or None, routed int32 [B, Hkv, nb, slots] or None)."""
    B, Hq, T, d = q.shape
    Hkv = K.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty(B, Hq, T, d, dtype=torch.float32, device=dev)
    if lse is True:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=dev)
    nb = -(-T // BLOCK_SIZE)
    if routed is True:
        routed = torch.empty(B, Hkv, nb, dkv_prefill_routed_slots(T, top_k), dtype=torch.int32, device=dev)
    need = dkv_prefill_workspace_bytes(B, Hq, Hkv, d, T, top_k)
    workspace = _ws(need, dev, workspace)
    lse_t = lse if isinstance(lse, torch.Tensor) else None
    routed_t = routed if isinstance(routed, torch.Tensor) else None
    _check(lib().dkv_prefill_attend(B, Hq, Hkv, d, T, int(top_k), _ptr(q), _ptr(K), _ptr(V), _ptr(out),
                                    _ptr(lse_t) if lse_t is not None else None,
                                    _ptr(routed_t) if routed_t is not None else None, _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "dkv_prefill_attend")
    return out, lse_t, routed_t


def dkv_debug_set_limits(stop_after_chunks: int = -1, wait_polls: int = 0) -> None:
    """Failure-path diagnostics: producers of the fragment layout's attention CTAs stop
    after `stop_after_chunks` chunks, bounded waits give up after `wait_polls` polls;
    (-1, 0) restores the defaults."""
    _check(lib().dkv_debug_set_limits(int(stop_after_chunks), int(wait_polls)), "dkv_debug_set_limits")


def dkv_debug_set_launch(programmatic: bool = True) -> None:
    """Timing aid: False launches the decode grids in plain stream order (no programmatic
    overlap with the grid before them); True restores the default."""
    _check(lib().dkv_debug_set_launch(1 if programmatic else 0), "dkv_debug_set_launch")


def dkv_get_error(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    """(status, device error word); clears the word."""
    w = ctypes.c_uint32(0)
    st = lib().dkv_get_error(_ptr(workspace), _stream(stream), ctypes.byref(w))
    return st, int(w.value)
