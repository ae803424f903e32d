"""Shared test helpers: oracle factors of synthetic units, fp16 packing for the
C ABI's plain factor import, and the parity comparison rules."""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

from compressed_kv_cache_dkv_gb300 import synth
from oracle import dkv_oracle as O

# Output tolerance of the decode parity (fp16 operands, fp32 accumulation)
# and the routing tie band, both on the oracle's c-scaled values.
ATOL_OUT = 2e-3
TIE_BAND = 1e-4

_POOL = None


def pool():
    """Process pool for oracle compression (spawn: safe next to a CUDA context)."""
    global _POOL
    if _POOL is None:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(k, "1")
        n = max(1, min(16, (os.cpu_count() or 2)))
        _POOL = cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))
    return _POOL


def _compress_job(args):
    w, layer, b, h, rank, rope = args
    K, V = synth.unit_kv(w, layer, b, h)
    return O.compress_unit(K, V, w.n_blocks, rank, w.n_residual, rope=rope)


def oracle_units(w: synth.Workload, layer: int, bh_list, parallel: bool = True, rope: O.Rope | None = None):
    """Oracle-compressed units of `w` (an un-rotated pool when `rope` is given: the
    synthetic keys are then read as keys before RoPE)."""
    jobs = [(w, layer, b, h, w.rank(layer), rope) for b, h in bh_list]
    if parallel and len(jobs) > 1:
        return list(pool().map(_compress_job, jobs))
    return [_compress_job(j) for j in jobs]


def round_unit(unit: O.Unit) -> O.Unit:
    """The same compressed unit with every factor rounded to fp16 (the stored operands);
    an un-rotated pool's boxes are stored as fp32."""
    h = lambda x: np.asarray(x, dtype=np.float16).astype(np.float64)
    bx = (lambda x: np.asarray(x, dtype=np.float32).astype(np.float64)) if unit.rope is not None else h
    blocks = [O.Block(a_k=h(b.a_k), a_v=h(b.a_v), U=h(b.U), V_K=h(b.V_K), V_V=h(b.V_V), S=b.S.copy(),
                      K_res=h(b.K_res), V_res=h(b.V_res), kmin=bx(b.kmin), kmax=bx(b.kmax)) for b in unit.blocks]
    return O.Unit(blocks=blocks, win_K=h(unit.win_K), win_V=h(unit.win_V), rope=unit.rope)


def factor_arrays(units: list, d: int, r: int, R: int, W: int) -> dict:
    """Plain fp16 factor arrays [U_][NB]... in the order of `units` (dkv_factors)."""
    n = len(units)
    NB = len(units[0].blocks)
    f16 = np.float16
    fb = np.float32 if units[0].rope is not None else f16  # an un-rotated pool's boxes are fp32
    out = {
        "a_k": np.zeros((n, NB, d), f16), "a_v": np.zeros((n, NB, d), f16),
        "U": np.zeros((n, NB, 255, r), f16), "V_K": np.zeros((n, NB, r, d), f16), "V_V": np.zeros((n, NB, r, d), f16),
        "res_pos": np.zeros((n, NB, R), np.int32), "K_res": np.zeros((n, NB, R, d), f16),
        "V_res": np.zeros((n, NB, R, d), f16), "kmin": np.zeros((n, NB, d), fb), "kmax": np.zeros((n, NB, d), fb),
        "win_K": np.zeros((n, W, d), f16), "win_V": np.zeros((n, W, d), f16),
    }
    for i, un in enumerate(units):
        for b, blk in enumerate(un.blocks):
            out["a_k"][i, b] = blk.a_k
            out["a_v"][i, b] = blk.a_v
            out["U"][i, b] = blk.U
            out["V_K"][i, b] = blk.V_K
            out["V_V"][i, b] = blk.V_V
            out["res_pos"][i, b] = blk.S
            out["K_res"][i, b] = blk.K_res
            out["V_res"][i, b] = blk.V_res
            out["kmin"][i, b] = blk.kmin
            out["kmax"][i, b] = blk.kmax
        out["win_K"][i] = un.win_K
        out["win_V"][i] = un.win_V
    return out


def to_device(arrs: dict, device="cuda"):
    import torch
    return {k: (torch.from_numpy(np.ascontiguousarray(v)).to(device) if v.size else None) for k, v in arrs.items()}


def check_routing(gpu_idx: np.ndarray, ref_idx: np.ndarray, bounds: np.ndarray) -> None:
    """Routed sets must be equal, except that a block may differ when its oracle
    bound lies within TIE_BAND of the oracle's K-th bound."""
    g, r = set(int(x) for x in gpu_idx), set(int(x) for x in ref_idx)
    assert len(g) == len(gpu_idx), "duplicate routed index"
    assert list(gpu_idx) == sorted(gpu_idx), "routed indices not ascending"
    if g == r:
        return
    kth = np.sort(bounds)[::-1][len(ref_idx) - 1]
    for b in g ^ r:
        assert abs(bounds[b] - kth) <= TIE_BAND, f"block {b} routed differently (bound {bounds[b]}, K-th {kth})"


def _compress_blocks_job(args):
    Kc, Vc, rank, R = args
    n = Kc.shape[0] // O.BLOCK_SIZE
    return [O.compress_block(Kc[i * 256:(i + 1) * 256], Vc[i * 256:(i + 1) * 256], rank, R) for i in range(n)]


def oracle_unit_blockwise(K: np.ndarray, V: np.ndarray, n_blocks: int, rank: int, R: int, per_job: int = 8) -> O.Unit:
    """compress_unit with the blocks spread over the process pool."""
    jobs = [(K[b * 256:min(n_blocks, b + per_job) * 256], V[b * 256:min(n_blocks, b + per_job) * 256], rank, R)
            for b in range(0, n_blocks, per_job)]
    blocks = [blk for part in pool().map(_compress_blocks_job, jobs) for blk in part]
    return O.Unit(blocks=blocks, win_K=np.asarray(K[n_blocks * 256:], np.float64),
                  win_V=np.asarray(V[n_blocks * 256:], np.float64))
