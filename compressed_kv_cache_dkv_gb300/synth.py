"""Seeded synthetic K/V/q generator for the DKV decode-attention workloads.

This module only draws numbers; it holds none of the method's arithmetic
(no SVD, no residual selection, no routing, no attention).  Both the fp64
oracle (through the tests) and the CUDA path read their inputs from here, so
the two sides always see the same fp16 arrays.

Value recipe (one "segment" = one 256-token block, or the recency window
treated as one more segment):

* per segment: block means mu_K, mu_V ~ N(0, 1)^d;
* per token: latent coordinates L_K, L_V ~ N(0, 1)^l (K and V have separate
  latents), mixed by per-segment W_K, W_V ~ N(0, 1/l)^(l x d);
* K = mu_K + L_K W_K + N(0, 0.05^2), V likewise;
* outliers: about 1 % of the token rows have their whole K row and V row
  multiplied by 8.  The tiny case picks single rows; the model-shaped cases
  place runs of 4..11 consecutive tokens until 1 % of the tokens are covered;
* queries q ~ N(0, 1).

The head shapes follow the Qwen2.5-1.5B attention layout quoted by the
Differential-KV README (section "Measured Paper Benchmarks": 12 query heads,
2 KV heads, head_dim 128, 28 layers), micro-block size 256 (README section
"Core Architecture & Paper Overview").  No model weights or text are used.

Every unit (layer, sequence b, KV head h) has its own seed, so any unit can
be regenerated alone on the host.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Iterable

import numpy as np

BLOCK_SIZE = 256
NOISE_STD = 0.05
OUTLIER_SCALE = 8.0
OUTLIER_FRAC = 0.01


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention workload: shapes, compression knobs, generator knobs."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_blocks: int          # compressed 256-token blocks per unit
    window: int            # dense recency-window tokens per unit
    ranks: tuple           # per-layer rank r (len == n_layers)
    n_residual: int        # exact residual rows R per block
    top_k: int             # blocks routed per query
    latent: int            # latent dimension l of the generator
    outlier_runs: bool     # runs of 4..11 tokens (True) or single rows (False)
    seed: int

    @property
    def n_layers(self) -> int:
        return len(self.ranks)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def context(self) -> int:
        return self.n_blocks * BLOCK_SIZE + self.window

    @property
    def units_per_layer(self) -> int:
        return self.batch * self.n_kv_heads

    def rank(self, layer: int) -> int:
        return self.ranks[layer]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _adaptive_ranks(n_layers: int, early: int, mid: int, late: int) -> tuple:
    # layers 0-6 early, 7-20 mid, 21-27 late for a 28-layer stack
    return tuple(early if i < 7 * n_layers // 28 else (mid if i < 21 * n_layers // 28 else late)
                 for i in range(n_layers))


WORKLOADS = {
    # 1 query, 1 q head / 1 kv head, d=64, 3 blocks + 256 window, r=8, R=16, K=2, rank-4 latent
    "tiny": Workload("tiny", 1, 1, 1, 64, 3, 256, (8,), 16, 2, 4, False, 1001),
    # Qwen2.5-1.5B-shaped single layer at 8k: 30 blocks + 512 window, r=32, R=40, K=8
    "8k": Workload("8k", 1, 12, 2, 128, 30, 512, (32,), 40, 8, 16, True, 2002),
    # same head shape at 32k, batch 4: 126 blocks + 512 window, r=32, R=40, K=16
    "32k": Workload("32k", 4, 12, 2, 128, 126, 512, (32,), 40, 16, 16, True, 3003),
    # 64k, batch 16, 28 layers, layer-adaptive rank 24/48/16, R=128, window 1024, K=16
    "64k": Workload("64k", 16, 12, 2, 128, 252, 1024, _adaptive_ranks(28, 24, 48, 16),
                    128, 16, 16, True, 4004),
    # throughput sweep: batch 64 x 16k, r=32, R=40, window 512, K in {4, 16, 62}
    "sweep16k": Workload("sweep16k", 64, 12, 2, 128, 62, 512, (32,), 40, 16, 16, True, 5005),
}
SWEEP_TOP_K = (4, 16, 62)


def _unit_rng(seed: int, layer: int, b: int, h: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, b, h, stream])))


def _outlier_rows(rng: np.random.Generator, n_tokens: int, runs: bool) -> np.ndarray:
    target = int(round(OUTLIER_FRAC * n_tokens))
    mask = np.zeros(n_tokens, dtype=bool)
    if target <= 0:
        return mask
    if not runs:
        mask[rng.choice(n_tokens, size=target, replace=False)] = True
        return mask
    covered = 0
    while covered < target:
        length = int(rng.integers(4, 12))           # U{4..11}
        start = int(rng.integers(0, max(1, n_tokens - length + 1)))
        seg = mask[start:start + length]
        covered += int((~seg).sum())
        seg[:] = True
    return mask


def unit_kv(w: Workload, layer: int, b: int, h: int) -> tuple[np.ndarray, np.ndarray]:
    """K, V of one unit as fp16 arrays of shape [T, d], T = n_blocks*256 + window."""
    d, lat = w.head_dim, w.latent
    seg_len = [BLOCK_SIZE] * w.n_blocks + ([w.window] if w.window > 0 else [])
    T = sum(seg_len)
    nseg = len(seg_len)
    rng = _unit_rng(w.seed, layer, b, h, 0)
    f32 = np.float32
    mu = rng.standard_normal((2, nseg, d), dtype=f32)
    lat_tok = rng.standard_normal((2, T, lat), dtype=f32)
    mix = rng.standard_normal((2, nseg, lat, d), dtype=f32) * f32(1.0 / np.sqrt(lat))
    noise = rng.standard_normal((2, T, d), dtype=f32)
    out = np.empty((2, T, d), dtype=f32)
    t0 = 0
    for s, n in enumerate(seg_len):
        # mean + latent mix for the segment, both K (index 0) and V (index 1)
        np.matmul(lat_tok[:, t0:t0 + n, :], mix[:, s], out=out[:, t0:t0 + n, :])
        out[:, t0:t0 + n, :] += mu[:, s, None, :]
        t0 += n
    out += f32(NOISE_STD) * noise
    rows = _outlier_rows(_unit_rng(w.seed, layer, b, h, 1), T, w.outlier_runs)
    out[:, rows, :] *= f32(OUTLIER_SCALE)
    kv = out.astype(np.float16)
    return kv[0], kv[1]


def queries(w: Workload, layer: int) -> np.ndarray:
    """Decode queries q ~ N(0, 1), fp16 [batch, n_q_heads, head_dim]."""
    rng = _unit_rng(w.seed, layer, 0xFFFF, 0xFFFF, 2)
    return rng.standard_normal((w.batch, w.n_q_heads, w.head_dim), dtype=np.float32).astype(np.float16)


def layer_kv(w: Workload, layer: int, units: Iterable[tuple[int, int]] | None = None,
             threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """K, V for a whole layer, fp16 [batch, n_kv_heads, T, d] (threaded over units)."""
    T, d = w.context, w.head_dim
    K = np.empty((w.batch, w.n_kv_heads, T, d), dtype=np.float16)
    V = np.empty_like(K)
    todo = list(units) if units is not None else [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]

    def one(bh):
        b, h = bh
        K[b, h], V[b, h] = unit_kv(w, layer, b, h)

    n = threads or min(len(todo), os.cpu_count() or 1)
    if n <= 1:
        for bh in todo:
            one(bh)
    else:
        with _cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(one, todo))
    return K, V


def layer_kv_torch(w: Workload, layer: int, device, replica: int = 0):
    """Same recipe as ``layer_kv``, drawn with torch's generator on `device`
    (a different random stream than the numpy one; used where throughput
    inputs are needed fast and no host-side reference is computed).
    Returns K, V fp16 [batch, n_kv_heads, T, d] on the device."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(np.random.SeedSequence([w.seed, layer, replica, 7]).generate_state(1)[0]))
    B, H, d, lat = w.batch, w.n_kv_heads, w.head_dim, w.latent
    NB, W = w.n_blocks, w.window
    T = w.context
    f32 = torch.float32
    out = torch.empty(2, B, H, T, d, dtype=f32, device=device)
    if NB:
        lt = torch.randn(2, B, H, NB, BLOCK_SIZE, lat, generator=g, device=device, dtype=f32)
        mix = torch.randn(2, B, H, NB, lat, d, generator=g, device=device, dtype=f32) / float(np.sqrt(lat))
        mu = torch.randn(2, B, H, NB, 1, d, generator=g, device=device, dtype=f32)
        out[:, :, :, :NB * BLOCK_SIZE] = (torch.matmul(lt, mix) + mu).reshape(2, B, H, NB * BLOCK_SIZE, d)
        del lt, mix, mu
    if W:
        lt = torch.randn(2, B, H, W, lat, generator=g, device=device, dtype=f32)
        mix = torch.randn(2, B, H, lat, d, generator=g, device=device, dtype=f32) / float(np.sqrt(lat))
        mu = torch.randn(2, B, H, 1, d, generator=g, device=device, dtype=f32)
        out[:, :, :, NB * BLOCK_SIZE:] = torch.matmul(lt, mix) + mu
        del lt, mix, mu
    out.add_(torch.randn(out.shape, generator=g, device=device, dtype=f32), alpha=NOISE_STD)
    rows = np.stack([np.stack([_outlier_rows(_unit_rng(w.seed, layer, b, h, 1 + 2 * replica), T, w.outlier_runs)
                               for h in range(H)]) for b in range(B)])
    scale = torch.from_numpy(np.where(rows, OUTLIER_SCALE, 1.0).astype(np.float32)).to(device)
    out.mul_(scale[None, :, :, :, None])
    kv = out.to(torch.float16)
    return kv[0].contiguous(), kv[1].contiguous()
