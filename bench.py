#!/usr/bin/env python3
"""Decode-attention throughput over the DKV compressed cache on GB300.

One step = one decode step of every layer of the workload: per layer one
dkv_decode_attend (route -> block/window attention -> LSE combine) over that
layer's packed cache, each layer with its own queries.  Default workload: the
64k configuration (batch 16, 28 layers of 12 q / 2 KV heads, head_dim 128,
252 blocks + 1024-token window per unit, layer-adaptive rank 24/48/16, 128
residual rows, top-K 16).

Prints ONE JSON line (rank 0).  `value` = queries/s of the device-timed
steps (inputs resident in HBM, K steps replayed from a CUDA graph);
`e2e` = the same metric through the C ABI with pinned host buffers (q copied
in, out copied back, every step); `roofline` = the block/window attention
kernel's algorithmic bytes per launch over its CUDA-event duration inside the
timed region; `cpu_baseline` = the fp64 oracle timed on host cores on a
bounded sample.  `--impl reference` times the oracle alone as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no data-path collective); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attention queries/s and HBM GB/s (% of roofline) over DKV cache"
FALLBACK_HBM_GBS = 6800.0


_T0 = time.perf_counter()


def log(*a):
    print(f"[{time.perf_counter() - _T0:7.1f} s]", *a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- multi-rank arithmetic

def max_over_ranks(values, device):
    """Elementwise maximum of per-rank timings over the process group (every rank gets it)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(world: int, queries_per_step: int, steps: int, ms: float) -> float:
    """Queries per second of the whole job: every rank runs its own replica of the
    workload (weak scaling), so all ranks' queries count over the slowest rank's time."""
    return world * queries_per_step * steps / (ms / 1e3)


# ----------------------------------------------------------------------------- byte accounting

def residual_token_bytes(d: int, bits: int) -> int:
    """Bytes of one residual token (its key row and value row): fp16 rows, or
    group-quantised rows (codes plus an fp16 scale and bias per 64 channels)."""
    return 4 * d if bits == 0 else 2 * (d * bits // 8 + 4 * (d // 64))


def attend_bytes(w, layer: int, top_k: int, bits: int = 0) -> int:
    """Algorithmic bytes the block/window attention kernel must read per launch:
    per unit K routed blocks (anchors 4d + V_K,V_V 4rd + U 2*255*r + residual
    rows R * (4d, or their quantised size) + mask 32) plus the window 4Wd; per
    launch the queries."""
    d, r, R, W, NB = w.head_dim, w.rank(layer), w.n_residual, w.window, w.n_blocks
    k = NB if (top_k == 0 or top_k >= NB) else top_k
    per_block = 4 * d + 4 * r * d + 2 * 255 * r + R * residual_token_bytes(d, bits) + 32
    per_unit = k * per_block + W * 4 * d
    return w.units_per_layer * per_unit + w.batch * w.n_q_heads * d * 2


def call_bytes(w, layer: int, top_k: int, bits: int = 0, rope: bool = False) -> int:
    """Algorithmic bytes of one dkv_decode_attend: the attention kernel's bytes,
    the router rows NB*4d per unit (NB*8d: an un-rotated pool's fp32 boxes), and
    the fp32 output."""
    return (attend_bytes(w, layer, top_k, bits) + w.units_per_layer * w.n_blocks * (8 if rope else 4) * w.head_dim
            + w.batch * w.n_q_heads * w.head_dim * 4)


def cache_replicas(bytes_per_pass: int, l2_bytes: int) -> int:
    """Cache replicas a step's calls rotate over, so that the bytes one step reads
    (bytes_per_pass per replica) span at least 4x the L2: 1 when one pass already does."""
    return max(1, -(-4 * l2_bytes // max(1, bytes_per_pass)))


# ----------------------------------------------------------------------------- clocks (NVML, read only)

REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    """Samples the SM clock and the clock-event reasons of this process's GPU every few ms."""

    def __init__(self, torch_device_index: int):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._h = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            bus = self._bus_id(torch_device_index)
            h = ctypes.c_void_p()
            if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nv, self._h = nv, h
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._reasons = fn
        except OSError:
            self._h = None

    @staticmethod
    def _bus_id(idx: int):
        try:
            import torch
            rt = ctypes.CDLL("libcudart.so.13")
            buf = ctypes.create_string_buffer(64)
            dev = torch.cuda.current_device() if idx is None else idx
            if rt.cudaDeviceGetPCIBusId(buf, 64, dev) != 0:
                return None
            return buf.value
        except OSError:
            return None

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0 and \
                    self._reasons(self._h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.003)

    def __enter__(self):
        if self._h is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._h is not None:
            self._t.join()

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        reasons = 0
        for _, r in busy:
            reasons |= r
        names = [n for b, n in REASONS.items() if reasons & b and b != 0x1]
        return {"sm_mhz": statistics.median(c for c, _ in busy), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(busy)}


# ----------------------------------------------------------------------------- CUDA events usable inside graphs

class ExtEvents:
    """cudaEvent_t objects recorded with cudaEventRecordExternal, so that a
    record placed in a captured stream becomes an event node of the graph."""

    def __init__(self):
        self.rt = ctypes.CDLL("libcudart.so.13")
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]
        self.events = []

    def new(self):
        ev = ctypes.c_void_p()
        if self.rt.cudaEventCreate(ctypes.byref(ev)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        self.events.append(ev)
        return ev

    def record(self, ev, stream_handle: int):
        if self.rt.cudaEventRecordWithFlags(ev, ctypes.c_void_p(stream_handle), 1) != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed")

    def elapsed_ms(self, a, b) -> float:
        ms = ctypes.c_float()
        if self.rt.cudaEventElapsedTime(ctypes.byref(ms), a, b) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return float(ms.value)

    def close(self):
        for ev in self.events:
            self.rt.cudaEventDestroy(ev)
        self.events = []


# ----------------------------------------------------------------------------- CPU oracle arm

def _oracle_decode_worker(args):
    """Child process (spawned, BLAS pinned to one thread): compress unit number
    `index` of the layer (sequence index // n_kv_heads, KV head index % n_kv_heads,
    wrapping over the batch) with the oracle (untimed), then time its decode for
    ~`seconds`."""
    cfg_name, layer, index, seconds, top_k = args
    import numpy as np

    from compressed_kv_cache_dkv_gb300 import synth
    from oracle import dkv_oracle as O
    w = synth.WORKLOADS[cfg_name]
    b, h = divmod(index % (w.batch * w.n_kv_heads), w.n_kv_heads)
    K, V = synth.unit_kv(w, layer, b, h)
    t0 = time.perf_counter()
    unit = O.compress_unit(K, V, w.n_blocks, w.rank(layer), w.n_residual)
    t_comp = time.perf_counter() - t0
    q = synth.queries(w, layer)[b, h * w.group:(h + 1) * w.group].astype(np.float64)
    n = 0
    t0 = time.perf_counter()
    while True:
        O.decode_unit(q, unit, top_k)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"decodes": n, "seconds": el, "queries": n * w.group, "compress_s": t_comp}


def host_cores(cap: int = 32) -> int:
    """Host cores this process may run on (its CPU affinity, not the machine's
    count), at most `cap`: one oracle process per core."""
    try:
        n = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        n = os.cpu_count() or 1
    return max(1, min(cap, n))


def cpu_oracle(cfg_name: str, layer: int, seconds: float, top_k: int, n_proc: int = 1) -> dict:
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    ctx = mp.get_context("spawn")
    with ctx.Pool(n_proc) as pool:
        res = pool.map(_oracle_decode_worker, [(cfg_name, layer, i, seconds, top_k) for i in range(n_proc)])
    q = sum(r["queries"] for r in res)
    t = max(r["seconds"] for r in res)
    return {"queries": q, "seconds": t, "qps": q / t, "cores": n_proc, "compress_s": max(r["compress_s"] for r in res)}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["dkv", "reference"], default="dkv")
    ap.add_argument("--config", default="64k")
    ap.add_argument("--top-k", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None, help="restrict to N layers (experiments only)")
    ap.add_argument("--layer-offset", type=int, default=0, help="first layer when --layers is given")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layout", choices=["fragment", "tc"], default="fragment",
                    help="cache layout and with it the decode kernel of the timed path: fragment = mma.sync "
                         "kernel, tc = tcgen05 kernel")
    ap.add_argument("--no-alt-layout", action="store_true",
                    help="skip timing the other cache layout's decode kernel over the same step")
    ap.add_argument("--no-dense-reference", action="store_true",
                    help="skip timing the dense fp16 decode kernel over the 16k sweep's uncompressed K, V")
    ap.add_argument("--reps", type=int, default=10, help="graph replays timed (the median is reported; >= 10)")
    ap.add_argument("--configs", default="32k,8k,sweep16k",
                    help="further workloads reported under `configs` (one layer each, several cache replicas)")
    ap.add_argument("--config-steps", type=int, default=20, help="steps per graph for the further workloads")
    ap.add_argument("--no-configs", action="store_true", help="skip the further workloads")
    ap.add_argument("--no-prefill", action="store_true", help="skip the block-sparse prefill measurement")
    ap.add_argument("--no-append", action="store_true", help="skip the streaming-append measurement")
    ap.add_argument("--no-unrotated", action="store_true", help="skip the un-rotated pool (RoPE at read) step")
    ap.add_argument("--rope-dims", type=int, default=0,
                    help="time the headline workload as an un-rotated pool with RoPE over this many channels")
    ap.add_argument("--prefill-tokens", type=int, default=32768, help="prompt length of the prefill measurement")
    ap.add_argument("--quant-bits", default="8,4",
                    help="also time the headline workload with residual rows group-quantised to these widths")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from compressed_kv_cache_dkv_gb300 import synth
    w = synth.WORKLOADS[args.config]
    top_k = w.top_k if args.top_k is None else args.top_k
    n_layers = w.n_layers if args.layers is None else min(args.layers, w.n_layers - args.layer_offset)
    layer_ids = [args.layer_offset + i for i in range(n_layers)] if args.layers is not None else list(range(n_layers))
    wl_name = (f"{w.name}: batch {w.batch}, {n_layers} layer(s) of {w.n_q_heads}q/{w.n_kv_heads}kv heads x d{w.head_dim}, "
               f"{w.n_blocks} blocks of 256 + {w.window}-token window, r {sorted(set(w.ranks[i] for i in layer_ids))}, "
               f"R {w.n_residual}, top-K {top_k}")
    queries_per_step = w.batch * w.n_q_heads * n_layers

    if args.impl == "reference":
        if rank != 0:
            return
        K = args.steps
        per = max(0.5, args.cpu_seconds / max(1, K + args.warmup))
        r = cpu_oracle(w.name, 0, per * (K + args.warmup), top_k, n_proc=host_cores())
        qps = r["qps"]
        line = {"impl": "reference", "metric": METRIC, "value": qps, "unit": "queries/s", "n_gpus": args.gpus,
                "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * queries_per_step / qps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": wl_name,
                                                "sample": f"{r['cores']} units of layer 0, one per host core"},
                "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": r["cores"], "kind": "oracle",
                                 "sample": f"fp64 oracle decode of {r['cores']} units of layer 0 ({w.group} queries "
                                           f"each), one spawned process per host core, each repeated for "
                                           f"{r['seconds']:.1f} s; compression excluded"},
                "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import numpy as np  # noqa: F401
    import torch

    from compressed_kv_cache_dkv_gb300 import dkv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    dkv.lib()
    reps = max(10, args.reps)

    layout_ids = {"fragment": dkv.DKV_LAYOUT_FRAGMENT, "tc": dkv.DKV_LAYOUT_TC}
    kernel_names = {"fragment": "attend_kernel (mma.sync, block + window attention)",
                    "tc": "attend_tc_kernel (tcgen05 + TMEM, block + window attention) + combine_kernel"}
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    ext = ExtEvents()
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak = float(json.load(open(peaks_path))["hbm_gbs"])
        peak_src = "measured"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"

    def timed(g, n_rep):
        """Replay graph `g` n_rep times, each bracketed by events on its stream (after a
        barrier and a device synchronisation on both sides); returns the per-replay
        times (ms) and the clocks sampled during them."""
        times = []
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk, torch.cuda.stream(stream):
            for _ in range(n_rep):
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                g.replay()
                t1.record(stream)
                stream.synchronize()
                times.append(t0.elapsed_time(t1))
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return times, clk

    class Setup:
        """Packed caches, queries and outputs of one workload at one top-K; small
        workloads rotate a step's calls over cache replicas so that the bytes one step
        reads span at least 4x the L2 and every call reads its cache from HBM."""

        def __init__(self, w, layer_ids, top_k, layout, ws_bytes=None, min_call_bytes=None, bits=0, rope=(0, 0.0)):
            self.w, self.top_k, self.layout, self.bits, self.rope = w, top_k, layout, bits, rope
            base = sum(call_bytes(w, l, top_k, bits, rope[0] > 0) for l in layer_ids)
            self.n_rep = cache_replicas(min_call_bytes or base, l2_bytes)
            self.layer_ids = layer_ids * self.n_rep
            self.n_layers = len(self.layer_ids)
            self.descs = [dkv.dkv_layout(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window,
                                         w.rank(l), w.n_residual, layout=layout_ids[layout], residual_bits=bits,
                                         rope_dims=rope[0], rope_base=rope[1])
                          for l in self.layer_ids]
            need = max(dkv.dkv_decode_workspace_bytes(d, k) for d in self.descs for k in {top_k, 0})
            self.ws = torch.zeros(max(need, ws_bytes or 0), dtype=torch.uint8, device=dev)
            self.caches = []
            for i, layer in enumerate(self.layer_ids):
                K, V = synth.layer_kv_torch(w, layer, dev, replica=rank)
                self.caches.append(dkv.dkv_compress_layout(self.descs[i], K, V, workspace=self.ws))
                del K, V
            torch.cuda.synchronize()
            st_, word_ = dkv.dkv_get_error(self.ws)
            if st_ != dkv.DKV_OK:
                raise RuntimeError(f"compression raised device error word {word_:#x}")
            self.qs = [torch.from_numpy(synth.queries(w, l)).to(dev) for l in self.layer_ids]
            self.outs = [torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.float32, device=dev)
                         for _ in self.layer_ids]
            self.lses = [torch.empty(w.batch, w.n_q_heads, dtype=torch.float32, device=dev) for _ in self.layer_ids]
            self.cache_gb = sum(c.numel() for c in self.caches) / 1e9

        def measure(self, top_k, steps, warmup, n_rep, stage_timing=True, latency=True):
            """Warm up, capture `steps` steps (one call per cache of the set) into a CUDA graph,
            time n_rep replays of it (median taken); with stage_timing also a second graph of
            the same steps run as the stage calls with events around every attention launch
            (its events split the programmatic launches, so that graph runs a little slower);
            with latency one call alone, captured in its own graph and replayed n_rep times."""
            n = self.n_layers

            def call(i, events=None):
                if events is None:
                    dkv.dkv_decode_attend(self.descs[i], self.qs[i], self.caches[i], top_k, out=self.outs[i],
                                          lse=self.lses[i], routed=False, workspace=self.ws, stream=sh)
                    return
                dkv.dkv_decode_route(self.descs[i], self.qs[i], self.caches[i], top_k, self.ws, stream=sh)
                ext.record(events[0], sh)
                dkv.dkv_decode_blocks(self.descs[i], self.qs[i], self.caches[i], top_k, self.ws, stream=sh)
                ext.record(events[1], sh)
                dkv.dkv_decode_combine(self.descs[i], top_k, self.outs[i], self.ws, lse=self.lses[i], stream=sh)

            with torch.cuda.stream(stream):
                for _ in range(warmup):
                    for i in range(n):
                        call(i)
            stream.synchronize()
            res = {}
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(steps):
                    for i in range(n):
                        call(i)
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
            times, clk = timed(g, n_rep)
            res["ms_replays"] = times
            res["ms"] = statistics.median(times)
            res["clocks"] = clk.summary()
            if stage_timing:
                # (1) every attention launch between a pair of events of its own; the bracket itself
                #     costs about 4 us of launch and event latency (measured in (3))
                ev = [[(ext.new(), ext.new()) for _ in range(n)] for _ in range(steps)]
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2, stream=stream):
                    for k in range(steps):
                        for i in range(n):
                            call(i, ev[k][i])
                with torch.cuda.stream(stream):
                    g2.replay()
                stream.synchronize()
                t2, clk2 = timed(g2, 1)
                res["ms_ev"] = t2[0]
                res["attend_ms_bracketed"] = [ext.elapsed_ms(ev[k][i][0], ev[k][i][1])
                                              for k in range(steps) for i in range(n)]
                del g2
                # (2) the same attention launches back to back: per step every call's router first
                #     (each call keeps its routed list in a workspace of its own), then all the
                #     attention grids in plain stream order (none overlaps the one before it) between
                #     one pair of events, then the combines; time per launch = region / calls
                wss = [torch.zeros_like(self.ws) for _ in range(n)]
                evr = [(ext.new(), ext.new()) for _ in range(steps)]
                g3 = torch.cuda.CUDAGraph()
                dkv.dkv_debug_set_launch(False)
                try:
                    with torch.cuda.graph(g3, stream=stream):
                        for k in range(steps):
                            for i in range(n):
                                dkv.dkv_decode_route(self.descs[i], self.qs[i], self.caches[i], top_k, wss[i],
                                                     stream=sh)
                            ext.record(evr[k][0], sh)
                            for i in range(n):
                                dkv.dkv_decode_blocks(self.descs[i], self.qs[i], self.caches[i], top_k, wss[i],
                                                      stream=sh)
                            ext.record(evr[k][1], sh)
                            for i in range(n):
                                dkv.dkv_decode_combine(self.descs[i], top_k, self.outs[i], wss[i],
                                                       lse=self.lses[i], stream=sh)
                finally:
                    dkv.dkv_debug_set_launch(True)
                with torch.cuda.stream(stream):
                    g3.replay()
                stream.synchronize()
                _, clk3 = timed(g3, 1)
                res["attend_ms"] = [ext.elapsed_ms(a, b) / n for a, b in evr]
                res["clocks_ev"] = clk3.summary()
                for x in wss:
                    st_, word_ = dkv.dkv_get_error(x, stream=sh)
                    if st_ != dkv.DKV_OK:
                        raise RuntimeError(f"decode raised device error word {word_:#x}")
                del g3, wss
                # (3) the bracket of (1) around an empty kernel
                evb = [(ext.new(), ext.new()) for _ in range(n)]
                g4 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g4, stream=stream):
                    for i in range(n):
                        ext.record(evb[i][0], sh)
                        torch.cuda._sleep(0)
                        ext.record(evb[i][1], sh)
                with torch.cuda.stream(stream):
                    g4.replay()
                    g4.replay()
                stream.synchronize()
                res["bracket_ms"] = statistics.median(ext.elapsed_ms(a, b) for a, b in evb)
                del g4
            if latency:
                g1 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g1, stream=stream):
                    call(0)
                with torch.cuda.stream(stream):
                    g1.replay()
                stream.synchronize()
                t1, _ = timed(g1, max(20, n_rep))
                res["latency_us"] = 1e3 * statistics.median(t1)
                del g1
            del g
            st_, word_ = dkv.dkv_get_error(self.ws, stream=sh)
            if st_ != dkv.DKV_OK:
                raise RuntimeError(f"decode raised device error word {word_:#x}")
            return res

        def free(self):
            del self.caches, self.ws, self.qs, self.outs, self.lses
            torch.cuda.empty_cache()

    # ---------------- headline workload (untimed setup: compress every layer's K, V)
    w = synth.WORKLOADS[args.config]
    top_k = w.top_k if args.top_k is None else args.top_k
    n_layers0 = w.n_layers if args.layers is None else min(args.layers, w.n_layers - args.layer_offset)
    base_ids = [args.layer_offset + i for i in range(n_layers0)] if args.layers is not None else list(range(n_layers0))
    wl_name = (f"{w.name}: batch {w.batch}, {n_layers0} layer(s) of {w.n_q_heads}q/{w.n_kv_heads}kv heads x d{w.head_dim}, "
               f"{w.n_blocks} blocks of 256 + {w.window}-token window, r {sorted(set(w.ranks[i] for i in base_ids))}, "
               f"R {w.n_residual}, top-K {top_k}")
    t_setup = time.perf_counter()
    if args.rope_dims:
        wl_name += f"; un-rotated pool (RoPE over {args.rope_dims} channels at read, base 1e6)"
    S = Setup(w, base_ids, top_k, args.layout, rope=(args.rope_dims, 1e6 if args.rope_dims else 0.0))
    t_setup = time.perf_counter() - t_setup
    if S.n_rep > 1:
        wl_name += f"; each step {S.n_rep} calls over {S.n_rep} cache replicas"
    n_layers = S.n_layers
    queries_per_step = w.batch * w.n_q_heads * n_layers
    log(f"[bench] rank {rank}: setup {t_setup:.1f} s, packed caches {S.cache_gb:.2f} GB over {n_layers} layers")
    K_steps = args.steps
    launches_per_call = [dkv.dkv_decode_launches(d_, top_k) for d_ in S.descs]
    R = S.measure(top_k, K_steps, args.warmup, reps)
    log(f"[bench] headline step timed: {R['ms'] / K_steps:.3f} ms/step")
    ms, ms_ev, attend_ms = R["ms"], R["ms_ev"], R["attend_ms"]

    # ---------------- e2e through the C ABI with pinned host buffers
    # Every step copies all its layers' queries in (one pinned copy) and reads all its layers'
    # outputs back (one copy): the same bytes as one copy per layer, without putting
    # 2 x n_layers small copies between the decode kernels.  The headline runs the copies on
    # their own streams with two device buffers each way, as a server overlaps them: step k+1's
    # queries go in and step k's outputs come back while the decode kernels run.  The serial
    # form (copy in, decode, copy out, all on one stream) is reported beside it.
    e2e_steps = args.e2e_steps or max(10, min(K_steps, 50))
    q_host = torch.stack([q.cpu() for q in S.qs]).pin_memory()
    q_devs = [torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) for _ in range(2)]
    o_shape = (n_layers,) + tuple(S.outs[0].shape)
    o_devs = [torch.empty(o_shape, dtype=S.outs[0].dtype, device=dev) for _ in range(2)]
    o_hosts = [torch.empty(o_shape, dtype=S.outs[0].dtype, pin_memory=True) for _ in range(2)]
    e_ws = torch.zeros(S.ws.numel(), dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_dec = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def decode_layers(bi):
        for layer in range(n_layers):
            dkv.dkv_decode_attend(S.descs[layer], q_devs[bi][layer], S.caches[layer], top_k, out=o_devs[bi][layer],
                                  lse=False, routed=False, workspace=e_ws, stream=sh)

    def e2e_step_serial():
        with torch.cuda.stream(stream):
            q_devs[0].copy_(q_host, non_blocking=True)
            decode_layers(0)
            o_hosts[0].copy_(o_devs[0], non_blocking=True)

    def e2e_step(k):
        bi = k & 1
        if used[bi]:
            s_in.wait_event(ev_dec[bi])    # step k - 2's decode has read q_devs[bi]
            stream.wait_event(ev_out[bi])  # step k - 2's outputs have left o_devs[bi]
        with torch.cuda.stream(s_in):
            q_devs[bi].copy_(q_host, non_blocking=True)
        ev_in[bi].record(s_in)
        stream.wait_event(ev_in[bi])
        decode_layers(bi)
        ev_dec[bi].record(stream)
        s_out.wait_event(ev_dec[bi])
        with torch.cuda.stream(s_out):
            o_hosts[bi].copy_(o_devs[bi], non_blocking=True)
        ev_out[bi].record(s_out)
        used[bi] = True

    def timed_e2e(step_fn, end_stream):
        for k in range(3):
            step_fn(k)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for k in range(e2e_steps):
            step_fn(k)
        e1.record(end_stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    e2e_ms_serial = timed_e2e(lambda k: e2e_step_serial(), stream)
    e2e_ms = timed_e2e(e2e_step, s_out)
    q_host_bytes = q_host.numel() * q_host.element_size()
    o_host_bytes = o_hosts[0].numel() * o_hosts[0].element_size()
    step_bytes = sum(call_bytes(w, l, top_k, 0, args.rope_dims > 0) for l in S.layer_ids)
    att_bytes_step = sum(attend_bytes(w, l, top_k) for l in S.layer_ids)
    S.free()
    del q_devs, o_devs, e_ws
    log(f"[bench] e2e timed: {e2e_ms / e2e_steps:.3f} ms/step (copies overlapped), "
        f"{e2e_ms_serial / e2e_steps:.3f} ms/step (serial)")

    # ---------------- the other cache layout's decode kernel over the same step (same inputs)
    alt = None
    if not args.no_alt_layout:
        alt_layout = "tc" if args.layout == "fragment" else "fragment"
        if all(dkv.dkv_layout_supported(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_blocks, w.window,
                                        w.rank(l), w.n_residual, layout_ids[alt_layout]) for l in base_ids):
            A = Setup(w, base_ids, top_k, alt_layout)
            AR = A.measure(top_k, K_steps, args.warmup, reps, latency=False)
            A.free()
            log(f"[bench] {alt_layout} layout timed: {AR['ms'] / K_steps:.3f} ms/step")
            alt = {"layout": alt_layout, "kernel": kernel_names[alt_layout], "ms": AR["ms"], "ms_ev": AR["ms_ev"],
                   "attend_ms_mean": statistics.fmean(AR["attend_ms"]),
                   "attend_ms_bracketed": statistics.fmean(AR["attend_ms_bracketed"]), "clocks": AR["clocks"]}

    # ---------------- the other workloads: 32k, 8k and the 16k top-K sweep beside the dense fp16 kernel
    configs = {}
    if not args.no_configs and args.layers is None:
        def config_entry(wc, k, R_, S_, steps_c):
            cb = sum(call_bytes(wc, l, k, S_.bits, S_.rope[0] > 0) for l in S_.layer_ids)
            ab = sum(attend_bytes(wc, l, k, S_.bits) for l in S_.layer_ids)
            ms_call = R_["ms"] / (steps_c * S_.n_layers)
            att_us = 1e3 * statistics.fmean(R_["attend_ms"])
            return {"workload": (f"{wc.name}: batch {wc.batch}, {wc.n_q_heads}q/{wc.n_kv_heads}kv x d{wc.head_dim}, "
                                 f"{wc.n_blocks} blocks + {wc.window}-token window, r {wc.rank(0)}, R {wc.n_residual}, "
                                 f"top-K {k}; {S_.n_rep} cache replicas"),
                    "queries_per_s": wc.batch * wc.n_q_heads / (ms_call / 1e3),
                    "us_per_call": 1e3 * ms_call, "bytes_per_call": cb / S_.n_layers,
                    "gbs": cb / (R_["ms"] / steps_c / 1e3) / 1e9,
                    "frac_call": cb / (R_["ms"] / steps_c / 1e3) / 1e9 / peak,
                    "steps_per_replay": steps_c,
                    "attend_us_mean": att_us, "attend_bytes_per_launch": ab / S_.n_layers,
                    "attend_us_bracketed": 1e3 * statistics.fmean(R_["attend_ms_bracketed"]),
                    "attend_frac": (ab / S_.n_layers) / (att_us / 1e6) / 1e9 / peak,
                    "latency_us": R_["latency_us"],
                    "replays": len(R_["ms_replays"]), "clocks": R_["clocks"]}
        # the headline workload with group-quantised residual rows (README "Core Innovations" item 2)
        for bits in ([int(x) for x in args.quant_bits.split(",")] if args.quant_bits else []):
            Sq = Setup(w, base_ids, top_k, "fragment", bits=bits)
            Rq = Sq.measure(top_k, K_steps, args.warmup, reps)
            ent = config_entry(w, top_k, Rq, Sq, K_steps)
            ent["workload"] = f"{wl_name}; residual rows group-quantised to int{bits} (64-channel groups)"
            ent["queries_per_s"] = queries_per_step * K_steps / (Rq["ms"] / 1e3)
            ent["ms_per_step"] = Rq["ms"] / K_steps
            configs[f"{w.name}_int{bits}_residuals"] = ent
            log(f"[bench] int{bits} residuals timed: {ent['ms_per_step']:.3f} ms/step")
            Sq.free()
        # the headline workload as an un-rotated pool (README knob DKV_ROTATED_POOL=0: keys stored
        # before RoPE, every attended key rotated to its absolute position at read)
        if not args.no_unrotated:
            Sr = Setup(w, base_ids, top_k, "fragment", rope=(w.head_dim, 1e6))
            Rr = Sr.measure(top_k, K_steps, args.warmup, reps)
            ent = config_entry(w, top_k, Rr, Sr, K_steps)
            ent["workload"] = (f"{wl_name}; un-rotated pool: keys stored before RoPE and rotated at read "
                               f"(all {w.head_dim} channels, RoPE base 1e6), fp32 router boxes")
            ent["queries_per_s"] = queries_per_step * K_steps / (Rr["ms"] / 1e3)
            ent["ms_per_step"] = Rr["ms"] / K_steps
            ent["step_time_vs_rotated_pool"] = Rr["ms"] / R["ms"]
            configs[f"{w.name}_unrotated_pool"] = ent
            log(f"[bench] un-rotated pool timed: {ent['ms_per_step']:.3f} ms/step")
            Sr.free()
        for name in args.configs.split(","):
            wc = synth.WORKLOADS[name]
            ks = [wc.top_k] if name != "sweep16k" else [4, 16, wc.n_blocks]
            min_b = min(call_bytes(wc, 0, k) for k in ks)
            Sc = Setup(wc, [0], ks[0], "fragment", min_call_bytes=min_b)
            steps_c = max(1, min(args.config_steps, 1200 // Sc.n_layers))  # about 1200 calls per graph at most
            for k in ks:
                Rc = Sc.measure(k, steps_c, args.warmup, reps)
                configs[f"{name}_top{k}" if len(ks) > 1 else name] = config_entry(wc, k, Rc, Sc, steps_c)
                log(f"[bench] {name} top-K {k} timed")
            Sc.free()
            if name == "sweep16k" and not args.no_dense_reference:
                # dense fp16 decode over the uncompressed K, V of the same seed (config 5's reference)
                Kd, Vd = synth.layer_kv_torch(wc, 0, dev, replica=rank)
                od = torch.empty(wc.batch, wc.n_q_heads, wc.head_dim, dtype=torch.float32, device=dev)
                ld = torch.empty(wc.batch, wc.n_q_heads, dtype=torch.float32, device=dev)
                wsd = torch.zeros(max(256, dkv.dkv_dense_workspace_bytes(wc.batch, wc.n_q_heads, wc.n_kv_heads,
                                                                          wc.head_dim, wc.context)),
                                  dtype=torch.uint8, device=dev)
                qd = torch.from_numpy(synth.queries(wc, 0)).to(dev)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        dkv.dkv_dense_decode(qd, Kd, Vd, out=od, lse=ld, workspace=wsd, stream=sh)
                gd = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gd, stream=stream):  # each call reads K and V once (far larger than L2)
                    dkv.dkv_dense_decode(qd, Kd, Vd, out=od, lse=ld, workspace=wsd, stream=sh)
                with torch.cuda.stream(stream):
                    gd.replay()
                stream.synchronize()
                td, clkd = timed(gd, reps)
                dense_ms = statistics.median(td)
                log(f"[bench] dense fp16 decode timed: {1e3 * dense_ms:.1f} us")
                dense_bytes = 2 * Kd.numel() * 2 + wc.batch * wc.n_q_heads * wc.head_dim * (2 + 4)
                st, word = dkv.dkv_get_error(wsd, stream=sh)
                if st != dkv.DKV_OK:
                    raise RuntimeError(f"dense decode raised device error word {word:#x}")
                configs["sweep16k_dense_fp16"] = {
                    "workload": f"dense fp16 decode over the uncompressed K, V of {wc.name} (same seed), "
                                f"{wc.context} tokens per unit",
                    "kernel": "dense_kernel + combine (dkv_dense_decode)",
                    "queries_per_s": wc.batch * wc.n_q_heads / (dense_ms / 1e3), "us_per_call": 1e3 * dense_ms,
                    "bytes_per_call": dense_bytes, "gbs": dense_bytes / (dense_ms / 1e3) / 1e9,
                    "frac_call": dense_bytes / (dense_ms / 1e3) / 1e9 / peak, "replays": len(td),
                    "clocks": clkd.summary()}
                del Kd, Vd, gd
                torch.cuda.empty_cache()

    # ---------------- block-sparse prefill (README "Sub-Quadratic Prefill") beside dense causal prefill
    if not args.no_prefill and args.layers is None:
        pw = synth.WORKLOADS["32k"]
        T, ktop = args.prefill_tokens, pw.top_k
        Bp, Hq, Hkv, d = 1, pw.n_q_heads, pw.n_kv_heads, pw.head_dim
        gen = torch.Generator(device=dev).manual_seed(4242 + rank)
        qp = torch.randn(Bp, Hq, T, d, generator=gen, device=dev).half()
        Kp = torch.randn(Bp, Hkv, T, d, generator=gen, device=dev).half()
        Vp = torch.randn(Bp, Hkv, T, d, generator=gen, device=dev).half()
        op = torch.empty(Bp, Hq, T, d, dtype=torch.float32, device=dev)
        lp = torch.empty(Bp, Hq, T, dtype=torch.float32, device=dev)
        res = {}
        for tk in (ktop, 0):
            wsp = torch.zeros(max(256, dkv.dkv_prefill_workspace_bytes(Bp, Hq, Hkv, d, T, tk)), dtype=torch.uint8,
                              device=dev)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    dkv.dkv_prefill_attend(qp, Kp, Vp, tk, out=op, lse=lp, routed=False, workspace=wsp, stream=sh)
            stream.synchronize()
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp, stream=stream):
                dkv.dkv_prefill_attend(qp, Kp, Vp, tk, out=op, lse=lp, routed=False, workspace=wsp, stream=sh)
            with torch.cuda.stream(stream):
                gp.replay()
            stream.synchronize()
            tp, clkp = timed(gp, reps)
            res[tk] = (statistics.median(tp), clkp.summary())
            log(f"[bench] prefill {T} tokens top-K {tk}: {res[tk][0]:.3f} ms")
            del gp, wsp
        nb = -(-T // 256)
        pairs = lambda k: sum((min(T, (i + 1) * 256) - i * 256) * (min(T, (i + 1) * 256) - i * 256 + 1) // 2 +
                              (min(T, (i + 1) * 256) - i * 256) * (i if (k == 0 or k >= i) else k) * 256
                              for i in range(nb))
        flops = lambda k: 4.0 * d * pairs(k) * Bp * Hq  # q.k and p.v, 2d flops each per scored pair
        tf_peak = float(json.load(open(peaks_path))["bf16_tflops"]) if os.path.exists(peaks_path) else 1900.0
        ms_s, ms_d = res[ktop][0], res[0][0]
        configs["prefill32k"] = {
            "workload": f"block-sparse prefill, batch {Bp}, {Hq}q/{Hkv}kv x d{d}, {T} tokens, top-K {ktop} earlier "
                        f"256-token blocks per query block (random fp16 q, K, V)",
            "kernel": "prefill_stats + prefill_route + prefill_attend_tc (tcgen05, fp16 operands, P as fp16 hi + lo, fp32 accumulation in tensor memory)",
            "ms_per_call": ms_s, "tokens_per_s": Bp * T / (ms_s / 1e3),
            "tflops": flops(ktop) / (ms_s / 1e3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": flops(ktop) / (ms_s / 1e3) / 1e12, "peak": tf_peak,
                         "unit": "TFLOP/s", "frac": flops(ktop) / (ms_s / 1e3) / 1e12 / tf_peak,
                         "peak_source": "measured bf16 dense (MEASURED_PEAKS.json; fp16 has the same nominal rate)",
                         "flops_per_call": flops(ktop)},
            "dense_causal_ms_per_call": ms_d,
            "dense_causal_tflops": flops(0) / (ms_d / 1e3) / 1e12,
            "speedup_vs_dense_causal": ms_d / ms_s,
            "scored_pairs_fraction": pairs(ktop) / pairs(0),
            "replays": reps, "clocks": res[ktop][1]}
        del qp, Kp, Vp, op, lp
        torch.cuda.empty_cache()

    # ---------------- streaming append (README "Core Architecture": the window's oldest 256 tokens
    # become a new block when it overflows): one token per (sequence, KV head) per call
    if not args.no_append and args.layers is None:
        n_cyc = 2
        wa = dataclasses.replace(synth.WORKLOADS["64k"], name="append64k", n_blocks=synth.WORKLOADS["64k"].n_blocks + n_cyc)
        nb0, W0, ra = wa.n_blocks - n_cyc, wa.window, wa.rank(0)
        T0 = nb0 * 256 + W0
        Ka, Va = synth.layer_kv_torch(wa, 0, dev, replica=rank)
        desc_a = dkv.dkv_layout(wa.batch, wa.n_q_heads, wa.n_kv_heads, wa.head_dim, nb0, W0, ra, wa.n_residual,
                                block_capacity=wa.n_blocks, window_capacity=W0)
        ws_a = torch.zeros(max(dkv.dkv_append_workspace_bytes(desc_a), dkv.dkv_compress_workspace_bytes(desc_a), 256),
                           dtype=torch.uint8, device=dev)
        cache_a = torch.empty(desc_a.total_bytes, dtype=torch.uint8, device=dev)
        dkv.dkv_compress_layout(desc_a, Ka[:, :, :T0].contiguous(), Va[:, :, :T0].contiguous(), cache=cache_a,
                                workspace=ws_a)
        # the appended tokens, one contiguous [B, Hkv, 1, d] slab per call
        Kn = Ka[:, :, T0:].permute(2, 0, 1, 3).contiguous().unsqueeze(3)
        Vn = Va[:, :, T0:].permute(2, 0, 1, 3).contiguous().unsqueeze(3)
        del Ka, Va
        n_new = Kn.shape[0]
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_new)]
        cut = []
        torch.cuda.synchronize()
        with ClockSampler(local) as clka, torch.cuda.stream(stream):
            for i in range(n_new):
                if i % 64 == 0:
                    # keep the stream busy while the host queues the next calls, so that each event
                    # pair spans device time only
                    stream.synchronize()
                    torch.cuda._sleep(20_000_000)
                cut.append(desc_a.window == W0)
                ev[i][0].record(stream)
                dkv.dkv_append(desc_a, Kn[i], Vn[i], cache_a, workspace=ws_a, stream=sh)
                ev[i][1].record(stream)
            stream.synchronize()
        st_a, word_a = dkv.dkv_get_error(ws_a)
        if st_a != dkv.DKV_OK:
            raise RuntimeError(f"append raised device error word {word_a:#x}")
        if (desc_a.n_blocks, desc_a.window) != (wa.n_blocks, W0):
            raise RuntimeError("append left an unexpected (n_blocks, window)")
        ta = [e0.elapsed_time(e1) * 1e3 for e0, e1 in ev]
        t_cut = [t for t, c in zip(ta, cut) if c]
        t_tok = [t for t, c in zip(ta, cut) if not c]
        units_a = wa.batch * wa.n_kv_heads
        amort = sum(ta) / n_new
        # a cut reads the 256 oldest window tokens (K and V) and writes the block and its router box
        blk_bytes = 256 * 4 * wa.head_dim + int(desc_a.block_stride) + 4 * wa.head_dim
        configs["append64k"] = {
            "workload": (f"streaming append into the 64k layer-0 cache: batch {wa.batch}, {wa.n_kv_heads} KV heads x "
                         f"d{wa.head_dim}, r {ra}, R {wa.n_residual}, window {W0}; {n_new} calls of one token per "
                         f"(sequence, KV head), every 256th compressing the window's oldest 256 tokens into a new "
                         f"block"),
            "kernel": "append_write (window row store) / append_compress (GPU block compression + window slide)",
            "token_us_median": statistics.median(t_tok), "cut_us_median": statistics.median(t_cut),
            "amortised_us_per_token": amort, "sequence_tokens_per_s": wa.batch / (amort / 1e6),
            "calls": n_new, "cuts": len(t_cut),
            "cut_bytes_min": units_a * blk_bytes,
            "cut_gbs": units_a * blk_bytes / (statistics.median(t_cut) / 1e6) / 1e9,
            "timing": "events around each call on its stream, queued behind a sleep kernel (device time only)",
            "clocks": clka.summary()}
        log(f"[bench] append: token {configs['append64k']['token_us_median']:.1f} us, "
            f"cut {configs['append64k']['cut_us_median']:.1f} us")
        del Kn, Vn, cache_a, ws_a
        torch.cuda.empty_cache()

    # ---------------- reduce over ranks (max time)
    if world > 1:
        ms, e2e_ms, e2e_ms_serial, ms_ev = max_over_ranks([ms, e2e_ms, e2e_ms_serial, ms_ev], dev)
        if alt is not None:
            alt["ms"], alt["ms_ev"], alt["attend_ms_mean"] = max_over_ranks(
                [alt["ms"], alt["ms_ev"], alt["attend_ms_mean"]], dev)
    ms_step = ms / K_steps
    value = whole_job_rate(world, queries_per_step, K_steps, ms)
    e2e_value = whole_job_rate(world, queries_per_step, e2e_steps, e2e_ms)
    e2e_serial_value = whole_job_rate(world, queries_per_step, e2e_steps, e2e_ms_serial)

    att_ms_mean = statistics.fmean(attend_ms)
    att_ms_bracketed = statistics.fmean(R["attend_ms_bracketed"])
    achieved_gbs = (att_bytes_step / n_layers) / (att_ms_mean / 1e3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "attend_traffic.json")
    if os.path.exists(tpath):
        # ncu's DRAM bytes per launch, valid while the kernel's source file is the one measured
        src_name = "attend.cu" if args.layout == "fragment" else "attend_tc.cu"
        src = open(os.path.join(ROOT, "compressed_kv_cache_dkv_gb300", "csrc", src_name), "rb").read()
        sha = hashlib.sha1(src).hexdigest()
        for entry in json.load(open(tpath)).get("captures", []):
            if entry.get("source") == src_name and entry.get("source_sha1") == sha and entry.get("config") == w.name:
                traffic = entry.get("bytes_per_launch")
    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": K_steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": wl_name, "cache_layout": args.layout,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {S.cache_gb:.1f} GB of packed caches per step cycle, each "
                         f"{'cache replica' if S.n_rep > 1 else 'layer'} read once per step",
                   "graph": f"K steps captured in one CUDA graph; value from the median of {reps} replays"},
        "hbm_gbs": step_bytes / (ms_step / 1e3) / 1e9,
        "hbm_frac_of_measured": step_bytes / (ms_step / 1e3) / 1e9 / peak,
        "hbm_frac_of_nominal_8tbs": step_bytes / (ms_step / 1e3) / 1e9 / 8000.0,
        "bytes_per_step": step_bytes,
        "single_call_latency_us": R["latency_us"],
        "roofline": {"bound": "hbm", "kernel": kernel_names[args.layout], "achieved": achieved_gbs,
                     "peak": peak, "unit": "GB/s", "frac": achieved_gbs / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
                     "bytes_per_launch": att_bytes_step / n_layers, "mean_launch_us": att_ms_mean * 1e3,
                     "timed_in": "a replay of the same K steps as stage calls: per step every call's router, "
                                 "then all the attention grids back to back in plain stream order between one "
                                 "pair of events (time per launch = region / calls), then the combines",
                     "mean_launch_us_bracketed": att_ms_bracketed * 1e3,
                     "bracketed_in": "a replay with events around every attention launch",
                     "bracket_overhead_us": R["bracket_ms"] * 1e3,
                     "launches_per_call": max(launches_per_call),
                     "ms_per_step_with_events": ms_ev / K_steps,
                     "clocks": R["clocks_ev"]},
        "e2e": {"value": e2e_value, "unit": "queries/s", "steps": e2e_steps,
                "h2d_bytes_per_step": q_host_bytes, "d2h_bytes_per_step": o_host_bytes,
                "copies": "own streams, two buffers each way, overlapping the decode kernels",
                "serial_value": e2e_serial_value},
        "gpu_launches": K_steps * sum(launches_per_call),
        "clocks": R["clocks"],
        "setup_s": t_setup,
        "replays_ms": [round(x, 4) for x in R["ms_replays"]],
        "configs": configs or None,
        "other_layout": None if alt is None else {
            "layout": alt["layout"], "kernel": alt["kernel"], "ms_per_step": alt["ms"] / K_steps,
            "value": whole_job_rate(world, queries_per_step, K_steps, alt["ms"]),
            "mean_call_us": alt["attend_ms_mean"] * 1e3, "mean_call_us_bracketed": alt["attend_ms_bracketed"] * 1e3,
            "achieved_gbs": (att_bytes_step / n_layers) / (alt["attend_ms_mean"] / 1e3) / 1e9,
            "frac": (att_bytes_step / n_layers) / (alt["attend_ms_mean"] / 1e3) / 1e9 / peak,
            "ms_per_step_with_events": alt["ms_ev"] / K_steps, "clocks": alt["clocks"]},
    }
    ext.close()
    if rank == 0 and not args.no_cpu_baseline:
        # all host cores (one spawned process per core, one unit each), then one core
        n_cores = host_cores()
        cb = cpu_oracle(w.name, 0, args.cpu_seconds, top_k, n_proc=n_cores)
        log(f"[bench] oracle on {n_cores} host cores timed")
        cb1 = cpu_oracle(w.name, 0, args.cpu_seconds, top_k) if n_cores > 1 else cb
        log("[bench] oracle on one host core timed")
        line["cpu_baseline"] = {"value": cb["qps"], "unit": "queries/s", "cores": cb["cores"], "kind": "oracle",
                                "sample": f"fp64 oracle decode of {cb['cores']} units of layer 0 ({w.group} queries "
                                          f"each), one spawned process per host core, each repeated for "
                                          f"{cb['seconds']:.1f} s; oracle compression ({cb['compress_s']:.1f} s) "
                                          f"excluded",
                                "single_core": {"value": cb1["qps"], "unit": "queries/s", "cores": 1}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
