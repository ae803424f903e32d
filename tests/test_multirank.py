"""Host logic of the multi-rank bench (weak scaling, one replica per rank) on
CPU: two gloo ranks reduce their timings to the maximum, and the whole-job rate
counts every rank's queries over the slowest rank's time.  The decode path
itself has no collective (units are independent), so nothing else crosses ranks."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed (ms, e2e_ms, ms_with_events) = (10 + r, 20 - r, 30 + 2r)
        got = bench.max_over_ranks([10.0 + rank, 20.0 - rank, 30.0 + 2 * rank], "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert out[r] == [11.0, 20.0, 32.0]


def test_whole_job_rate_counts_every_replica():
    import bench
    # 192 queries per step, 100 steps in 250 ms on each of 4 ranks -> 4 * 19200 / 0.25 s
    assert bench.whole_job_rate(4, 192, 100, 250.0) == pytest.approx(4 * 192 * 100 / 0.25)
    assert bench.whole_job_rate(1, 192, 100, 250.0) * 4 == pytest.approx(bench.whole_job_rate(4, 192, 100, 250.0))


def test_small_workloads_rotate_over_enough_cache_replicas():
    import bench
    from compressed_kv_cache_dkv_gb300 import synth
    l2 = 126 << 20
    # the 64k step reads 2 GB: no replicas
    w = synth.WORKLOADS["64k"]
    assert bench.cache_replicas(sum(bench.call_bytes(w, l, w.top_k) for l in range(w.n_layers)), l2) == 1
    # 32k and 8k read 9.0 and 1.4 MB per call: a step's reads reach 4x the L2, and one replica
    # fewer would not
    for name in ("32k", "8k"):
        w = synth.WORKLOADS[name]
        per = bench.call_bytes(w, 0, w.top_k)
        n = bench.cache_replicas(per, l2)
        assert n * per >= 4 * l2 > (n - 1) * per


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores, no GPU) prints one
    JSON line with the keys of the benchmark contract."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "8k",
           "--steps", "2", "--warmup", "3", "--cpu-seconds", "1"]
    res = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "queries/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
