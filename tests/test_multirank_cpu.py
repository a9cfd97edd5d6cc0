"""Host-side logic of bench.py's multi-rank (torchrun) mode, on CPU with gloo.

Each rank times its own batch shard (weak scaling); the job's time is the slowest
rank's, and its throughput counts every rank's work.  The only collectives are the
timing barrier and that max.  These tests run two gloo ranks on the CPU; the GPU
kernels play no part.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shards_partition_the_global_batch():
    wl = si.tiny_conv3d()
    world = 2
    shards = [bench.shard_inputs(wl, r, world) for r in range(world)]
    x = wl.spec("x")
    glob = si.draw(wl.seed, 0, (x.shape[0] * world,) + tuple(x.shape[1:]), x.dist)
    np.testing.assert_array_equal(np.concatenate([s["x"] for s in shards]), glob)
    # weights and bias come after the whole global x in the stream and are shared
    for name in ("w", "b"):
        np.testing.assert_array_equal(shards[0][name], shards[1][name])
    # a single rank's inputs are the workload's own draws
    one = bench.shard_inputs(wl, 0, 1)
    own = wl.generate_all()
    for name in own:
        np.testing.assert_array_equal(one[name], own[name])


def test_job_throughput_counts_every_rank():
    assert bench.job_gflops(2e9, 1, 1000.0) == pytest.approx(2000.0)
    assert bench.job_gflops(2e9, 4, 1000.0) == pytest.approx(8000.0)


def _max_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        q.put((rank, bench.max_over_ranks(1.5 + 2.0 * rank, True, device="cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}
    assert bench.max_over_ranks(2.5, False) == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "tiny"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("workload", ["tiny", "conv3d_s2"])
def test_reference_arm_json_line(workload):
    # Rank 0 (or no launcher): one JSON line with the benchmark contract's keys, the
    # oracle timed on a bounded sample of the workload.
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", workload], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
