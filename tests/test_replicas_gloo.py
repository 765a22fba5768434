"""bench.py's multi-rank logic on CPU: two gloo ranks, replicas of the same
per-GPU workload with no data-path collective; the step time is the max over
ranks and only rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(10.0 + rank, world, "cpu")

        class A:  # the reference arm on a non-zero rank does no work
            config, seed, steps, warmup = "tiny", 0, 1, 3
        if rank != 0:
            bench.run_reference(A, world, rank)
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 11.0, 1: 11.0}


def test_bench_gpus_2_starts_two_ranks():
    """`bench.py --gpus 2` without a torchrun environment starts the two
    ranks itself (torch.distributed.run, gloo on CPU for the reference arm);
    rank 0 alone prints one line, for the whole job."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--config", "tiny", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    # the line the driver parses: every key of the bench contract, with the
    # reference arm's own e2e (no host copies) and its cpu_baseline
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["steps"] == 1 and rec["warmup"] == 3 and rec["higher_is_better"] is True
    assert rec["scaling"] == "weak" and rec["vs_baseline"] is None
    assert rec["value"] > 0 and rec["ms_per_step"] > 0
    assert "workload" in rec["config"] and "N=16" in rec["config"]["workload"]
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == rec["value"] and cb["cores"] >= 1
    assert rec["e2e"] == {"value": rec["value"], "unit": rec["unit"],
                          "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
