"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank decodes its own shard of sequences (no collective on the data path);
the only cross-rank operations are a barrier around the timed region and the
maximum of the ranks' times. These tests run them with world size 2 and check
the reference arm's rank rule (rank 0 reports, the others do no work).
"""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world)  # rank 1 is the slowest
        bench.barrier(world)
        out[rank] = t
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        ps = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(120)
        assert all(p.exitcode == 0 for p in ps), [p.exitcode for p in ps]
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)  # no-op without a process group


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched like the multi-GPU run: rank 0 prints
    one JSON line, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "3", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # a whole step of the workload is batch / (sampled fraction) sampled steps
    frac = 8 / 128  # one sequence, 8 of the layer's 128 heads per sampled step
    assert abs(d["ms_per_workload_step"] - d["ms_per_step"] * 256 / frac) <= 0.05 * d["ms_per_workload_step"]
    assert abs(d["ms_per_workload_step"] - 1e3 * 256 / d["value"]) <= 0.01 * d["ms_per_workload_step"]
