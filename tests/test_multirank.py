"""The multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

The DyRA forward shards by sample with no data-path collective (every sample is its own
least-squares problem), so N GPUs run N independent replicas. What crosses ranks is only the
timing: a barrier around the timed region and the max of the step time over ranks. These
tests run that logic as two processes on the gloo backend, and the reference arm under
torchrun, where rank 0 alone runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank i took (i + 1) ms for 1000 tokens: the job's step is the slowest rank's
    value, ms = bench.weak_scaling_value(1000, float(rank + 1), w)
    out.put((rank, value, ms))
    dist.destroy_process_group()


def test_weak_scaling_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get() for _ in range(2))
    for rank, value, ms in got:
        assert ms == 2.0
        assert value == pytest.approx(2 * 1000 / 2e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.weak_scaling_value(500, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(500 / 4e-3)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "20", "--warmup", "3",
           "--config", "c1"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
