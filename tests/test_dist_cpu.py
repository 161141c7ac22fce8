"""The benchmark's multi-process host logic on CPU, world size 2 (gloo): the
timing barrier and the max over ranks, the whole-job throughput, and the
reference arm printing one line from rank 0 under torchrun.  The ranks run
independent replicas (the forward shards over (b, h) with no exchange), so these
are the only collectives there are."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(None)
    bench.barrier(w)
    slowest = bench.max_over_ranks(0.25 * (r + 1), w)
    q.put((r, w, dist.get_backend(), slowest))
    dist.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks():
    import torch.multiprocessing as tmp
    ctx = tmp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get() for _ in range(2))
    assert res == [(0, 2, "gloo", 0.5), (1, 2, "gloo", 0.5)]


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tokens_per_s(1, 50, 2, 8, 2048, 0.016)
    two = bench.job_tokens_per_s(2, 50, 2, 8, 2048, 0.016)
    assert one == pytest.approx(50 * 2 * 8 * 2048 / 0.016)
    assert two == pytest.approx(2 * one)            # weak scaling at equal time
    assert bench.job_tokens_per_s(2, 50, 2, 8, 2048, 0.032) == pytest.approx(one)


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "kla_fp32_small", "--steps", "1", "--warmup", "0",
           "--cpu-sample-heads", "1"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
