"""The multi-process (N > 1) path of bench.py on CPU with the gloo backend.

The GEMM has no exchange step, so N GPUs run N independent replicas; what
the N > 1 path adds is the rendezvous, the barriers around the timed region,
the max-over-ranks of the elapsed time and the whole-job aggregation. These
run here as two gloo ranks on the CPU; the reference arm is also run under
torchrun with two ranks (rank 0 alone works and prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    elapsed = 10.0 + 5.0 * rank                      # rank 1 is the slower one
    slowest = bench.max_over_ranks(w, elapsed)
    value = bench.replica_value(2.0e12, 4, w, slowest)
    out.put((rank, slowest, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 15.0
        # 2 ranks × 4 steps × 2 TFLOP in 15 ms
        assert abs(value - 2 * 4 * 2.0 / 0.015) < 1e-6


def test_single_process_aggregation():
    assert bench.max_over_ranks(1, 3.5) == 3.5
    assert abs(bench.replica_value(1e12, 10, 1, 5.0) - 2000.0) < 1e-9


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--workload", "gemm_256", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["value"] > 0
    import synth
    # the same config as the GPU arm's line at this N (the kernel's choices sit apart, in kernel_config)
    assert d["config"] == bench.workload_config(synth.WORKLOADS["gemm_256"], 2)
    assert d["config"]["parallelism"] == "replicas"
