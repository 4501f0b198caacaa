"""Host-side logic of the multi-GPU benchmark, run as world-size-2 gloo ranks on CPU.

Each rank processes its own batch (weak scaling); the only communication is a barrier and the
max-reduction of the timed region, so the job time is the slowest rank's.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.rank_info()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 10.0 + rank)       # rank 1 is the slow one
    out[rank] = (r, w, local, slowest)
    dist.destroy_process_group()


def test_two_rank_barrier_and_max():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][:3] == (0, 2, 0) and res[1][:3] == (1, 2, 1)
    assert res[0][3] == res[1][3] == 11.0


def test_weak_scaling_value():
    import bench
    import workloads
    w = workloads.get("headline")
    ops = bench.step_ops(w)
    assert ops == 14.0 * 2 * 16 * 8192 * 8192 * 128
    assert bench.step_ops(workloads.get("headline", causal=True)) == ops / 2
    assert bench.fwd_ops(w) + bench.bwd_ops(w) == ops
    # quantise call: Q, K, V read once, int8 codes and their fp16 operand copies written, float32
    # block scales and the K mean
    n = 2 * 16 * 8192 * 128
    small = 4 * (3 * 2 * 16 * 128 + 2 * 16 * 128)
    assert bench.quant_bytes(w) == 15 * n + small
    assert bench.quant_bytes(w, ops16=False) == 9 * n + small


def test_qat_step_ops_and_cli():
    """The Attn-QAT leg counts the method's 16 B H N^2 d tensor ops a step (6 forward: S, P^ V',
    P~ V'; 10 backward), halved when causal, and the CLI offers it."""
    import subprocess
    import sys
    import bench
    import workloads
    w = workloads.get("headline")
    assert bench.qat_step_ops(w) == 16.0 * 2 * 16 * 8192 * 8192 * 128
    assert bench.qat_step_ops(workloads.get("headline", causal=True)) == bench.qat_step_ops(w) / 2
    assert bench.qat_step_ops(w) == bench.step_ops(w) + 2.0 * 2 * 16 * 8192 * 8192 * 128
    out = subprocess.run([sys.executable, "bench.py", "--help"], capture_output=True, text=True,
                         cwd=bench.ROOT, timeout=120).stdout
    assert "--qat" in out
