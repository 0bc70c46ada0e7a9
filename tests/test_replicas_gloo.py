"""The multi-GPU path is replicas only (independent (batch, head) problems, no exchange step):
the host logic bench.py runs under torchrun - per-rank inputs, the slowest rank's time, the
whole-job rate - checked with two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from exact_attention_gb300 import synth
        import oracle
        # each rank times a different amount of "work"; the job is as slow as the slowest rank
        t_max = bench.max_over_ranks(0.5 + rank, world, device="cpu")
        rate = bench.whole_job_rate(100.0, 10, t_max, world)
        # each rank draws its own replica of the workload (seed = rank), and solves it alone
        q, k, v = synth.attention_inputs(1, 1, 16, 24, 8, "f16", seed=rank)
        o, lse = oracle.forward(synth.to_f64(q[0, 0], "f16"), synth.to_f64(k[0, 0], "f16"),
                                synth.to_f64(v[0, 0], "f16"), 0.25, False)
        bench.barrier(world)
        out[rank] = (t_max, rate, float(q.astype(np.float64).sum()), float(o.sum()), float(lse.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork: this process may already hold a CUDA context
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert sorted(out.keys()) == [0, 1]
    (t0, r0, q0, o0, l0), (t1, r1, q1, o1, l1) = out[0], out[1]
    assert t0 == t1 == 1.5                      # max over ranks
    assert r0 == r1 == pytest.approx(2 * 10 * 100.0 / 1.5)  # whole job: both ranks' units / slowest time
    assert q0 != q1 and o0 != o1 and l0 != l1   # the replicas are different problems
