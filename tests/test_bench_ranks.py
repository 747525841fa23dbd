"""The benchmark's multi-rank logic on CPU: two gloo ranks (world size 2).

Each rank runs its own copy of the workload (weak scaling: the (sequence,
head) units are independent, so there is no data-path collective); the job's
time is the slowest rank's and the job's throughput counts every rank's
units.  These checks run the same helpers bench.py uses, with the gloo
backend in place of NCCL.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from chunked_gated_delta_kda_gb300.inputs import WORKLOADS, custom, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        w_, r_, l_ = bench.rank_env()
        local_ms = 10.0 + 5.0 * rank                       # rank 1 is the slower one
        slowest = bench.max_over_ranks(local_ms, "cpu", w_)
        rate = bench.job_rate(1000, w_, slowest)
        # every rank draws its own inputs (seed offset = rank)
        x = make_inputs(custom("r", B=1, T=128, H=1, seed=3), seed_offset=r_)
        dist.barrier()
        out[rank] = (w_, r_, l_, slowest, rate, float(x["q"].float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][:3] == (2, 0, 0) and res[1][:3] == (2, 1, 1)
    for r in range(2):
        assert res[r][3] == 15.0                         # max over ranks
        assert res[r][4] == pytest.approx(2 * 1000 / 15e-3)
    assert res[0][5] != res[1][5]                        # ranks hold different data


def test_single_rank_identity():
    assert bench.max_over_ranks(7.5, "cpu", 1) == 7.5
    assert bench.job_rate(2_097_152, 1, 2.0) == pytest.approx(2_097_152 / 2e-3)
