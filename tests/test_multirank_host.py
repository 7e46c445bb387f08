"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank draws
its own batch (weak scaling, no data-path collective) and the job's time is the
max over ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank sets the job time
        t = bench.max_over_ranks(10.0 + rank, world, "cpu")
        # each rank's batch differs (weak scaling), deterministically
        from randomized_norm_clipping_gb300 import workloads as wl
        wk = wl.WORKLOADS["hutch_b4_t128_64x64_k8_f32"]
        seeded = wl.Workload(**{**wk.__dict__, "seed": bench.shard_seed(wk.seed, rank)})
        A, _, _ = wl.layer_inputs(seeded, 0, device="cpu")
        sums = [torch.zeros(1) for _ in range(world)]
        dist.all_gather(sums, A.sum().reshape(1))
        bench.barrier(world)
        out[rank] = (t, [float(s) for s in sums])
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    (t0, s0), (t1, s1) = out[0], out[1]
    assert t0 == t1 == 11.0
    assert s0 == s1 and s0[0] != s0[1]
