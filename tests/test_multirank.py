"""The bench's multi-rank (weak scaling) logic with world_size 2 on CPU (gloo).

bench.py --gpus N runs one process per GPU over NCCL; the path has no
data-path collective (each rank processes its own independent copy of the
workload), so what needs checking is the host logic the ranks share: rank
setup from the torchrun environment, per-rank seeds that give different
inputs, the max-over-ranks timing and the whole-job value.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    from long_context_causal_gb300.inputs import WORKLOADS, make
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world, backend="gloo")
    wl = WORKLOADS["single_head_s1k_fp32"]
    q, *_ = make(1, 1, 1, 64, 64, torch.float32, seed=bench.rank_seed(wl.seed, r))
    bench.barrier(w)
    # each rank "took" a different time; the job is as slow as its slowest rank
    slowest = bench.max_over_ranks(10.0 * (r + 1), w, device="cpu")
    value = bench.job_value(1e12, slowest, w)
    out.put((r, w, local, float(q.sum()), slowest, value))
    dist.destroy_process_group()


def test_two_ranks_share_timing_and_sum_work():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1] and all(x[1] == world and x[2] == x[0] for x in res)
    assert res[0][3] != res[1][3], "ranks must draw different inputs"
    assert all(x[4] == 20.0 for x in res), "timing is the max over ranks"
    # 2 ranks x 1e12 flop in 20 ms = 100 TFLOP/s for the whole job
    assert all(x[5] == pytest.approx(100.0) for x in res)
