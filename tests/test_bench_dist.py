"""bench.py's multi-rank plumbing on CPU: two gloo ranks on 127.0.0.1.

The GPU bench runs N replicas of the step (no data-path collective); what
the ranks share is the barrier and the max-over-ranks timing, checked here
without a GPU, plus the reference arm's rule that only rank 0 works.
"""
import argparse
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env() == (ws, rank, rank)
        bench.barrier(ws)
        # rank r took 10 + r ms for 4 steps, each rank compressed 1 GB per step
        ms, gbs = bench.replica_throughput(1e9, 4, 10.0 + rank, ws)
        args = argparse.Namespace(config="c1", steps=1, warmup=1, cpu_budget=0.5)
        ref = bench.run_reference(args, ws, rank)
        bench.barrier(ws)
        q.put((rank, ms, gbs, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_reference_on_rank0():
    import torch.multiprocessing as mp
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(ws):
            rank, ms, gbs, ref = q.get(timeout=120)
            out[rank] = (ms, gbs, ref)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # both ranks report the slowest rank's time: 11 ms / 4 steps
    for rank in range(ws):
        ms, gbs, _ = out[rank]
        assert ms == pytest.approx(11.0 / 4)
        assert gbs == pytest.approx(2 * 1e9 / (11.0 / 4 * 1e-3) / 1e9)
    # the reference arm: rank 0 prints one line, the other ranks do nothing
    assert out[1][2] is None
    ref = out[0][2]
    assert ref["impl"] == "reference" and ref["n_gpus"] == ws and ref["value"] > 0
    assert ref["e2e"]["h2d_bytes_per_step"] == 0 and ref["cpu_baseline"]["kind"] == "oracle"
