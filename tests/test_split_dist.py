"""The split step's decomposition across processes, on CPU (gloo, 2 ranks).

The page runs one worker per GPU and sums P and Q by all-reduce (PowerSGD
review page, main findings, bullets 1 and 6).  The library's split step
(psgd_step_begin / mid / end) computes, per process, the sum of its own
workers' M_w Q, then -- after the caller's all-reduce -- Gram-Schmidt of the
summed P, its workers' Q_w and (1 / W_total) sum of them, then -- after the
second all-reduce -- U.  This test runs that decomposition with the
oracle's own functions on two gloo ranks holding two workers each, and
checks that it gives the oracle's single-process W = 4 step: the reading
that the split step is the same step, which rests on the compression being
linear in M (proposed method, bullet 2).  The GPU test of the library's
calls is tests/test_gpu_split.py.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import workloads
from oracle import powersgd as O

WORLD = 2
LOCAL = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _all_reduce(x: np.ndarray) -> np.ndarray:
    import torch
    import torch.distributed as dist
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    dist.all_reduce(t)
    return t.numpy()


def _rank_main(rank, port, steps, errq):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        cfg = workloads.scaled(workloads.c1_single_matrix(), [(90, 40), (17, 0), (33, 70)], rank=2,
                               workers=WORLD * LOCAL)
        full = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
        mine = range(rank * LOCAL, (rank + 1) * LOCAL)
        E = {li: {w: np.zeros((n, m)) for w in mine} for li, (n, m) in enumerate(cfg.layers) if m}
        Q = {li: full.Q[li].copy() for li in E}
        sig = {}
        worst = 0.0
        for t in range(steps):
            grads = workloads.gradients(cfg, t, sig)
            ref = full.step(grads)
            for li, (n, m) in enumerate(cfg.layers):
                if m == 0:
                    u = _all_reduce(sum(np.asarray(grads[w][li], np.float64) for w in mine) / cfg.workers)
                    worst = max(worst, np.abs(u - ref.U[li]).max())
                    continue
                M = {w: np.asarray(grads[w][li], np.float64) + E[li][w] for w in mine}
                P = _all_reduce(sum(M[w] @ Q[li] for w in mine))            # first all-reduce
                Ph = O.gram_schmidt(P)
                Qw = {w: M[w].T @ Ph for w in mine}
                Qbar = _all_reduce(sum(Qw.values()) / cfg.workers)           # second all-reduce
                U = Ph @ Qbar.T
                for w in mine:
                    E[li][w] = M[w] - Ph @ Qw[w].T
                    worst = max(worst, np.abs(E[li][w] - full.E[li][w]).max())
                    worst = max(worst, np.abs(Qw[w] - ref.Q_w[li][w]).max())
                Q[li] = Qbar
                for got, want in ((Ph, ref.Phat[li]), (Qbar, ref.Qbar[li]), (U, ref.U[li])):
                    worst = max(worst, np.abs(got - want).max())
        errq.put((rank, worst))
    except Exception as e:  # pragma: no cover - reported to the parent
        errq.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def test_split_step_equals_single_step_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    errq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, 3, errq)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = [errq.get(timeout=240) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst in results:
        assert not isinstance(worst, str), (rank, worst)
        # float64 on both sides; only the summation order differs
        assert worst < 1e-10, (rank, worst)
