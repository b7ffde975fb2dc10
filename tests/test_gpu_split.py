"""The split step (psgd_step_begin / mid / end) on the GPU.

1. One process, the identity as all-reduce: the split step must give what a
   one-kernel-per-phase context gives (the same kernels on the same values:
   matrix layers bit for bit; vector means differ only in how the 1 / W
   scale is applied, so to float32 rounding).  The split step has no
   one-pass project: P is all-reduced before its rows are complete.
2. Two processes sharing cuda:0, two workers each, with the all-reduces of
   P and of Q done by gloo (host copies): every process must match the
   oracle's single-process W = 4 step (PowerSGD review page, main findings,
   bullets 1 and 6: one worker per GPU, P and Q summed by all-reduce).
   The two processes never wait on each other's kernels: each process's
   collective runs on the host between its own kernels.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import workloads
from oracle import powersgd as O
from tests.harness import GpuRun, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_gradient_compression_layer_gb300 import build
    build()


@pytest.mark.parametrize("rank,workers", [(2, 4), (4, 3), (16, 2)])
def test_split_step_with_identity_exchange_matches_step(rank, workers):
    base = workloads.c2_resnet18()
    layers = [(64, 27), (128, 576), (32, 0), (512, 4608), (10, 0), (256, 128)]
    cfg = workloads.scaled(base, layers, rank=rank, workers=workers)
    split, ref = GpuRun(cfg), GpuRun(cfg)
    try:
        p, q = split.ctx.exchange_sizes()
        assert p == sum(n * rank for n, m in layers if m)
        assert q == sum(m * rank for n, m in layers if m) + sum(n for n, m in layers if m == 0)
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            split.load(grads)
            split.ctx.step_split(split.bufs, split.upd)
            split.ctx.sync()
            ref.step(grads)
            for li, (n, m) in enumerate(layers):
                if m == 0:
                    np.testing.assert_allclose(split.update(li), ref.update(li), rtol=1e-6, atol=0)
                    continue
                assert np.array_equal(split.update(li), ref.update(li)), (t, li)
                assert all(np.array_equal(a, b) for a, b in zip(split.PQ(li), ref.PQ(li))), (t, li)
                for w in range(workers):
                    assert np.array_equal(split.E(li, w), ref.E(li, w)), (t, li, w)
        assert split.ctx.stats()["steps"] == 3
    finally:
        split.close()
        ref.close()


def test_split_calls_out_of_order_are_rejected():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PsgdError

    cfg = workloads.scaled(workloads.c1_single_matrix(), [(40, 30)], rank=2, workers=2)
    run = GpuRun(cfg, total_workers=4)
    try:
        x = torch.zeros(1024, device="cuda")
        with pytest.raises(PsgdError) as ei:
            run.ctx.step_mid(x, x)
        assert ei.value.code == PSGD_ERR_INVALID
        with pytest.raises(PsgdError):  # its workers are a share: psgd_step is refused
            run.ctx.step(run.bufs, run.upd)
    finally:
        run.close()


WORLD, LOCAL = 2, 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, errq):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from rank_gradient_compression_layer_gb300 import PowerSGD
        torch.cuda.set_device(0)
        cfg = workloads.scaled(workloads.c2_resnet18(), [(64, 27), (256, 1152), (64, 0), (512, 4608)], rank=2,
                               workers=WORLD * LOCAL)
        ctx = PowerSGD(cfg.layers, cfg.rank, LOCAL, seed=cfg.seed, total_workers=cfg.workers)
        bufs = [ctx.empty_buffer() for _ in range(LOCAL)]
        upd = ctx.empty_buffer()
        st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
        mine = list(range(rank * LOCAL, (rank + 1) * LOCAL))

        def all_reduce(t):
            c = t.cpu()
            dist.all_reduce(c)
            t.copy_(c)

        sig = {}
        worst = 0.0
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            for k, w in enumerate(mine):
                ctx.pack([torch.from_numpy(g).cuda() for g in grads[w]], out=bufs[k])
            ctx.step_split(bufs, upd, all_reduce)
            ctx.sync()
            ref = st.step(grads)
            tol = 1e-4 if t == 0 else 1e-3
            for li, (n, m) in enumerate(cfg.layers):
                errs = [rel_fro(ctx.layer_view(upd, li).cpu().numpy(), ref.U[li])]
                if m:
                    P, Q = ctx.get_PQ(li)
                    errs += [rel_fro(P.cpu().numpy(), ref.Phat[li]), rel_fro(Q.cpu().numpy(), ref.Qbar[li])]
                    for k, w in enumerate(mine):
                        errs.append(rel_fro(ctx.get_Qw(li, k).cpu().numpy(), ref.Q_w[li][w]))
                        errs.append(rel_fro(ctx.get_error(li, k).cpu().numpy(), st.E[li][w]))
                worst = max(worst, max(errs) / tol)
        ctx.close()
        errq.put((rank, worst))
    except Exception as e:  # pragma: no cover - reported to the parent
        errq.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def test_split_step_over_two_processes_matches_oracle():
    ctx = mp.get_context("spawn")
    errq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, errq)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = [errq.get(timeout=300) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst in results:
        assert not isinstance(worst, str), (rank, worst)
        assert worst <= 1.0, (rank, worst)  # every error within its step's tolerance
