"""The fused step (options.fused: one launch per step at padded rank <= 4) on the GPU.

The fused step against the oracle and against the four phase kernels (the
same tile bodies; only the back-project's row grouping, the project tile
rows and so the float32 summation order differ), its launch count, and the
bounded wait:
a flag that is never raised (a test hook) must end the step with
PSGD_ERR_TIMEOUT at the next synchronising call, leave the CUDA context
usable, and a new context must then run normally.
"""
import numpy as np
import pytest

import workloads
from oracle import powersgd as O
from tests.harness import GpuRun, compare_step, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_gradient_compression_layer_gb300 import build
    build()


@pytest.mark.parametrize("rank,workers", [(1, 2), (2, 4), (4, 3), (3, 9)])
def test_fused_matches_four_launches(rank, workers):
    cfg = workloads.scaled(workloads.c2_resnet18(), workloads.c2_resnet18().layers, rank=rank, workers=workers)
    fused, four = GpuRun(cfg, fused=True), GpuRun(cfg)
    try:
        assert fused.ctx.fused and not four.ctx.fused
        assert fused.ctx.stats()["launches_per_step"] == 1
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            fused.step(grads)
            four.step(grads)
            for li, (n, m) in enumerate(cfg.layers):
                assert rel_fro(fused.update(li), four.update(li)) <= 1e-5, (t, li, "U")
                if m == 0:
                    continue
                Pf, Qf = fused.PQ(li)
                P4, Q4 = four.PQ(li)
                assert rel_fro(Pf, P4) <= 1e-5 and rel_fro(Qf, Q4) <= 1e-5, (t, li)
                for w in range(workers):
                    assert rel_fro(fused.E(li, w), four.E(li, w)) <= 1e-5, (t, li, "E", w)
    finally:
        fused.close()
        four.close()


def test_fused_resnet18_ten_steps_against_oracle():
    cfg = workloads.c2_resnet18()
    run = GpuRun(cfg, fused=True)
    st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
    try:
        sig = {}
        for t in range(10):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads)
            ref = st.step(grads)
            if t in (0, 4, 9):
                worst, bad = compare_step(run, ref, st, 1e-4 if t == 0 else 1e-3, grads=grads)
                assert not bad, (t, sorted(bad.items(), key=lambda kv: -kv[1])[:5])
    finally:
        run.close()


def test_fused_without_update_and_timing():
    # no update buffer: the queue without the decompress tiles; timing: one
    # slot for the whole launch
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(300, 200), (64, 0), (1000, 130)], rank=2, workers=3)
    run = GpuRun(cfg, timing=True, fused=True)
    st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
    try:
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads, update=(t == 2))
            ref = st.step(grads)
        worst, bad = compare_step(run, ref, st, 1e-3, grads=grads)
        assert not bad, bad
        pt = run.ctx.phase_times()
        assert set(pt) == {"step"} and pt["step"] > 0
    finally:
        run.close()


def test_wait_that_runs_out_reports_timeout():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_TIMEOUT, PsgdError

    cfg = workloads.scaled(workloads.c2_resnet18(), [(256, 1152), (64, 576), (10, 0)], rank=2, workers=4)
    # layer 1's R flag is never raised: its orthonormalise tiles wait 50 ms
    run = GpuRun(cfg, fused=True, wait_ms=50, test_stall=2)
    try:
        grads = workloads.gradients(cfg, 0, {})
        run.load(grads)
        run.ctx.step(run.bufs, run.upd)
        with pytest.raises(PsgdError) as ei:
            run.ctx.sync()
        assert ei.value.code == PSGD_ERR_TIMEOUT
        with pytest.raises(PsgdError):  # the context stays unusable
            run.ctx.get_PQ(0)
    finally:
        run.close()
    torch.cuda.synchronize()  # the CUDA context is fine
    # and a new context runs normally
    run = GpuRun(cfg, fused=True)
    st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
    try:
        grads = workloads.gradients(cfg, 0, {})
        run.step(grads)
        ref = st.step(grads)
        worst, bad = compare_step(run, ref, st, 1e-4, grads=grads)
        assert not bad, bad
        assert np.isfinite(worst)
    finally:
        run.close()
