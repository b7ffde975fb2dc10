"""GPU parity of the unbiased rank-r variant (psgd_options.unbiased) against
the oracle's unbiased_step, through the C ABI.

Tolerance: 1e-4 relative Frobenius error on P and U every step (there is no
state carried between steps, so no drift); the step's Q is the same draw
on both sides (float32 from the same double-precision Box-Muller values).
"""
import numpy as np
import pytest

import workloads
from oracle import powersgd as O
from tests.harness import GpuRun, rel_fro

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_gradient_compression_layer_gb300 import build
    build()


def _check(cfg, steps):
    run = GpuRun(cfg, unbiased=True)
    try:
        sig = {}
        for t in range(steps):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads)
            ref = O.unbiased_step(grads, cfg.layers, cfg.rank, cfg.seed, t)
            for li, (n, m) in enumerate(cfg.layers):
                assert rel_fro(run.update(li), ref.U[li]) <= TOL, (t, li, "U")
                if m:
                    P, Q = run.PQ(li)
                    np.testing.assert_allclose(Q, ref.Qbar[li], rtol=2.5e-7, atol=1e-30)
                    assert rel_fro(P, ref.Phat[li]) <= TOL, (t, li, "P")
        s = run.ctx.stats()
        assert s["floats_sent_per_step"] == O.unbiased_data_sent(cfg.layers, cfg.rank)
        assert s["launches_per_step"] == 3
    finally:
        run.close()


@pytest.mark.parametrize("rank", [1, 2, 3, 8, 16])
def test_unbiased_matches_oracle(rank):
    layers = [(64, 27), (128, 576), (9, 0), (257, 650), (40, 512), (3, 0)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=rank, workers=3, seed=17)
    _check(cfg, 3)


def test_unbiased_resnet18_full_set():
    _check(workloads.scaled(workloads.c2_resnet18(), workloads.resnet18_cifar_layers(), name="resnet18"), 2)


def test_unbiased_keeps_no_state():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PsgdError
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(30, 20)], rank=2, workers=2)
    run = GpuRun(cfg, unbiased=True)
    try:
        run.step(workloads.gradients(cfg, 0))
        assert np.all(run.E(0, 1) == 0.0)
        with pytest.raises(PsgdError) as ei:
            run.ctx.get_Qw(0, 0)
        assert ei.value.code == PSGD_ERR_INVALID
        with pytest.raises(PsgdError):
            run.ctx.set_state(0, torch.zeros(20, 2))
    finally:
        run.close()
