"""GPU parity of the step with the fused momentum-SGD update
(psgd_step_momentum) against the oracle's step followed by its
momentum_update, through the C ABI.

Tolerance: 1e-4 relative Frobenius error on params and momentum after the
first step, 1e-3 after later ones (the update inherits the step's error).
"""
import numpy as np
import pytest

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


@pytest.mark.parametrize("rank,with_update", [(2, True), (4, False), (8, True), (16, False)])
def test_momentum_update_matches_oracle(rank, with_update):
    import torch
    layers = [(64, 27), (128, 576), (9, 0), (257, 650), (20, 512), (33, 0)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=rank, workers=3)
    lr, beta = 0.5, 0.9
    run = GpuRun(cfg)
    try:
        ctx = run.ctx
        rng = np.random.default_rng(3)
        x0 = [0.01 * rng.standard_normal((n, m) if m else (n,)) for n, m in layers]
        X = ctx.pack([torch.from_numpy(v.astype(np.float32)).cuda() for v in x0])
        Mom = torch.zeros_like(X)
        # the oracle starts from the float32 values the GPU starts from
        xs = [ctx.layer_view(X, li).double().cpu().numpy() for li in range(len(layers))]
        x_start = [v.copy() for v in xs]
        ms = [np.zeros_like(v) for v in xs]
        st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
        sig = {}
        for t in range(4):
            grads = workloads.gradients(cfg, t, sig)
            run.load(grads)
            ctx.step_momentum(run.bufs, X, Mom, lr, beta, run.upd if with_update else None)
            ctx.sync()
            ref = st.step(grads)
            tol = 1e-4 if t == 0 else 1e-3
            for li in range(len(layers)):
                xs[li], ms[li] = O.momentum_update(xs[li], ms[li], ref.U[li], lr, beta)
                got_x = ctx.layer_view(X, li).double().cpu().numpy()
                got_m = ctx.layer_view(Mom, li).double().cpu().numpy()
                assert rel_fro(got_m, ms[li]) <= tol, (t, li, "momentum")
                # params: measured on what the updates moved
                assert rel_fro(got_x - x_start[li], xs[li] - x_start[li]) <= tol, (t, li, "params")
                if with_update:
                    assert rel_fro(run.update(li), ref.U[li]) <= tol, (t, li, "U")
    finally:
        run.close()


def test_momentum_leaves_padding_alone():
    import torch
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(20, 6), (5, 0)], rank=2, workers=2)
    run = GpuRun(cfg)
    try:
        ctx = run.ctx
        X = torch.zeros(ctx.total, device="cuda")
        Mom = torch.zeros_like(X)
        n, m = cfg.layers[0]
        ld = ctx.lds[0]
        X[:n * ld].view(n, ld)[:, m:] = 7.0
        Mom[:n * ld].view(n, ld)[:, m:] = -3.0
        run.load(workloads.gradients(cfg, 0))
        ctx.step_momentum(run.bufs, X, Mom, 0.1, 0.9)
        ctx.sync()
        assert torch.all(X[:n * ld].view(n, ld)[:, m:] == 7.0)
        assert torch.all(Mom[:n * ld].view(n, ld)[:, m:] == -3.0)
        assert torch.count_nonzero(ctx.layer_view(Mom, 0)) > 0
    finally:
        run.close()
