"""GPU parity of the one-pass project (padded rank <= 4).

With one Cholesky-QR pass, Phat = P R^-1, so the back-projection
Q_w = M_w^T Phat equals (M_w^T P) R^-1 (proposed method, bullet 1: Q = M^T
Phat, written with Phat's factor pulled out).  The project phase
accumulates Y_w = M_w^T P while each row block's M is on chip, and the
back-project forms Q_w = Y_w R^-1 without reading M again.  Its rounding is
amplified by about kappa(P), so a layer takes this form only when
kappa_F(R) <= 128; otherwise the back-project reads M as before.  The
oracle knows nothing of this: it orthonormalises P by Gram-Schmidt and
multiplies by M_w^T, and every result must match it as in the two-pass form.
"""
import numpy as np
import pytest

import workloads
from oracle import powersgd as O
from tests.harness import GpuRun, compare_step, rel_fro

pytestmark = pytest.mark.gpu

TOL1, TOL10 = 1e-4, 1e-3

# ragged shapes (min(n, m) >= 5, above every rank tested): m not a multiple
# of 4, a row slice wider than the threads of a CTA, rows not a multiple of a
# block, tiny layers
RAGGED = [(7, 5), (33, 6), (100, 4100), (1000, 300), (64, 27), (513, 2305), (16, 0), (5, 9), (130, 130)]


def _oracle_run(cfg, steps, check_steps, **kw):
    run = GpuRun(cfg, one_pass=True, **kw)
    st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
    sig = {}
    flags = []
    try:
        for t in range(steps):
            g = workloads.gradients(cfg, t, sig)
            ref = st.step(g)
            run.step(g)
            if t in check_steps:
                worst, bad = compare_step(run, ref, st, TOL1 if t == 0 else TOL10, grads=g)
                assert not bad, (t, bad)
            flags.append({li: run.ctx.layer_flags(li) for li, (n, m) in enumerate(cfg.layers) if m})
        return flags, run.ctx.one_pass
    finally:
        run.close()


def test_one_pass_applies_at_low_rank_only():
    from rank_gradient_compression_layer_gb300 import PowerSGD

    shapes = [(64, 576), (128, 1152), (10, 0)]
    on = {"one_pass": True}
    for rank, kw, want in [(1, on, True), (2, on, True), (4, on, True), (3, on, True), (8, on, False),
                           (16, on, False), (2, {}, False), (2, dict(on, unbiased=True), False),
                           (2, dict(on, fused=True), False), (2, dict(on, compressor="rtopk"), False)]:
        ctx = PowerSGD(shapes, rank, 4, **kw)
        try:
            assert ctx.one_pass is want, (rank, kw)
        finally:
            ctx.close()


@pytest.mark.parametrize("rank,workers", [(1, 2), (2, 3), (3, 5), (4, 4), (2, 8)])
def test_one_pass_matches_oracle_on_ragged_layers(rank, workers):
    cfg = workloads.scaled(workloads.c2_resnet18(), RAGGED, rank=rank, workers=workers)
    flags, one_pass = _oracle_run(cfg, 4, check_steps=(0, 1, 3))
    assert one_pass
    # the well-conditioned large layers took the one-pass form once warm
    big = [li for li, (n, m) in enumerate(RAGGED) if m and min(n, m) >= 64]
    assert all(flags[-1][li]["q_from_y"] for li in big), flags[-1]


def test_one_pass_matches_two_pass_over_ten_steps():
    layers = [(256, 2304), (512, 4608), (64, 27), (130, 650), (10, 512)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers)
    one, two = GpuRun(cfg, one_pass=True), GpuRun(cfg)
    sig = {}
    try:
        assert one.ctx.one_pass and not two.ctx.one_pass
        for t in range(10):
            g = workloads.gradients(cfg, t, sig)
            one.step(g)
            two.step(g)
            for li in range(len(layers)):
                P1, Q1 = one.PQ(li)
                P2, Q2 = two.PQ(li)
                assert rel_fro(P1, P2) <= 1e-5, (t, li)
                assert rel_fro(Q1, Q2) <= 1e-5, (t, li)
                assert rel_fro(one.update(li), two.update(li)) <= 1e-5, (t, li)
                assert rel_fro(one.E(li, 1), two.E(li, 1)) <= 1e-4, (t, li)
            assert all(one.ctx.layer_flags(li)["q_from_y"] for li in range(len(layers)))
            assert not any(two.ctx.layer_flags(li)["q_from_y"] for li in range(len(layers)))
    finally:
        one.close()
        two.close()


def test_one_pass_lstm_layers_match_oracle():
    """kappa_F(R) near 66 on these layers (a rank-4 signal with singular
    values 4 : 2 : 1 : 0.5 under heavy-tailed noise): the one-pass form with
    its largest amplification on the page's workloads."""
    cfg = workloads.scaled(workloads.c3_lstm(), [(4096, 650), (2600, 650), (2600, 0)], steps=6)
    flags, one_pass = _oracle_run(cfg, 6, check_steps=(0, 2, 5))
    assert one_pass
    assert flags[-1][0]["q_from_y"] and flags[-1][1]["q_from_y"]


def test_ill_conditioned_layer_falls_back_to_reading_m():
    """Every worker's gradient is the same rank-1 matrix: at r = 4 the last
    three columns of P are rounding noise, kappa(P) is far past the bound,
    and the back-project must read M (q_from_y off) -- with the result still
    the oracle's U (the rank-1 gradient itself)."""
    rng = np.random.default_rng(5)
    n, m, W = 300, 200, 3
    u, v = rng.standard_normal(n), rng.standard_normal(m)
    G = np.outer(u, v).astype(np.float32)
    cfg = workloads.scaled(workloads.c2_resnet18(), [(n, m)], rank=4, workers=W)
    run = GpuRun(cfg, one_pass=True)
    st = O.OracleState(cfg.layers, 4, W, cfg.seed)
    try:
        for t in range(3):
            grads = [[G] for _ in range(W)]
            ref = st.step(grads)
            run.step(grads)
            assert not run.ctx.layer_flags(0)["q_from_y"], t
            assert rel_fro(run.update(0), ref.U[0]) <= 1e-4, t
    finally:
        run.close()


def test_one_pass_resnet18_full_set():
    cfg = workloads.c2_resnet18()
    flags, one_pass = _oracle_run(cfg, 4, check_steps=(0, 3))
    assert one_pass
    assert all(f["q_from_y"] for f in flags[-1].values()), flags[-1]
