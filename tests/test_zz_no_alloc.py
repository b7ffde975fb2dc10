"""psgd_step_noalloc (one layer, caller-owned state, scratch in a fixed device
array) against psgd_step on a one-layer context, through the C ABI.

Runs last (file name) and alone: two calls in a row per shape, the first
without and the second with the previous call's state, each compared with
the context's step on the same gradients.  Tolerance: the parity tests'
1e-4 relative Frobenius error (both paths run the same kernels, so the
results are expected to agree far more closely).
"""
import numpy as np
import pytest

import workloads
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


def _noalloc_matches_context(n, m, r, W, seed):
    import torch
    from rank_gradient_compression_layer_gb300 import step_noalloc

    cfg = workloads.scaled(workloads.c2_resnet18(), [(n, m)], rank=r, workers=W, seed=seed)
    run = GpuRun(cfg)
    try:
        ld = run.ctx.lds[0]
        dev = torch.device("cuda")
        _, Q0 = run.ctx.get_PQ(0)
        B = torch.zeros(W, n, ld, device=dev)
        Phat = torch.zeros(n, r, device=dev)
        Qbar = torch.zeros(ld, r, device=dev)
        Qbar[:m] = Q0.to(dev)
        Qw = torch.zeros(W, ld, r, device=dev)
        U = torch.full((n, ld), float("nan"), device=dev)
        sig = {}
        for t in range(2):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads)
            gviews = [b[:n * ld].view(n, ld) for b in run.bufs]
            step_noalloc(n, m, r, gviews, B, Phat, Qbar, Qw, U, has_prev=t > 0)
            torch.cuda.synchronize()
            P_ref, Q_ref = run.PQ(0)
            got_P = Phat.double().cpu().numpy()
            got_Q = Qbar.double().cpu().numpy()
            got_U = U.double().cpu().numpy()
            assert rel_fro(got_P, P_ref) <= TOL, (t, "Phat")
            assert rel_fro(got_Q[:m], Q_ref) <= TOL, (t, "Qbar")
            assert np.all(got_Q[m:] == 0.0)
            assert rel_fro(got_U[:, :m], run.update(0)) <= TOL, (t, "U")
            assert np.all(got_U[:, m:] == 0.0)
            for w in range(W):
                qw = Qw[w].double().cpu().numpy()
                assert rel_fro(qw[:m], run.Qw(0, w)) <= TOL, (t, "Qw", w)
                # new error E_w = B_w - Phat Q_w^T (B_w holds M_w after the call);
                # every shape here has rank far above r, so E_w is not near zero
                E = B[w].double().cpu().numpy()[:, :m] - got_P @ qw[:m].T
                assert rel_fro(E, run.E(0, w)) <= TOL, (t, "E", w)
    finally:
        run.close()


@pytest.mark.parametrize("n,m,r,W", [
    (64, 27, 1, 2),       # one segment, ragged row (m % 4 == 3)
    (300, 130, 2, 3),     # two segments, ragged tail
    (1536, 1000, 4, 4),   # several row tiles in every phase
    (512, 4608, 2, 4),    # the largest ResNet-18 layer
    (257, 650, 8, 5),     # r = 8, odd worker count
    (1000, 300, 16, 3),   # r = 16: the register-tiled project and decompress kernels
    (511, 260, 32, 2),    # r = 32, ragged row tile
    (63, 27, 1, 2),       # n r not a multiple of 4: the caller's Phat is not padded
])
def test_noalloc_matches_context_two_calls(n, m, r, W):
    _noalloc_matches_context(n, m, r, W, seed=21)


def test_noalloc_rejects_what_it_cannot_run():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PsgdError, step_noalloc

    t = torch.zeros(64, device="cuda")
    # scratch beyond the fixed array: an 8192 x 8192 layer at r = 4, W = 8
    with pytest.raises(PsgdError) as ei:
        step_noalloc(8192, 8192, 4, [t] * 8, t, t, t, t, None)
    assert ei.value.code == PSGD_ERR_INVALID and "scratch" in str(ei.value)
    # rank must be a power of two (the kernels' rank, no padding columns)
    with pytest.raises(PsgdError) as ei:
        step_noalloc(16, 8, 3, [t] * 2, t, t, t, t, None)
    assert ei.value.code == PSGD_ERR_INVALID
    # a misaligned state pointer
    with pytest.raises(PsgdError) as ei:
        step_noalloc(16, 8, 2, [t] * 2, t[1:], t, t, t, None)
    assert ei.value.code == PSGD_ERR_INVALID
    # nothing was enqueued by the rejected calls: the device is still fine
    torch.cuda.synchronize()
