"""GPU parity of rTop-k sparsification (psgd_options.compressor = PSGD_RTOPK)
against the oracle's RTopKState, through the C ABI.

Both sides compute M, E, S and U in float32 with the same operations in the
same order and select with the same integer keys, so the sent indices,
values, the error buffers and U of the matrix layers must agree exactly;
vector layers (a float64 mean in the oracle) to 1e-6.
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


def _run(cfg, top_div, sample_div, steps, grads_of=None):
    run = GpuRun(cfg, compressor="rtopk", top_div=top_div, sample_div=sample_div)
    st = O.RTopKState(cfg.layers, cfg.workers, cfg.seed, top_div, sample_div)
    try:
        sig = {}
        for t in range(steps):
            grads = grads_of(t) if grads_of else workloads.gradients(cfg, t, sig)
            run.step(grads)
            U, sent = st.step(grads)
            for li, (n, m) in enumerate(cfg.layers):
                got = run.update(li)
                if m == 0:
                    assert rel_fro(got, U[li]) < 1e-6, (t, li)
                    continue
                assert np.array_equal(got, U[li]), (t, li, "U")
                for w in range(cfg.workers):
                    idx, val = run.ctx.get_sparse(li, w)
                    idx = idx.cpu().numpy().astype(np.int64)
                    assert np.array_equal(idx, sent[li][w]), (t, li, w, "indices")
                    M_val = val.cpu().numpy()
                    E = run.E(li, w)
                    assert np.array_equal(E, st.E[li][w]), (t, li, w, "E")
                    assert len(M_val) == O.rtopk_counts(n * m, top_div, sample_div)[1]
        s = run.ctx.stats()
        assert s["floats_sent_per_step"] == O.rtopk_data_sent(cfg.layers, top_div, sample_div)
    finally:
        run.close()


@pytest.mark.parametrize("top_div,sample_div", [(4, 2), (7, 3), (1, 1), (50, 1)])
def test_rtopk_matches_oracle(top_div, sample_div):
    layers = [(12, 9), (5, 0), (37, 130), (64, 27), (300, 70)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=2, workers=3, seed=23)
    _run(cfg, top_div, sample_div, 3)


def test_rtopk_resnet18_full_set():
    cfg = workloads.scaled(workloads.c2_resnet18(), workloads.resnet18_cifar_layers(), name="resnet18")
    _run(cfg, 100, 4, 2)


def test_rtopk_ties_and_zero_gradient():
    # all-zero gradients: every magnitude ties, the top set is the lowest indices
    layers = [(20, 33), (3, 0)]
    cfg = workloads.scaled(workloads.c1_single_matrix(), layers, rank=1, workers=2, seed=4)
    zero = [[np.zeros((20, 33), np.float32), np.zeros(3, np.float32)] for _ in range(2)]
    _run(cfg, 5, 2, 2, grads_of=lambda t: zero)


def test_rtopk_host_path_message():
    import torch
    layers = [(40, 27), (4, 0), (33, 64)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=2, workers=2, seed=8)
    a = GpuRun(cfg, compressor="rtopk", top_div=6, sample_div=2)
    b = GpuRun(cfg, compressor="rtopk", top_div=6, sample_div=2)
    try:
        grads = workloads.gradients(cfg, 0)
        a.step(grads)
        host = [b.ctx.pack([torch.from_numpy(g) for g in grads[w]],
                           out=torch.zeros(b.ctx.total, dtype=torch.float32).pin_memory()) for w in range(2)]
        msg = torch.zeros(b.ctx.message_floats, dtype=torch.float32)
        b.ctx.step_host(host, msg)
        at = 0
        for li, (n, m) in enumerate(layers):
            if not m:
                continue
            for w in range(2):
                idx, val = a.ctx.get_sparse(li, w)
                k = idx.numel()
                assert torch.equal(msg[at:at + k].view(torch.int32), idx.cpu())
                assert torch.equal(msg[at + k:at + 2 * k], val.cpu())
                at += 2 * k
        assert at == msg.numel()
    finally:
        a.close()
        b.close()


def test_rtopk_rejects_factor_calls():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PowerSGD, PsgdError
    ctx = PowerSGD([(16, 8)], 2, 2, compressor="rtopk", top_div=4, sample_div=2)
    try:
        for call in (lambda: ctx.get_PQ(0), lambda: ctx.get_Qw(0, 0), lambda: ctx.set_state(0, torch.zeros(8, 2))):
            with pytest.raises(PsgdError) as ei:
                call()
            assert ei.value.code == PSGD_ERR_INVALID
    finally:
        ctx.close()
    with pytest.raises(PsgdError):
        PowerSGD([(16, 8)], 2, 2, compressor="rtopk", top_div=0)


def test_rtopk_many_steps_predicted_digit():
    # from the second step on, pass 0 may resolve the second magnitude digit
    # from the previous step's first digit; error feedback keeps the
    # threshold near it, so most of these steps take that path
    layers = [(96, 300), (7, 0), (64, 129), (33, 64)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=2, workers=2, seed=31)
    _run(cfg, 20, 3, 10)


def test_rtopk_scale_jumps_between_steps():
    # the gradient scale changes by 2^8 between steps: the previous step's
    # first digit predicts nothing, and pass 0 falls back to one digit
    layers = [(64, 200), (9, 0)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=2, workers=2, seed=5)
    scale = [1.0, 256.0, 1.0 / 256.0, 256.0, 1.0]

    def grads_of(t):
        g = workloads.gradients(cfg, t)
        return [[(x * np.float32(scale[t])).astype(np.float32) for x in gw] for gw in g]

    _run(cfg, 10, 2, len(scale), grads_of=grads_of)


def test_rtopk_many_workers():
    # more workers than the apply kernel keeps in registers (its general path)
    layers = [(40, 96), (6, 0), (17, 33)]
    cfg = workloads.scaled(workloads.c2_resnet18(), layers, rank=2, workers=9, seed=17)
    _run(cfg, 8, 2, 3)
