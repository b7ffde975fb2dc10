"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances (relative Frobenius error on Phat, Qbar, U, every Q_w and every
E_w): 1e-4 after the first step, 1e-3 after later steps.
"""
import os

import numpy as np
import pytest

import workloads
from oracle import powersgd as O
from tests.harness import GpuRun, compare_step, rel_fro

pytestmark = pytest.mark.gpu

TOL1, TOLN = 1e-4, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_gradient_compression_layer_gb300 import build
    build()


def _run_config(cfg, steps, check_every=1, check_e=True, **kw):
    run = GpuRun(cfg, **kw)
    st = O.OracleState(cfg.layers, cfg.rank, cfg.workers, cfg.seed)
    sig = {}
    worst_all = []
    try:
        for t in range(steps):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads)
            ref = st.step(grads)
            if t == 0 or (t + 1) % check_every == 0 or t == steps - 1:
                tol = TOL1 if t == 0 else TOLN
                worst, bad = compare_step(run, ref, st, tol, check_e=check_e, grads=grads)
                worst_all.append(worst)
                assert not bad, f"step {t}: {sorted(bad.items(), key=lambda kv: -kv[1])[:5]}"
        s = run.ctx.stats()
        comp, unc = O.data_sent_per_step(cfg.layers, cfg.rank)
        assert s["floats_sent_per_step"] == comp and s["floats_uncompressed_per_step"] == unc
        assert s["floats_sent"] == steps * comp and s["steps"] == steps
    finally:
        run.close()
    return worst_all


def test_q_init_matches_oracle():
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(40, 17), (9, 0), (300, 130)], rank=3, workers=2)
    run = GpuRun(cfg)
    try:
        for li, (n, m) in enumerate(cfg.layers):
            if m == 0:
                continue
            _, Q = run.PQ(li)
            want = O.q_init(cfg.seed, li, m, cfg.rank).astype(np.float64)
            np.testing.assert_allclose(Q, want, rtol=2.5e-7, atol=1e-30)
    finally:
        run.close()


def test_c1_single_matrix_ten_steps():
    _run_config(workloads.c1_single_matrix(), 10)


def test_c2_resnet18_ten_steps():
    _run_config(workloads.c2_resnet18(), 10)


def test_c3_lstm_twenty_steps():
    _run_config(workloads.c3_lstm(), 20, check_every=5)


@pytest.mark.parametrize("rank", [1, 2, 3, 4, 8, 16, 32])
def test_c5_rank_sweep_reduced(rank):
    # the 8192 x 8192, W = 8 rank sweep at a size the oracle finishes in
    # seconds: 1536 rows (several P3 row tiles), 1000 columns (a ragged segment)
    cfg = workloads.scaled(workloads.c5_rank_sweep(rank), [(1536, 1000)])
    _run_config(cfg, 10, check_every=3)


def test_ragged_shapes_and_padding():
    layers = [(1, 1), (3, 5), (33, 27), (7, 0), (130, 1), (64, 129), (257, 650), (5, 0), (2049, 13)]
    cfg = workloads.Workload("ragged", tuple(layers), rank=1, workers=3, steps=4, seed=11,
                             sigma=lambda n, m: np.array([3.0, 1.0]), noise="gaussian_abs", noise_abs=0.2)
    _run_config(cfg, 4)
    layers = [(3, 5), (33, 27), (64, 129), (257, 650), (2049, 13), (6, 0)]
    cfg3 = workloads.Workload("ragged_r3", tuple(layers), rank=3, workers=3, steps=4, seed=12,
                              sigma=lambda n, m: np.array([3.0, 2.0, 1.0, 0.5]), noise="gaussian_abs",
                              noise_abs=0.2)
    _run_config(cfg3, 4)


def test_garbage_in_padding_is_ignored():
    import torch
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(50, 27), (20, 6)], rank=2, workers=2)
    a, b = GpuRun(cfg), GpuRun(cfg)
    try:
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            a.step(grads)
            b.load(grads)
            for buf in b.bufs:  # poison the ld - m padding columns
                for li, (n, m) in enumerate(cfg.layers):
                    off, ld = b.ctx.offsets[li], b.ctx.lds[li]
                    buf[off:off + n * ld].view(n, ld)[:, m:] = float("nan")
            b.ctx.step(b.bufs, b.upd)
            b.ctx.sync()
            for li in range(len(cfg.layers)):
                assert torch.equal(a.ctx.layer_view(a.upd, li), b.ctx.layer_view(b.upd, li))
                assert np.array_equal(a.E(li, 0), b.E(li, 0))
    finally:
        a.close()
        b.close()


def test_zero_gradient():
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(40, 24), (8, 0)], rank=2, workers=2)
    run = GpuRun(cfg)
    try:
        grads = [[np.zeros((40, 24), np.float32), np.zeros(8, np.float32)] for _ in range(2)]
        for _ in range(2):
            run.step(grads)
            P, Q = run.PQ(0)
            assert np.all(P == 0) and np.all(Q == 0)
            assert np.all(run.update(0) == 0) and np.all(run.update(1) == 0)
            assert np.all(run.E(0, 0) == 0) and np.all(run.E(0, 1) == 0)
    finally:
        run.close()


def test_exact_rank_r_recovery():
    rng = np.random.default_rng(5)
    n, m, r, W = 300, 200, 3, 2
    A = (rng.standard_normal((n, r)) @ rng.standard_normal((r, m))).astype(np.float32)
    cfg = workloads.scaled(workloads.c1_single_matrix(), [(n, m)], rank=r, workers=W)
    run = GpuRun(cfg)
    try:
        for t in range(10):
            run.step([[A] for _ in range(W)])
            assert rel_fro(run.update(0), A) < 1e-5
            for w in range(W):
                assert np.abs(run.E(0, w)).max() < 1e-5 * np.abs(A).max()
            P, _ = run.PQ(0)
            np.testing.assert_allclose(P.T @ P, np.eye(r), atol=1e-6)
    finally:
        run.close()


def _outputs(run):
    out = []
    for li, (n, m) in enumerate(run.cfg.layers):
        out.append(run.update(li))
        if m:
            out += list(run.PQ(li))
            out += [run.E(li, w) for w in range(run.cfg.workers)]
    return out


def test_first_context_of_a_process_plans_like_the_rest():
    # the tile planner reads the kernels' occupancy, which depends on their
    # shared-memory limits: a fresh process's first context must see them set
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from rank_gradient_compression_layer_gb300 import PowerSGD\n"
        "layers = [(256, 1152), (512, 4608), (64, 0)]\n"
        "rows = [PowerSGD(layers, r, 4).stats()['tile_rows'] for r in (16, 16, 32, 32)]\n"
        "assert rows[0] == rows[1] and rows[2] == rows[3], rows\n"
        "print('ok')\n" % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and "ok" in out.stdout, out.stderr[-2000:]


@pytest.mark.parametrize("rank", [2, 16])
def test_bit_reproducible_across_contexts_and_timing(rank):
    # r = 16: the back-project needs more than 48 KB of dynamic shared memory,
    # and every context (the first of the process too) must plan the same tiles
    cfg = workloads.scaled(workloads.c2_resnet18(), workloads.resnet18_cifar_layers()[:12] + [(64, 0)], rank=rank)
    runs = [GpuRun(cfg), GpuRun(cfg), GpuRun(cfg, timing=True)]
    try:
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            outs = []
            for r in runs:
                r.step(grads)
                outs.append(_outputs(r))
            for o in outs[1:]:
                for x, y in zip(outs[0], o):
                    assert np.array_equal(x, y)
    finally:
        for r in runs:
            r.close()


def test_checkpoint_resume_is_bit_exact():
    import torch
    cfg = workloads.scaled(workloads.c2_resnet18(), [(64, 27), (128, 576), (10, 512), (64, 0)], rank=2)
    sig = {}
    grads = [workloads.gradients(cfg, t, sig) for t in range(10)]
    straight = GpuRun(cfg)
    first = GpuRun(cfg)
    try:
        for t in range(10):
            straight.step(grads[t])
        for t in range(5):
            first.step(grads[t])
        # checkpoint: Q (warm start) and E_w of every matrix layer
        ck = {}
        for li, (n, m) in enumerate(cfg.layers):
            if m:
                _, Q = first.ctx.get_PQ(li)
                ck[li] = (Q, [first.ctx.get_error(li, w) for w in range(cfg.workers)])
        first.close()
        resumed = GpuRun(cfg, )
        for li, (Q, Es) in ck.items():
            resumed.ctx.set_state(li, Q, Es)
        for t in range(5, 10):
            resumed.step(grads[t])
        for x, y in zip(_outputs(straight), _outputs(resumed)):
            assert np.array_equal(x, y)
        resumed.close()
    finally:
        straight.close()


def test_step_host_matches_step():
    import torch
    cfg = workloads.scaled(workloads.c2_resnet18(), [(64, 27), (128, 576), (9, 0), (10, 512)], rank=2)
    a, b = GpuRun(cfg), GpuRun(cfg)
    try:
        sig = {}
        for t in range(3):
            grads = workloads.gradients(cfg, t, sig)
            a.step(grads)
            host = [b.ctx.pack([torch.from_numpy(g) for g in grads[w]],
                               out=torch.zeros(b.ctx.total, dtype=torch.float32).pin_memory())
                    for w in range(cfg.workers)]
            msg = torch.zeros(b.ctx.message_floats, dtype=torch.float32).pin_memory()
            upd = torch.zeros(b.ctx.total, dtype=torch.float32).pin_memory()
            b.ctx.step_host(host, msg, upd)
            got = upd.cuda()
            for li in range(len(cfg.layers)):  # the layers (padding after a vector is not written)
                assert torch.equal(b.ctx.layer_view(got, li), a.ctx.layer_view(a.upd, li))
            pos = 0
            for li, (n, m) in enumerate(cfg.layers):
                if m:
                    P, Q = a.ctx.get_PQ(li)
                    assert torch.equal(msg[pos:pos + n * 2].view(n, 2), P.cpu())
                    pos += n * 2
                    assert torch.equal(msg[pos:pos + m * 2].view(m, 2), Q.cpu())
                    pos += m * 2
    finally:
        a.close()
        b.close()


def test_phase_timing():
    # the phase kernels one by one (the fused step has one slot: test_gpu_fused.py)
    cfg = workloads.scaled(workloads.c2_resnet18(), [(128, 576), (9, 0)], rank=2)
    run = GpuRun(cfg, timing=True)
    try:
        sig = {}
        run.step(workloads.gradients(cfg, 0, sig))
        t = run.ctx.phase_times()
        assert set(t) == {"project", "orthonormalise", "back_project", "decompress"}
        assert all(v >= 0.0 for v in t.values()) and t["project"] > 0.0
        s = run.ctx.stats()
        assert s["launches_per_step"] in (3, 4) and s["tiles"]["project"] > 0
        # timing off: steps still run, phase times are refused; on again: averaged anew
        from rank_gradient_compression_layer_gb300 import PsgdError
        run.ctx.set_timing(False)
        run.step(workloads.gradients(cfg, 1, sig))
        with pytest.raises(PsgdError):
            run.ctx.phase_times()
        run.ctx.set_timing(True)
        run.step(workloads.gradients(cfg, 2, sig))
        assert run.ctx.phase_times()["project"] > 0.0
    finally:
        run.close()


def test_invalid_arguments_are_rejected():
    import torch
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PowerSGD, PsgdError
    ctx = PowerSGD([(16, 8)], 2, 2)
    try:
        good = ctx.empty_buffer()
        bad = torch.zeros(ctx.total + 1, device="cuda")[1:]  # 4-byte offset: not 16-byte aligned
        with pytest.raises(PsgdError) as ei:
            ctx.step([good, bad])
        assert ei.value.code == PSGD_ERR_INVALID
        with pytest.raises(PsgdError):
            ctx.get_PQ(5)
        ctx.step([good, good])
        ctx.sync()
    finally:
        ctx.close()
    with pytest.raises(PsgdError):
        PowerSGD([(16, 8)], 9, 2)  # rank > min(n, m)



@pytest.mark.parametrize("rank,workers", [(2, 9), (4, 64), (16, 9)])
def test_many_workers(rank, workers):
    # more workers than warps in a project CTA (warps loop over workers), up
    # to the limit of 64 pointers in the step arguments
    # (the rank-sweep signal: 32 decaying singular values, so even r = 16
    # keeps a spectral gap between ranks r and r + 1)
    layers = [(40, 27), (7, 0), (96, 130), (33, 64)]
    cfg = workloads.scaled(workloads.c5_rank_sweep(rank), layers, rank=rank, workers=workers, seed=31)
    _run_config(cfg, 3)


def test_vector_layers_only():
    # no matrix at all: only the decompress kernel's vector tiles run
    layers = [(5, 0), (1, 0), (8195, 0)]
    cfg = workloads.scaled(workloads.c1_single_matrix(), layers, rank=1, workers=3, seed=2)
    run = GpuRun(cfg)
    try:
        sig = {}
        for t in range(2):
            grads = workloads.gradients(cfg, t, sig)
            run.step(grads)
            for li in range(len(layers)):
                want = sum(np.asarray(grads[w][li], dtype=np.float64) for w in range(3)) / 3
                assert rel_fro(run.update(li), want) < 1e-6
        s = run.ctx.stats()
        assert s["floats_sent_per_step"] == sum(n for n, _ in layers) and s["tiles"]["project"] == 0
    finally:
        run.close()
