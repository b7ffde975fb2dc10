"""Shared test helpers: run the CUDA path and the oracle side by side."""
from __future__ import annotations

import numpy as np

import workloads
from oracle import powersgd as O


def rel_fro(got, want, floor: float = 0.0) -> float:
    """||got - want||_F / max(||want||_F, floor)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = max(float(np.linalg.norm(want)), floor)
    num = np.linalg.norm(got - want)
    if den == 0.0:
        return float(num)
    return float(num / den)


class GpuRun:
    """A PowerSGD context fed from the seeded numpy generators."""

    def __init__(self, cfg: workloads.Workload, **kw):
        import torch
        from rank_gradient_compression_layer_gb300 import PowerSGD

        self.torch = torch
        self.cfg = cfg
        self.ctx = PowerSGD(cfg.layers, cfg.rank, cfg.workers, seed=cfg.seed, **kw)
        self.bufs = [self.ctx.empty_buffer() for _ in range(cfg.workers)]
        self.upd = self.ctx.empty_buffer()

    def load(self, grads):
        t = self.torch
        for w in range(self.cfg.workers):
            self.ctx.pack([t.from_numpy(g).cuda() for g in grads[w]], out=self.bufs[w])

    def step(self, grads, update=True):
        self.load(grads)
        self.ctx.step(self.bufs, self.upd if update else None)
        self.ctx.sync()

    def update(self, layer):
        return self.ctx.layer_view(self.upd, layer).double().cpu().numpy()

    def PQ(self, layer):
        P, Q = self.ctx.get_PQ(layer)
        return P.double().cpu().numpy(), Q.double().cpu().numpy()

    def E(self, layer, w):
        return self.ctx.get_error(layer, w).double().cpu().numpy()

    def Qw(self, layer, w):
        return self.ctx.get_Qw(layer, w).double().cpu().numpy()

    def close(self):
        self.ctx.close()


def compare_step(run: GpuRun, ref: O.StepOut, st: O.OracleState, tol: float, layers=None, check_e=True,
                 grads=None):
    """Max relative Frobenius error over Phat, Qbar, U, every Q_w and E_w.

    E_w is measured against its own norm, except on a layer whose rank r
    reaches min(n, m): there M_w lies in span(Phat), the exact new error is
    zero and only float32 rounding is left, so its own norm is no scale;
    such a layer's E_w is measured against max(||E_w||, 1e-2 ||G_w||).
    """
    cfg = run.cfg
    worst = {}
    todo = range(len(cfg.layers)) if layers is None else layers
    for li in todo:
        n, m = cfg.layers[li]
        if m == 0:
            worst[(li, "U")] = rel_fro(run.update(li), ref.U[li])
            continue
        P, Q = run.PQ(li)
        worst[(li, "P")] = rel_fro(P, ref.Phat[li])
        worst[(li, "Q")] = rel_fro(Q, ref.Qbar[li])
        worst[(li, "U")] = rel_fro(run.update(li), ref.U[li])
        if check_e:
            for w in range(cfg.workers):
                worst[(li, f"Qw{w}")] = rel_fro(run.Qw(li, w), ref.Q_w[li][w])
                exact_zero = cfg.rank >= min(n, m)
                floor = 1e-2 * float(np.linalg.norm(grads[w][li])) if (grads is not None and exact_zero) else 0.0
                worst[(li, f"E{w}")] = rel_fro(run.E(li, w), st.E[li][w], floor)
    bad = {k: v for k, v in worst.items() if not v <= tol}
    return max(worst.values()), bad
