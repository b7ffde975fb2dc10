"""Seeded synthetic gradient workloads for the PowerSGD compression step.

This module only describes layer shapes and draws random inputs. It holds none
of the compression arithmetic, so both the CPU oracle (``oracle/``) and the
GPU path (``rank_gradient_compression_layer_gb300``) can take their inputs from
it without sharing any of the method's code.

The shapes stand in for the workloads of the PowerSGD review page
("PowerSGD: Practical Low-Rank Gradient Compression for Distributed
Optimization", sections 提案手法 and 主な発見): ResNet-18 on CIFAR-10 and a
3-layer LSTM on Wikitext-2. No dataset is used; only the layer shapes are
reproduced, and every gradient is ``S + noise`` with a low-rank signal ``S``
(shared by all workers and steps) and fresh noise per (worker, step, layer).

Layer convention: ``(n, m)`` with ``m > 0`` is a gradient matrix of n rows and
m columns (a conv weight reshaped to out_ch x in_ch*k*k); ``m == 0`` is a 1-D
tensor of length n (a bias or batch-norm vector) that is averaged, not
compressed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, List, Sequence, Tuple

import numpy as np

Shape = Tuple[int, int]


# --------------------------------------------------------------------------
# Layer shape tables
# --------------------------------------------------------------------------

def resnet18_cifar_layers() -> List[Shape]:
    """ResNet-18 (CIFAR variant, 10 classes) parameter shapes.

    Conv weights are reshaped to out_ch x (in_ch*k*k).  Every conv is followed
    by a batch norm with a weight and a bias vector of out_ch entries; the fc
    layer has a 10x512 weight and a bias of 10.  21 matrices with
    11,164,352 elements and 41 vectors with 9,610 elements.
    """
    mats: List[Shape] = [(64, 27)]                       # conv1 3x3, 3->64
    bn: List[int] = [64]
    mats += [(64, 576)] * 4                               # layer1
    bn += [64] * 4
    mats += [(128, 576)] + [(128, 1152)] * 3 + [(128, 64)]   # layer2 (+1x1 downsample)
    bn += [128] * 5
    mats += [(256, 1152)] + [(256, 2304)] * 3 + [(256, 128)]  # layer3
    bn += [256] * 5
    mats += [(512, 2304)] + [(512, 4608)] * 3 + [(512, 256)]  # layer4
    bn += [512] * 5
    mats += [(10, 512)]                                   # fc
    vecs: List[Shape] = []
    for c in bn:
        vecs += [(c, 0), (c, 0)]                          # BN weight, BN bias
    vecs += [(10, 0)]                                     # fc bias
    return mats + vecs


def lstm_wikitext2_layers(vocab: int = 33278, hidden: int = 650, num_layers: int = 3) -> List[Shape]:
    """3-layer LSTM language model, hidden 650, tied embedding/softmax.

    One vocab x hidden matrix (embedding tied with the decoder), and per layer
    an input and a recurrent weight of 4*hidden x hidden.  Vectors: two gate
    biases of 4*hidden per layer and the decoder bias of vocab entries.
    """
    mats: List[Shape] = [(vocab, hidden)]
    vecs: List[Shape] = []
    for _ in range(num_layers):
        mats += [(4 * hidden, hidden), (4 * hidden, hidden)]
        vecs += [(4 * hidden, 0), (4 * hidden, 0)]
    vecs += [(vocab, 0)]
    return mats + vecs


def transformer_1p2b_layers(blocks: int = 24, d: int = 2048, ff: int = 8192) -> List[Shape]:
    """24 blocks of 4 attention matrices d x d and 2 MLP matrices d x ff."""
    mats: List[Shape] = []
    for _ in range(blocks):
        mats += [(d, d)] * 4 + [(d, ff)] * 2
    return mats


# --------------------------------------------------------------------------
# Workload configurations
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, rank, workers, signal and noise recipe."""

    name: str
    layers: Tuple[Shape, ...]
    rank: int
    workers: int
    steps: int
    seed: int
    # singular values of the shared low-rank signal, given the layer shape
    sigma: Callable[[int, int], np.ndarray]
    # "gaussian_rel": N(0, s^2), s = noise_rel * ||S||_F / sqrt(n m)
    # "gaussian_abs": N(0, noise_abs^2)
    # "student_t3":   noise_abs * t_3
    noise: str
    noise_rel: float = 0.0
    noise_abs: float = 0.0

    @property
    def matrices(self) -> List[Shape]:
        return [s for s in self.layers if s[1] > 0]

    @property
    def vectors(self) -> List[Shape]:
        return [s for s in self.layers if s[1] == 0]

    def matrix_elements(self) -> int:
        return sum(n * m for n, m in self.matrices)

    def vector_elements(self) -> int:
        return sum(n for n, _ in self.vectors)


def _decay(base: float, k: int) -> Callable[[int, int], np.ndarray]:
    return lambda n, m: base ** np.arange(min(k, n, m), dtype=np.float64)


def _lstm_sigma(n: int, m: int) -> np.ndarray:
    c = 1e-3 * math.sqrt(3.0 * n * m) / 4.0
    return c * np.array([4.0, 2.0, 1.0, 0.5])


def c1_single_matrix() -> Workload:
    return Workload("single_256x128_r1_w2", ((256, 128),), rank=1, workers=2, steps=10, seed=0,
                    sigma=lambda n, m: np.array([10.0, 5.0, 2.0, 1.0]),
                    noise="gaussian_abs", noise_abs=0.1)


def c2_resnet18() -> Workload:
    return Workload("resnet18_r2_w4", tuple(resnet18_cifar_layers()), rank=2, workers=4, steps=10,
                    seed=1, sigma=_decay(0.7, 8), noise="gaussian_rel", noise_rel=0.1)


def c3_lstm() -> Workload:
    return Workload("lstm650_r4_w4", tuple(lstm_wikitext2_layers()), rank=4, workers=4, steps=20,
                    seed=2, sigma=_lstm_sigma, noise="student_t3", noise_abs=1e-3)


def c4_transformer() -> Workload:
    return Workload("transformer1p2b_r4_w4", tuple(transformer_1p2b_layers()), rank=4, workers=4,
                    steps=3, seed=3, sigma=_decay(0.8, 16), noise="gaussian_rel", noise_rel=0.1)


def c5_rank_sweep(rank: int) -> Workload:
    return Workload(f"square8192_r{rank}_w8", ((8192, 8192),), rank=rank, workers=8, steps=10,
                    seed=4, sigma=_decay(0.85, 32), noise="gaussian_rel", noise_rel=0.1)


def scaled(w: Workload, layers: Sequence[Shape], name: str | None = None, **kw) -> Workload:
    """A copy of ``w`` with other layer shapes (used to shrink a config for tests)."""
    return dataclasses.replace(w, layers=tuple(layers), name=name or w.name + "_small", **kw)


# --------------------------------------------------------------------------
# Seeded generators (numpy, host)
# --------------------------------------------------------------------------

def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


def signal(w: Workload, layer: int) -> np.ndarray:
    """Shared low-rank signal S = U diag(sigma) V^T of one matrix layer (float64).

    U and V are the orthonormal Q factors of seeded Gaussian matrices, so the
    singular values of S are exactly ``w.sigma``.
    """
    n, m = w.layers[layer]
    assert m > 0
    sig = np.asarray(w.sigma(n, m), dtype=np.float64)
    k = min(len(sig), n, m)
    g = _rng(w.seed, 1, layer)
    U, _ = np.linalg.qr(g.standard_normal((n, k)))
    V, _ = np.linalg.qr(g.standard_normal((m, k)))
    return (U * sig[:k]) @ V.T


def _noise(w: Workload, layer: int, step: int, worker: int, shape, s_fro: float) -> np.ndarray:
    g = _rng(w.seed, 2, layer, step, worker)
    size = int(np.prod(shape))
    if w.noise == "gaussian_abs":
        return w.noise_abs * g.standard_normal(shape)
    if w.noise == "gaussian_rel":
        s = w.noise_rel * s_fro / math.sqrt(size) if size else 0.0
        return s * g.standard_normal(shape)
    if w.noise == "student_t3":
        return w.noise_abs * g.standard_t(3, shape)
    raise ValueError(w.noise)


def vector_gradient(w: Workload, layer: int, step: int, worker: int) -> np.ndarray:
    """A 1-D gradient: a shared seeded mean plus per-worker noise (float32)."""
    n, m = w.layers[layer]
    assert m == 0
    base = _rng(w.seed, 3, layer).standard_normal(n)
    return (base + 0.1 * _rng(w.seed, 4, layer, step, worker).standard_normal(n)).astype(np.float32)


def gradients(w: Workload, step: int, signals: dict | None = None) -> List[List[np.ndarray]]:
    """All gradients of one step: ``out[worker][layer]``, float32, layer shape (n, m) or (n,).

    ``signals`` may cache the per-layer signals across steps (it is filled in).
    """
    if signals is None:
        signals = {}
    out: List[List[np.ndarray]] = []
    for wk in range(w.workers):
        per: List[np.ndarray] = []
        for li, (n, m) in enumerate(w.layers):
            if m == 0:
                per.append(vector_gradient(w, li, step, wk))
                continue
            if li not in signals:
                signals[li] = signal(w, li)
            S = signals[li]
            noise = _noise(w, li, step, wk, (n, m), float(np.linalg.norm(S)))
            per.append((S + noise).astype(np.float32))
        out.append(per)
    return out


# --------------------------------------------------------------------------
# Seeded generators (torch, on a device) for the multi-GB configs
# --------------------------------------------------------------------------

def device_gradient_matrix(w: Workload, layer: int, step: int, worker: int, device, out=None):
    """One matrix gradient generated on ``device`` (float32).

    Same recipe as :func:`gradients` (low-rank signal with orthonormal factors
    plus Gaussian noise): the thin factors come from a seeded numpy QR (small,
    n x k and m x k), the n x m noise is drawn on the device with torch's
    seeded generator, so the multi-GB configurations need no large host round
    trip.  Returns a (n, m) tensor, or writes into ``out`` (a (n, m) view).
    """
    import torch

    n, m = w.layers[layer]
    sig = np.asarray(w.sigma(n, m), dtype=np.float64)
    k = min(len(sig), n, m)
    g = _rng(w.seed, 5, layer)
    U, _ = np.linalg.qr(g.standard_normal((n, k)))
    V, _ = np.linalg.qr(g.standard_normal((m, k)))
    Ud = torch.as_tensor((U * sig[:k]).astype(np.float32), device=device)
    Vd = torch.as_tensor(V.astype(np.float32), device=device)
    s_fro = float(np.linalg.norm(sig[:k]))
    gen = torch.Generator(device=device)
    gen.manual_seed(((w.seed * 1_000_003 + layer) * 7919 + step * 131 + worker + 1) & 0x7FFFFFFFFFFF)
    std = w.noise_rel * s_fro / math.sqrt(n * m) if w.noise == "gaussian_rel" else w.noise_abs
    if out is None:
        out = torch.empty(n, m, device=device, dtype=torch.float32)
    out.normal_(0.0, std, generator=gen)
    out.add_(Ud @ Vd.T)
    return out


ALL = {
    "c1": c1_single_matrix,
    "c2": c2_resnet18,
    "c3": c3_lstm,
    "c4": c4_transformer,
}
