"""CPU oracle of the PowerSGD compression step (float64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
path; the only common module is ``workloads.py``, which draws inputs and holds
none of the method's arithmetic.

Source of every step: the PowerSGD review page ("PowerSGD: Practical Low-Rank
Gradient Compression for Distributed Optimization", Vogels, Karimireddy,
Jaggi 2019), section 提案手法 (proposed method):
  * each layer's gradient is a matrix M (n x m), compressed on its own, to
    P Q^T with P in R^{n x r}, Q in R^{m x r}, r small (bullet 4);
  * one step of subspace / power iteration, warm-started from the previous
    step's Q (bullet 1);
  * the compressor is linear, so the W workers' messages are aggregated with
    an all-reduce (bullet 2) -- here a sum over the worker axis;
  * the error left after compression is fed back into the next step (bullet 3);
  * the update is decompressed as P Q^T (bullet 5).
Section 主な発見 (main findings), bullet 5: warm-started power iteration
approaches the best rank-r approximation without an SVD.

Where the page leaves a step open, the plainest reading is taken (each one
is listed where it is used):
  * orthonormalisation = Gram-Schmidt (modified, column by column, each
    column orthogonalised twice), the thin-QR factor with a positive diagonal
    of R; a column whose remainder is exactly zero stays zero;
  * P is the SUM of the workers' M_w Q; Q is the MEAN of the workers' M_w^T P,
    so the decompressed P Q^T approximates the mean gradient;
  * the error is worker-local: E_w <- M_w - Phat Q_w^T with the worker's own
    Q_w (the sum over workers equals W times the mean-gradient residual);
  * the next step is warm-started with the mean Q, not re-normalised;
  * Q starts as N(0,1) draws (see ``q_init``); E starts at zero;
  * 1-D tensors are averaged over workers and not compressed.

All arithmetic is float64.  Parity of every function here is pinned by
``tests/test_oracle_pins.py`` against closed forms, library routines (QR, SVD)
and the results table on the page; nothing here is "parity unpinned".
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence, Tuple

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15


# --------------------------------------------------------------------------
# Q initialisation: splitmix64 (Steele, Lea & Flood, "Fast splittable
# pseudorandom number generators", OOPSLA 2014) + Box-Muller (1958).
# --------------------------------------------------------------------------

def splitmix64_mix(z: int) -> int:
    """The splitmix64 output function applied to a 64-bit state value."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, count: int) -> List[int]:
    """The first ``count`` outputs of splitmix64 seeded with ``seed``.

    Output k (k = 1, 2, ...) is mix(seed + k * golden_gamma) mod 2^64.
    """
    out = []
    s = seed & MASK64
    for _ in range(count):
        s = (s + GOLDEN_GAMMA) & MASK64
        out.append(splitmix64_mix(s))
    return out


def uniform_open0(x: int) -> float:
    """Top 53 bits of a 64-bit word -> a double in (0, 1]."""
    return ((x >> 11) + 1) * (1.0 / 9007199254740992.0)


def q_init(seed: int, layer: int, m: int, r: int) -> np.ndarray:
    """Initial Q of one matrix layer: m x r N(0,1) draws, rounded to float32.

    Layer stream key: k_l = mix(seed + (layer+1) * gamma).  Element pair t of
    the row-major m x r array uses outputs 2t+1 and 2t+2 of splitmix64 seeded
    with k_l as u1, u2 in (0, 1]; Box-Muller gives
    z0 = sqrt(-2 ln u1) cos(2 pi u2) for element 2t and
    z1 = sqrt(-2 ln u1) sin(2 pi u2) for element 2t+1 (dropped past the end).
    The 64-bit arithmetic is done on numpy uint64 arrays, which wrap mod 2^64.
    """
    key = splitmix64_mix((seed + (layer + 1) * GOLDEN_GAMMA) & MASK64)
    total = m * r
    pairs = (total + 1) // 2
    k = np.arange(1, 2 * pairs + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + k * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    u = ((z >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = rad * np.cos(2.0 * np.pi * u2)
    out[1::2] = rad * np.sin(2.0 * np.pi * u2)
    return out[:total].reshape(m, r).astype(np.float32)


# --------------------------------------------------------------------------
# One compression (section 提案手法, bullets 1, 2, 4, 5)
# --------------------------------------------------------------------------

def gram_schmidt(P: np.ndarray) -> np.ndarray:
    """Gram-Schmidt on the columns of P (float64), each column orthogonalised twice.

    Column k has the projections on the already finished columns 0..k-1
    removed one at a time (modified Gram-Schmidt), and then once more, and
    is scaled to unit length.  The result is the thin-QR factor of P whose R
    has a positive diagonal.  A column whose remainder has norm exactly 0 is
    left as the zero vector.

    The second pass changes nothing in exact arithmetic.  In floating point a
    single pass leaves column k off orthogonal by about eps times the ratio
    of its norm to its remainder's, which reaches 1e-2 when the warm-started
    Q's last column carries almost nothing outside the other columns' span
    (a rank-deficient P); the error feedback then compounds it step after
    step.  One more pass brings the columns back to orthogonal to working
    precision ("twice is enough": Giraud, Langou and Rozloznik, 2005).
    """
    Ph = np.array(P, dtype=np.float64, copy=True)
    n, r = Ph.shape
    for k in range(r):
        v = Ph[:, k]
        for _ in range(2):
            for j in range(k):
                v -= (Ph[:, j] @ v) * Ph[:, j]
        nrm = math.sqrt(float(v @ v))
        if nrm > 0.0:
            v /= nrm
        else:
            v[:] = 0.0
        Ph[:, k] = v
    return Ph


@dataclasses.dataclass
class Compressed:
    P: np.ndarray            # n x r, sum over workers of M_w Q
    Phat: np.ndarray         # n x r, orthonormalised P
    Q_w: List[np.ndarray]    # per worker, m x r, M_w^T Phat
    Qbar: np.ndarray         # m x r, mean over workers of Q_w
    U: np.ndarray            # n x m, Phat Qbar^T (decompressed update)
    E_new: List[np.ndarray]  # per worker, n x m, M_w - Phat Q_w^T


def compress(M: Sequence[np.ndarray], Q: np.ndarray) -> Compressed:
    """One warm-started power-iteration compression of W workers' matrices M_w.

    P = sum_w M_w Q (the first all-reduce), Phat = GramSchmidt(P),
    Q_w = M_w^T Phat, Qbar = (1/W) sum_w Q_w (the second all-reduce),
    U = Phat Qbar^T, E_new_w = M_w - Phat Q_w^T.
    """
    W = len(M)
    M = [np.asarray(x, dtype=np.float64) for x in M]
    Q = np.asarray(Q, dtype=np.float64)
    P = np.zeros((M[0].shape[0], Q.shape[1]))
    for Mw in M:
        P += Mw @ Q
    Phat = gram_schmidt(P)
    Q_w = [Mw.T @ Phat for Mw in M]
    Qbar = np.zeros_like(Q_w[0])
    for q in Q_w:
        Qbar += q
    Qbar /= W
    U = Phat @ Qbar.T
    E_new = [Mw - Phat @ q.T for Mw, q in zip(M, Q_w)]
    return Compressed(P, Phat, Q_w, Qbar, U, E_new)


# --------------------------------------------------------------------------
# The optimiser update after the step (section 提案手法, bullet 5: the
# decompressed P Q^T drives a momentum SGD update, "EF-SGD with momentum")
# --------------------------------------------------------------------------

def momentum_update(x: np.ndarray, mom: np.ndarray, U: np.ndarray, lr: float, beta: float):
    """One momentum-SGD update of the parameters ``x`` by the decompressed ``U``.

    The page names the optimiser without its formula.  Reading taken:
    heavy-ball momentum ``mom <- beta * mom + U`` and a Nesterov-style step
    ``x <- x - lr * (U + mom)`` with the new ``mom``.  Element-wise, so it is
    the same for a matrix layer's U and a vector layer's worker mean.
    Returns ``(x_new, mom_new)`` in float64.
    """
    U = np.asarray(U, dtype=np.float64)
    mom_new = beta * np.asarray(mom, dtype=np.float64) + U
    x_new = np.asarray(x, dtype=np.float64) - lr * (U + mom_new)
    return x_new, mom_new


# --------------------------------------------------------------------------
# The step with error feedback and warm start, over a whole layer set
# --------------------------------------------------------------------------

def data_sent_per_step(layers: Sequence[Tuple[int, int]], rank: int) -> Tuple[int, int]:
    """Floats one worker sends per step: (compressed, uncompressed).

    A matrix n x m sends its two factors, (n + m) * r floats, instead of n*m;
    a 1-D tensor of length n is sent whole either way.
    """
    comp = unc = 0
    for n, m in layers:
        if m == 0:
            comp += n
            unc += n
        else:
            comp += (n + m) * rank
            unc += n * m
    return comp, unc


@dataclasses.dataclass
class StepOut:
    Phat: List[np.ndarray | None]   # per layer (None for vectors)
    Qbar: List[np.ndarray | None]
    Q_w: List[List[np.ndarray] | None]
    U: List[np.ndarray]             # per layer: n x m update, or length-n mean for vectors


# --------------------------------------------------------------------------
# Unbiased rank-r compression (section 主な発見, bullet 4: the page sets
# PowerSGD's biased, error-fed compressor against an unbiased rank-r one and
# reports the unbiased one far less accurate; the page does not define it)
# --------------------------------------------------------------------------
#
# Reading taken: the textbook unbiased low-rank estimate by random
# projection.  Every step draws a fresh Q of N(0,1) entries from a seed all
# workers share, so only P travels: P = sum_w G_w Q (the one all-reduce) and
# U = P Q^T / (W r).  E[Q Q^T] = r I, so E[U] = mean_w G_w.  No error
# feedback, no warm start, no orthonormalisation.

def step_seed(seed: int, step: int) -> int:
    """Seed of step t's fresh Q: the splitmix64 mix of seed + (t + 1) gamma.

    Step t's Q of layer l is ``q_init(step_seed(seed, t), l, m, r)``.
    """
    return splitmix64_mix((seed + (step + 1) * GOLDEN_GAMMA) & MASK64)


def unbiased_compress(G: Sequence[np.ndarray], Q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """(P, U) of the unbiased rank-r estimate: P = sum_w G_w Q, U = P Q^T / (W r)."""
    W = len(G)
    Q = np.asarray(Q, dtype=np.float64)
    P = np.zeros((np.asarray(G[0]).shape[0], Q.shape[1]))
    for Gw in G:
        P += np.asarray(Gw, dtype=np.float64) @ Q
    U = (P @ Q.T) / (W * Q.shape[1])
    return P, U


def unbiased_step(grads: Sequence[Sequence[np.ndarray]], layers: Sequence[Tuple[int, int]], rank: int,
                  seed: int, step: int) -> StepOut:
    """Step t of the unbiased variant over a layer set (vectors averaged).

    StepOut.Phat holds P (not orthonormalised), StepOut.Qbar the step's Q.
    """
    W = len(grads)
    L = len(layers)
    out = StepOut([None] * L, [None] * L, [None] * L, [None] * L)
    s = step_seed(seed, step)
    for li, (n, m) in enumerate(layers):
        if m == 0:
            acc = np.zeros(n)
            for w in range(W):
                acc += np.asarray(grads[w][li], dtype=np.float64)
            out.U[li] = acc / W
            continue
        Q = q_init(s, li, m, rank).astype(np.float64)
        P, U = unbiased_compress([grads[w][li] for w in range(W)], Q)
        out.Phat[li], out.Qbar[li], out.U[li] = P, Q, U
    return out


def unbiased_data_sent(layers: Sequence[Tuple[int, int]], rank: int) -> int:
    """Floats one worker sends per step in the unbiased variant: n r per matrix (P only), vectors whole."""
    return sum(n * rank if m else n for n, m in layers)


# --------------------------------------------------------------------------
# rTop-k sparsification (the rTop-k review page, "rTop-k: A Statistical
# Estimation Approach to Distributed SGD", section 제안 방법 / proposed method,
# bullet 3: a random subset of the top-k magnitude gradient entries)
# --------------------------------------------------------------------------
#
# Readings taken where the page is silent:
#   * the top set has r = ceil(d / top_div) entries of a layer's d, the sent
#     subset k = ceil(r / sample_div) of them, chosen uniformly at random;
#   * it runs on M_w = G_w + E_w with error feedback, E_w <- M_w - S_w (the
#     page calls it a compression operator with the convergence guarantees
#     of error-fed compressors);
#   * "largest magnitude" orders by |M| (float32) and then by the smaller
#     index; the random subset takes the k smallest of (upper 32 bits of a
#     splitmix64 draw keyed by (seed, step, worker, layer, index), index);
#   * U = (sum_w S_w) / W, summed in worker order in float32; 1-D tensors
#     are averaged, as in PowerSGD.
# M, E, S and U are float32 here, as on the GPU, so the selections (integer
# decisions) and the results agree exactly.

def rtopk_counts(d: int, top_div: int, sample_div: int) -> Tuple[int, int]:
    """(r, k) for a layer of d entries."""
    r = -(-d // top_div)
    return r, -(-r // sample_div)


def rtopk_draw_key(seed: int, step: int, worker: int, layer: int) -> int:
    """Stream key of one (step, worker, layer): splitmix64 mixes of the step seed."""
    return splitmix64_mix((step_seed(seed, step) + (worker * 65536 + layer + 1) * GOLDEN_GAMMA) & MASK64)


def rtopk_select(M: np.ndarray, r: int, k: int, key: int) -> np.ndarray:
    """Flat indices of the k entries sent out of the r largest |M| (float32 M)."""
    a = np.abs(np.asarray(M, dtype=np.float32).ravel())
    d = a.size
    idx = np.arange(d, dtype=np.int64)
    order = np.lexsort((idx, -a.astype(np.float64)))  # |M| descending, then index ascending
    top = order[:r]
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (top.astype(np.uint64) + np.uint64(1)) * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    hi = (z >> np.uint64(32)).astype(np.int64)
    pick = np.lexsort((top, hi))[:k]  # the k smallest (draw, index)
    return np.sort(top[pick])


class RTopKState:
    """Error buffers of W workers under rTop-k, over a layer set."""

    def __init__(self, layers: Sequence[Tuple[int, int]], workers: int, seed: int, top_div: int, sample_div: int):
        self.layers = [tuple(l) for l in layers]
        self.W, self.seed, self.top_div, self.sample_div = workers, seed, top_div, sample_div
        self.E = [None if m == 0 else [np.zeros((n, m), dtype=np.float32) for _ in range(workers)]
                  for n, m in self.layers]
        self.steps = 0

    def step(self, grads: Sequence[Sequence[np.ndarray]]):
        """One step: returns (U per layer, sent index lists [layer][worker])."""
        W = self.W
        U, sent = [], []
        for li, (n, m) in enumerate(self.layers):
            if m == 0:
                acc = np.zeros(n, dtype=np.float64)
                for w in range(W):
                    acc += np.asarray(grads[w][li], dtype=np.float64)
                U.append(acc / W)
                sent.append(None)
                continue
            r, k = rtopk_counts(n * m, self.top_div, self.sample_div)
            u = np.zeros(n * m, dtype=np.float32)
            per = []
            for w in range(W):
                M = (np.asarray(grads[w][li], dtype=np.float32) + self.E[li][w]).astype(np.float32)
                sel = rtopk_select(M, r, k, rtopk_draw_key(self.seed, self.steps, w, li))
                flat = M.ravel()
                u[sel] = (u[sel] + flat[sel]).astype(np.float32)
                E = flat.copy()
                E[sel] = 0.0
                self.E[li][w] = E.reshape(n, m)
                per.append(sel)
            U.append((u * np.float32(1.0 / W)).astype(np.float32).reshape(n, m))
            sent.append(per)
        self.steps += 1
        return U, sent


def rtopk_data_sent(layers: Sequence[Tuple[int, int]], top_div: int, sample_div: int) -> int:
    """Words one worker sends per step: k values + k indices per matrix, vectors whole."""
    tot = 0
    for n, m in layers:
        if m == 0:
            tot += n
        else:
            tot += 2 * rtopk_counts(n * m, top_div, sample_div)[1]
    return tot


class OracleState:
    """Per-layer error buffers E_w and warm-start Q of a W-worker PowerSGD run."""

    def __init__(self, layers: Sequence[Tuple[int, int]], rank: int, workers: int, seed: int,
                 Q0: Sequence[np.ndarray | None] | None = None):
        self.layers = [tuple(s) for s in layers]
        self.rank = rank
        self.workers = workers
        self.seed = seed
        self.E: List[List[np.ndarray] | None] = []
        self.Q: List[np.ndarray | None] = []
        for li, (n, m) in enumerate(self.layers):
            if m == 0:
                self.E.append(None)
                self.Q.append(None)
                continue
            self.E.append([np.zeros((n, m)) for _ in range(workers)])
            if Q0 is not None and Q0[li] is not None:
                self.Q.append(np.asarray(Q0[li], dtype=np.float64))
            else:
                self.Q.append(q_init(seed, li, m, rank).astype(np.float64))
        self.steps = 0
        self.floats_sent = 0
        self.floats_uncompressed = 0

    def step(self, grads: Sequence[Sequence[np.ndarray]], layers: Sequence[int] | None = None) -> StepOut:
        """One PowerSGD step.  ``grads[w][l]`` is worker w's gradient of layer l.

        ``layers`` restricts the work to a subset of layers (others untouched);
        the data-sent counters always count the whole layer set.
        """
        W = self.workers
        assert len(grads) == W
        todo = range(len(self.layers)) if layers is None else layers
        out = StepOut([None] * len(self.layers), [None] * len(self.layers),
                      [None] * len(self.layers), [None] * len(self.layers))
        for li in todo:
            n, m = self.layers[li]
            if m == 0:
                acc = np.zeros(n)
                for w in range(W):
                    acc += np.asarray(grads[w][li], dtype=np.float64)
                out.U[li] = acc / W
                continue
            M = [np.asarray(grads[w][li], dtype=np.float64).reshape(n, m) + self.E[li][w]
                 for w in range(W)]
            c = compress(M, self.Q[li])
            self.E[li] = c.E_new
            self.Q[li] = c.Qbar
            out.Phat[li], out.Qbar[li], out.Q_w[li], out.U[li] = c.Phat, c.Qbar, c.Q_w, c.U
        comp, unc = data_sent_per_step(self.layers, self.rank)
        self.steps += 1
        self.floats_sent += comp
        self.floats_uncompressed += unc
        return out
