"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each check below is chosen so that a plausible slip in the oracle (a dropped
error-feedback term, a sum where a mean belongs, a transposed operand, a
missing projection in Gram-Schmidt, a wrong sign) fails at least one of them;
``test_planted_mistakes_are_caught`` plants such slips in copies of the oracle
on the CPU and checks that the pins notice.

Sources (PowerSGD review page, "PowerSGD: Practical Low-Rank Gradient
Compression for Distributed Optimization"):
  * 提案手法 bullet 1: rank-r, one power/subspace-iteration step, warm start;
  * 提案手法 bullet 2: linear compressor, all-reduce aggregation over W workers;
  * 提案手法 bullet 3: error feedback;
  * 提案手法 bullet 4: P in R^{n x r}, Q in R^{m x r}, per-layer matrices;
  * 主な発見 table: data sent per epoch (SGD 1023 MB, rank 1/2/4: 4/8/14 MB);
  * 主な発見 bullet 5: warm start approaches the best rank-r approximation.
"""
import math
import os

import numpy as np
import pytest
import scipy.stats

import workloads
from oracle import powersgd as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rng(s):
    return np.random.default_rng(s)


def _qr_posdiag(P):
    """numpy's Householder QR with signs flipped so that diag(R) > 0."""
    Q, R = np.linalg.qr(P)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s


# ---------------------------------------------------------------- pins -----

def check_gram_schmidt(gs):
    for n, r, seed in [(7, 1, 0), (40, 3, 1), (300, 4, 2), (64, 8, 3), (1000, 32, 4)]:
        P = _rng(seed).standard_normal((n, r))
        Ph = gs(P)
        # special case reducing to a library routine: thin QR, positive diag R
        np.testing.assert_allclose(Ph, _qr_posdiag(P), atol=1e-12, rtol=0)
        # invariants: orthonormal columns, R = Ph^T P upper triangular, diag > 0
        np.testing.assert_allclose(Ph.T @ Ph, np.eye(r), atol=1e-13)
        R = Ph.T @ P
        assert np.all(np.abs(np.tril(R, -1)) < 1e-10 * np.abs(R).max())
        assert np.all(np.diag(R) > 0)
    # r = 1 closed form: p / ||p||
    p = _rng(9).standard_normal((50, 1))
    np.testing.assert_allclose(gs(p), p / np.linalg.norm(p), rtol=1e-15, atol=0)
    # ill-conditioned (nearly parallel columns): still QR's factor, to kappa*eps
    base = _rng(10).standard_normal((200, 1))
    P = base + 1e-6 * _rng(11).standard_normal((200, 4))
    np.testing.assert_allclose(gs(P), _qr_posdiag(P), atol=1e-7)
    # a last column within 1e-13 of the span of the others (what a warm start
    # gives when M has rank < r): the basis is still orthonormal to working
    # precision, and the leading columns are QR's
    a, b, c = (_rng(s).standard_normal((500, 1)) for s in (13, 14, 15))
    P = np.hstack([a, b, a - 2.0 * b + 1e-13 * c])
    Ph = gs(P)
    np.testing.assert_allclose(Ph.T @ Ph, np.eye(3), atol=1e-12)
    np.testing.assert_allclose(Ph[:, :2], _qr_posdiag(P[:, :2]), atol=1e-13)
    # zero columns stay zero; the all-zero matrix maps to zero
    P = _rng(12).standard_normal((30, 3))
    P[:, 1] = 0.0
    Ph = gs(P)
    assert np.all(Ph[:, 1] == 0.0)
    np.testing.assert_allclose(Ph[:, [0, 2]], _qr_posdiag(P[:, [0, 2]]), atol=1e-13)
    assert np.all(gs(np.zeros((5, 2))) == 0.0)


def check_exact_rank_recovery(compress):
    # If every worker's M is the same exact rank-r matrix and Q is generic,
    # P = W M Q spans col(M), so one compression returns U = M, E = 0.
    rng = _rng(20)
    for n, m, r, W in [(30, 20, 2, 2), (64, 48, 4, 3), (17, 33, 1, 2)]:
        A = rng.standard_normal((n, r)) @ rng.standard_normal((r, m))
        Q = rng.standard_normal((m, r))
        c = compress([A.copy() for _ in range(W)], Q)
        np.testing.assert_allclose(c.U, A, atol=1e-10 * np.abs(A).max())
        for E in c.E_new:
            assert np.abs(E).max() < 1e-10 * np.abs(A).max()
        # and the message sizes: P is n x r, Q is m x r
        assert c.Phat.shape == (n, r) and c.Qbar.shape == (m, r)


def check_linearity(compress):
    # A W-worker compression equals a 1-worker compression of the mean M.
    rng = _rng(30)
    n, m, r, W = 40, 25, 3, 4
    Ms = [rng.standard_normal((n, m)) for _ in range(W)]
    Q = rng.standard_normal((m, r))
    cw = compress(Ms, Q)
    Mbar = sum(Ms) / W
    c1 = compress([Mbar], Q)
    np.testing.assert_allclose(cw.P, W * c1.P, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(cw.Phat, c1.Phat, atol=1e-11)
    np.testing.assert_allclose(cw.Qbar, c1.Qbar, atol=1e-11)
    np.testing.assert_allclose(cw.U, c1.U, atol=1e-11)
    np.testing.assert_allclose(sum(cw.E_new) / W, c1.E_new[0], atol=1e-11)
    # and the sum of the workers' Q_w is (sum_w M_w)^T Phat
    np.testing.assert_allclose(sum(cw.Q_w), sum(Ms).T @ cw.Phat, atol=1e-11)


def check_conservation(compress):
    # Per worker: M_w = Phat Q_w^T + E_new_w, and Phat^T E_new_w = 0.
    rng = _rng(40)
    n, m, r, W = 50, 35, 2, 3
    Ms = [rng.standard_normal((n, m)) + 3.0 * np.outer(rng.standard_normal(n), rng.standard_normal(m))
          for _ in range(W)]
    c = compress(Ms, rng.standard_normal((m, r)))
    for w in range(W):
        np.testing.assert_allclose(c.Phat @ c.Q_w[w].T + c.E_new[w], Ms[w], atol=1e-12)
        assert np.abs(c.Phat.T @ c.E_new[w]).max() < 1e-11
        np.testing.assert_allclose(c.Q_w[w], Ms[w].T @ c.Phat, atol=1e-12)
    np.testing.assert_allclose(W * c.U + sum(c.E_new), sum(Ms), atol=1e-11)


def check_power_iteration_to_svd(compress):
    # Fixed M, no error feedback: warm-started compressions approach the best
    # rank-r approximation (Eckart-Young, from a brute-force SVD).
    rng = _rng(50)
    n, m, r = 12, 8, 2
    U0, _ = np.linalg.qr(rng.standard_normal((n, n)))
    V0, _ = np.linalg.qr(rng.standard_normal((m, m)))
    sig = np.array([10.0, 5.0, 2.0, 1.0, 0.5, 0.2, 0.1, 0.05])
    M = (U0[:, :m] * sig) @ V0.T
    u, s, vt = np.linalg.svd(M)
    Mr = (u[:, :r] * s[:r]) @ vt[:r]
    best = math.sqrt(float(np.sum(s[r:] ** 2)))
    Q = rng.standard_normal((m, r))
    errs = []
    for _ in range(40):
        c = compress([M], Q)
        Q = c.Qbar
        errs.append(np.linalg.norm(M - c.U))
    assert errs[-1] == pytest.approx(best, rel=1e-12)
    np.testing.assert_allclose(c.U, Mr, atol=1e-10)
    # the gap closes monotonically, roughly as (sigma_{r+1}/sigma_r)^(2k)
    gaps = np.array(errs) - best
    assert np.all(np.diff(gaps[:15]) <= 1e-12)
    assert gaps[5] < gaps[0] * 0.5


def check_error_feedback_telescopes(state_cls):
    # Over T steps with error feedback, everything the workers fed in is either
    # sent or still held as error:  sum_t sum_w G_w,t = W sum_t U_t + sum_w E_w,T.
    rng = _rng(60)
    layers = [(20, 12), (9, 0), (6, 30)]
    W, r, T = 3, 2, 5
    st = state_cls(layers, r, W, seed=7)
    tot_g = {0: 0.0, 2: 0.0}
    tot_u = {0: 0.0, 2: 0.0}
    for t in range(T):
        G = [[rng.standard_normal(s if s[1] else (s[0],)) for s in layers] for _ in range(W)]
        Qprev = [None if q is None else q.copy() for q in st.Q]
        Eprev = [None if e is None else [x.copy() for x in e] for e in st.E]
        out = st.step(G)
        for li in (0, 2):
            tot_g[li] = tot_g[li] + sum(G[w][li] for w in range(W))
            tot_u[li] = tot_u[li] + out.U[li]
            # the step compressed M_w = G_w + E_w with the previous Q
            c = O.compress([G[w][li] + Eprev[li][w] for w in range(W)], Qprev[li])
            np.testing.assert_allclose(out.U[li], c.U, atol=1e-12)
            # warm start: the next Q is this step's mean Q
            np.testing.assert_allclose(st.Q[li], out.Qbar[li], atol=0)
        np.testing.assert_allclose(out.U[1], sum(G[w][1] for w in range(W)) / W, atol=1e-14)
    for li in (0, 2):
        np.testing.assert_allclose(tot_g[li], W * tot_u[li] + sum(st.E[li]), atol=1e-10)


# --------------------------------------------------------------- tests -----

def test_gram_schmidt():
    check_gram_schmidt(O.gram_schmidt)


def test_exact_rank_recovery_one_step():
    check_exact_rank_recovery(O.compress)


def test_exact_rank_recovery_with_warm_start_and_ef():
    # W=2 workers feed the same exact rank-r gradient every step: every step
    # recovers it exactly and the error buffers stay zero.
    rng = _rng(21)
    n, m, r, W = 40, 24, 3, 2
    A = rng.standard_normal((n, r)) @ rng.standard_normal((r, m))
    st = O.OracleState([(n, m)], r, W, seed=5)
    for _ in range(10):
        out = st.step([[A] for _ in range(W)])
        np.testing.assert_allclose(out.U[0], A, atol=1e-10)
        for E in st.E[0]:
            assert np.abs(E).max() < 1e-10


def test_linearity():
    check_linearity(O.compress)


def test_conservation_and_orthogonality():
    check_conservation(O.compress)


def test_power_iteration_approaches_best_rank_r():
    check_power_iteration_to_svd(O.compress)


def test_error_feedback_telescopes():
    check_error_feedback_telescopes(O.OracleState)


def test_data_sent_matches_results_table(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "powersgd_results_table.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, rank, mb = line.split()
                rows.append((name, int(rank), int(mb)))
    layers = workloads.resnet18_cifar_layers()
    steps_per_epoch = 24
    for name, rank, mb in rows:
        comp, unc = O.data_sent_per_step(layers, max(rank, 1))
        floats = unc if rank == 0 else comp
        mib = floats * 4 * steps_per_epoch / 2 ** 20
        assert round(mib) == mb, (name, mib, mb)
    # the exact integers behind the table
    assert O.data_sent_per_step(layers, 1) == (45_935, 11_173_962)
    assert O.data_sent_per_step(layers, 2) == (82_260, 11_173_962)
    assert O.data_sent_per_step(layers, 4) == (154_910, 11_173_962)
    # "compresses gradients more than 120x" (main findings, bullet 1), at rank 2
    comp, unc = O.data_sent_per_step(layers, 2)
    assert unc / comp > 120


def test_resnet18_shape_inventory():
    layers = workloads.resnet18_cifar_layers()
    mats = [s for s in layers if s[1]]
    assert len(mats) == 21
    assert sum(n * m for n, m in mats) == 11_164_352
    assert sum(n for n, m in layers if m == 0) == 9_610


def test_q_init_distribution_and_determinism():
    q = O.q_init(123, 0, 4096, 8).astype(np.float64).ravel()
    assert q.dtype == np.float64 and q.size == 32768
    ks = scipy.stats.kstest(q, "norm")
    assert ks.pvalue > 1e-3
    assert abs(q.mean()) < 0.03 and abs(q.var() - 1.0) < 0.03
    # determinism, and distinct streams per layer and per seed
    np.testing.assert_array_equal(O.q_init(123, 0, 10, 3), O.q_init(123, 0, 10, 3))
    assert not np.allclose(O.q_init(123, 1, 10, 3), O.q_init(123, 0, 10, 3))
    assert not np.allclose(O.q_init(124, 0, 10, 3), O.q_init(123, 0, 10, 3))
    # odd m*r: the last pair's second draw is dropped, the rest is a prefix
    a = O.q_init(5, 2, 7, 1).ravel()
    b = O.q_init(5, 2, 8, 1).ravel()
    np.testing.assert_array_equal(a, b[:7])


def test_splitmix64_stream_matches_counter_form():
    # The stream (state += gamma; output mix(state)) equals the counter form
    # mix(seed + k*gamma), which the vectorised Q initialiser relies on.
    xs = O.splitmix64_stream(0xDEADBEEF, 5)
    for k, x in enumerate(xs, start=1):
        assert x == O.splitmix64_mix((0xDEADBEEF + k * O.GOLDEN_GAMMA) & O.MASK64)
    # mix is a bijection on 64-bit words: its three steps are each invertible
    # (xorshift by >= 32 bits is its own inverse; odd multipliers have inverses)
    def unmix(z):
        z = (z ^ (z >> 31) ^ (z >> 62)) & O.MASK64
        z = (z * pow(0x94D049BB133111EB, -1, 1 << 64)) & O.MASK64
        z = (z ^ (z >> 27) ^ (z >> 54)) & O.MASK64
        z = (z * pow(0xBF58476D1CE4E5B9, -1, 1 << 64)) & O.MASK64
        z = (z ^ (z >> 30) ^ (z >> 60)) & O.MASK64
        return z
    for v in [0, 1, 12345, O.MASK64, 0x0123456789ABCDEF]:
        assert unmix(O.splitmix64_mix(v)) == v
    # the first outputs of the generator's public reference code (Vigna's
    # splitmix64.c) seeded with 0
    assert O.splitmix64_stream(0, 4) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                         0x06C45D188009454F, 0xF88BB8A8724C81EC]
    assert O.uniform_open0(0) == 2.0 ** -53
    assert O.uniform_open0(O.MASK64) == 1.0


def test_zero_gradient_step():
    st = O.OracleState([(16, 8)], 2, 2, seed=1)
    out = st.step([[np.zeros((16, 8))] for _ in range(2)])
    assert np.all(out.Phat[0] == 0) and np.all(out.Qbar[0] == 0) and np.all(out.U[0] == 0)
    assert all(np.all(E == 0) for E in st.E[0])


def check_momentum_update(update):
    rng = np.random.default_rng(9)
    x0, U = rng.standard_normal((5, 3)), rng.standard_normal((5, 3))
    lr = 0.1
    # beta = 0: the step is x - 2 lr U and the momentum is U
    x1, m1 = update(x0, np.zeros_like(x0), U, lr, 0.0)
    np.testing.assert_allclose(m1, U, rtol=1e-15)
    np.testing.assert_allclose(x1, x0 - 2 * lr * U, rtol=1e-14, atol=1e-15)
    # constant U from zero momentum: closed forms of the geometric sums
    beta, k = 0.9, 7
    x, m = x0.copy(), np.zeros_like(x0)
    for _ in range(k):
        x, m = update(x, m, U, lr, beta)
    np.testing.assert_allclose(m, U * (1 - beta ** k) / (1 - beta), rtol=1e-13)
    summed = (k - beta * (1 - beta ** k) / (1 - beta)) / (1 - beta)  # sum of the k momenta / U
    np.testing.assert_allclose(x, x0 - lr * U * (k + summed), rtol=1e-13, atol=1e-14)


def test_momentum_update_closed_forms():
    check_momentum_update(O.momentum_update)


@pytest.mark.parametrize("kind", ["heavy_ball_step", "old_momentum_in_step", "sign"])
def test_planted_momentum_mistakes_are_caught(kind):
    def mutant(x, mom, U, lr, beta):
        m_new = beta * mom + U
        if kind == "heavy_ball_step":
            return x - lr * m_new, m_new
        if kind == "old_momentum_in_step":
            return x - lr * (U + mom), m_new
        return x + lr * (U + m_new), m_new
    with pytest.raises(AssertionError):
        check_momentum_update(mutant)


def check_unbiased(compress):
    rng = np.random.default_rng(13)
    n, m, W = 10, 6, 2
    G = [rng.standard_normal((n, m)) for _ in range(W)]
    Gbar = sum(G) / W
    # a Q with Q Q^T = r I exactly (r = m, Q = sqrt(r) I): U is the mean gradient
    _, U = compress(G, math.sqrt(m) * np.eye(m))
    np.testing.assert_allclose(U, Gbar, rtol=0, atol=1e-12)
    # unbiasedness: the mean of U over many fresh N(0,1) draws of Q approaches
    # the mean gradient within a few standard errors
    r, K = 2, 4000
    Us = np.stack([compress(G, O.q_init(O.step_seed(99, t), 0, m, r).astype(np.float64))[1] for t in range(K)])
    se = Us.std(axis=0) / math.sqrt(K)
    assert np.max(np.abs(Us.mean(axis=0) - Gbar) / se) < 5.0
    # and a single draw is far from it (the estimate is noisy, not exact)
    assert np.linalg.norm(Us[0] - Gbar) > 0.1 * np.linalg.norm(Gbar)


def test_unbiased_variant():
    check_unbiased(O.unbiased_compress)
    # fresh Q per step: distinct steps, same seed -> distinct draws; deterministic
    a = O.q_init(O.step_seed(5, 0), 1, 7, 2)
    assert not np.allclose(a, O.q_init(O.step_seed(5, 1), 1, 7, 2))
    np.testing.assert_array_equal(a, O.q_init(O.step_seed(5, 0), 1, 7, 2))
    # only P travels: n r per matrix, vectors whole
    layers = workloads.resnet18_cifar_layers()
    assert O.unbiased_data_sent(layers, 2) == 2 * sum(n for n, m in layers if m) + sum(n for n, m in layers if not m)
    # the layer-set step averages vectors and compresses matrices with step t's Q
    rng = np.random.default_rng(3)
    lay = [(8, 5), (4, 0)]
    grads = [[rng.standard_normal((8, 5)), rng.standard_normal(4)] for _ in range(3)]
    out = O.unbiased_step(grads, lay, 2, seed=7, step=4)
    Q = O.q_init(O.step_seed(7, 4), 0, 5, 2).astype(np.float64)
    np.testing.assert_allclose(out.Qbar[0], Q, atol=0)
    np.testing.assert_allclose(out.U[1], sum(g[1] for g in grads) / 3, atol=1e-15)


@pytest.mark.parametrize("kind", ["no_rank_scale", "sum_not_mean", "off_scale"])
def test_planted_unbiased_mistakes_are_caught(kind):
    def mutant(G, Q):
        W, r = len(G), Q.shape[1]
        P = sum(np.asarray(g, dtype=np.float64) @ Q for g in G)
        if kind == "no_rank_scale":
            return P, P @ Q.T / W
        if kind == "sum_not_mean":
            return P, P @ Q.T / r
        return P, (P @ Q.T / (W * r)) * (1.0 + 1e-3)
    with pytest.raises(AssertionError):
        check_unbiased(mutant)


def check_rtopk(select):
    rng = np.random.default_rng(21)
    # distinct magnitudes: the top set is numpy's partition of |M|
    M = rng.standard_normal((20, 15)).astype(np.float32)
    d = M.size
    r, k = O.rtopk_counts(d, 7, 1)
    sel = select(M, r, k, 12345)
    want = np.sort(np.argpartition(-np.abs(M.ravel()), r - 1)[:r])
    np.testing.assert_array_equal(sel, want)
    # with sampling: k distinct indices out of that top set
    r, k = O.rtopk_counts(d, 7, 3)
    sel = select(M, r, k, 99)
    assert len(sel) == k and len(set(sel.tolist())) == k and set(sel.tolist()) <= set(want.tolist())
    # every entry kept (r = k = d): all indices
    np.testing.assert_array_equal(select(M, d, d, 5), np.arange(d))
    # ties (all zero): the top set is the lowest indices
    Z = np.zeros((6, 5), dtype=np.float32)
    assert set(select(Z, 8, 8, 1).tolist()) == set(range(8))
    assert set(select(Z, 8, 3, 1).tolist()) <= set(range(8))
    # uniform subset: over many draws each top-set entry is sent k / r of the time
    r, k = 12, 4
    counts = np.zeros(d)
    draws = 3000
    for t in range(draws):
        counts[select(M, r, k, O.rtopk_draw_key(7, t, 0, 0))] += 1
    top = np.argpartition(-np.abs(M.ravel()), r - 1)[:r]
    p = k / r
    se = math.sqrt(draws * p * (1 - p))
    assert np.all(np.abs(counts[top] - draws * p) < 5 * se) and counts.sum() == draws * k


def test_rtopk_select():
    check_rtopk(O.rtopk_select)


def test_rtopk_step_conservation_and_full_case():
    rng = np.random.default_rng(4)
    layers = [(12, 9), (5, 0), (7, 13)]
    W = 3
    grads = lambda: [[rng.standard_normal(s if s[1] else (s[0],)).astype(np.float32) for s in layers] for _ in range(W)]
    # r = k = d: nothing left behind, U is the float32 mean
    st = O.RTopKState(layers, W, seed=3, top_div=1, sample_div=1)
    g = grads()
    U, sent = st.step(g)
    for li, (n, m) in enumerate(layers):
        if m:
            tot = np.zeros(n * m, dtype=np.float32)
            for w in range(W):
                tot = (tot + g[w][li].ravel()).astype(np.float32)
                assert np.all(st.E[li][w] == 0)
            np.testing.assert_array_equal(U[li].ravel(), (tot * np.float32(1.0 / W)).astype(np.float32))
    # sampling with error feedback: M = S + E exactly, k entries sent per worker
    st = O.RTopKState(layers, W, seed=3, top_div=4, sample_div=2)
    for t in range(3):
        Eold = [None if e is None else [x.copy() for x in e] for e in st.E]
        g = grads()
        U, sent = st.step(g)
        for li, (n, m) in enumerate(layers):
            if not m:
                continue
            r, k = O.rtopk_counts(n * m, 4, 2)
            u = np.zeros(n * m, dtype=np.float32)
            for w in range(W):
                M = (g[w][li] + Eold[li][w]).ravel().astype(np.float32)
                S = np.zeros_like(M)
                S[sent[li][w]] = M[sent[li][w]]
                assert len(sent[li][w]) == k
                np.testing.assert_array_equal(S + st.E[li][w].ravel(), M)
                u = (u + S).astype(np.float32)
            np.testing.assert_array_equal(U[li].ravel(), (u * np.float32(1.0 / W)).astype(np.float32))
    assert O.rtopk_data_sent(layers, 4, 2) == 2 * O.rtopk_counts(108, 4, 2)[1] + 2 * O.rtopk_counts(91, 4, 2)[1] + 5


@pytest.mark.parametrize("kind", ["smallest", "ties_high_index", "no_subset_draw"])
def test_planted_rtopk_mistakes_are_caught(kind):
    def mutant(M, r, k, key):
        a = np.abs(np.asarray(M, dtype=np.float32).ravel())
        idx = np.arange(a.size)
        if kind == "smallest":
            order = np.lexsort((idx, a.astype(np.float64)))
        elif kind == "ties_high_index":
            order = np.lexsort((-idx, -a.astype(np.float64)))
        else:
            order = np.lexsort((idx, -a.astype(np.float64)))
            return np.sort(order[:k])  # the k largest, not a random k of the top r
        return np.sort(order[:r][:k])
    with pytest.raises(AssertionError):
        check_rtopk(mutant)


# ------------------------------------------------- planted mistakes -----

def _mutant_compress(kind):
    def compress(M, Q):
        W = len(M)
        M = [np.asarray(x, dtype=np.float64) for x in M]
        P = sum(Mw @ Q for Mw in M)
        Ph = O.gram_schmidt(P) if kind != "no_orthonormalise" else P / np.linalg.norm(P, axis=0)
        Q_w = [Mw.T @ Ph for Mw in M]
        Qbar = sum(Q_w) / (1 if kind == "sum_not_mean" else W)
        U = Ph @ Qbar.T
        if kind == "error_uses_qbar":
            E = [Mw - Ph @ Qbar.T for Mw in M]
        elif kind == "error_sign":
            E = [Ph @ q.T - Mw for Mw, q in zip(M, Q_w)]
        elif kind == "transposed_q":
            E = [Mw - (q @ Ph.T).T * 0.5 - Ph @ q.T * 0.5 for Mw, q in zip(M, Q_w)]
            U = U * 1.0001
        else:
            E = [Mw - Ph @ q.T for Mw, q in zip(M, Q_w)]
        return O.Compressed(P, Ph, Q_w, Qbar, U, E)
    return compress


def _mutant_gs(kind):
    # "single_pass": plain modified Gram-Schmidt, one pass per column
    def gs(P):
        Ph = np.array(P, dtype=np.float64)
        for k in range(Ph.shape[1]):
            v = Ph[:, k]
            for _ in range(1 if kind == "single_pass" else 2):
                for j in range(k):
                    if kind == "skip_last_projection" and j == k - 1:
                        continue
                    coef = Ph[:, j] @ v
                    v -= (coef if kind != "projection_sign" else -coef) * Ph[:, j]
            Ph[:, k] = v / np.linalg.norm(v)
        return Ph
    return gs


class _NoFeedbackState(O.OracleState):
    def step(self, grads, layers=None):
        for e in self.E:
            if e is not None:
                for x in e:
                    x[:] = 0.0
        return super().step(grads, layers)


@pytest.mark.parametrize("kind", ["sum_not_mean", "error_uses_qbar", "error_sign",
                                  "no_orthonormalise", "transposed_q"])
def test_planted_mistakes_are_caught(kind):
    mut = _mutant_compress(kind)
    caught = 0
    for check in (check_exact_rank_recovery, check_linearity, check_conservation,
                  check_power_iteration_to_svd):
        try:
            check(mut)
        except AssertionError:
            caught += 1
    assert caught >= 1, kind


@pytest.mark.parametrize("kind", ["skip_last_projection", "projection_sign", "single_pass"])
def test_planted_gram_schmidt_mistakes_are_caught(kind):
    with pytest.raises(AssertionError):
        check_gram_schmidt(_mutant_gs(kind))


def test_planted_missing_error_feedback_is_caught():
    with pytest.raises(AssertionError):
        check_error_feedback_telescopes(_NoFeedbackState)
