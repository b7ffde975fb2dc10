"""The fused step's queue (host only, no GPU).

A fused step is one launch whose CTAs take queue positions in order and wait
for the flags of the phases they read.  That cannot deadlock if every tile
comes after all tiles of the phases it depends on: then each wait is on
positions already taken by running (or finished) CTAs.  These tests check
that order, and that the queue holds every tile of every phase exactly once,
on the layer sets of the workloads and on ragged shapes.
"""
import math
from collections import defaultdict

import pytest

import workloads

PROJECT, ORTHO, BACK, DECOMP = 0, 1, 2, 3
KSEG_COLS = 128   # columns per segment (32 float4)
PH_ROWS = 128     # rows per orthonormalise tile
U_ROWS = 128      # rows per decompress tile (r <= 4)
V_CHUNK = 8192    # vector elements per decompress tile


@pytest.fixture(scope="module")
def pkg():
    import rank_gradient_compression_layer_gb300 as p
    p.build()
    return p


def _sets():
    c2, c3 = workloads.c2_resnet18(), workloads.c3_lstm()
    ragged = [(1, 1), (3, 5), (33, 27), (7, 0), (130, 1), (64, 129), (257, 650), (5, 0), (2049, 13)]
    return [
        ("resnet18", c2.layers, 2, 4),
        ("lstm", c3.layers, 4, 4),
        ("ragged_r1_w3", ragged, 1, 3),
        ("ragged_r3_w9", [s for s in ragged if s[1] == 0 or min(s) >= 3], 3, 9),
    ]


@pytest.mark.parametrize("name,layers,rank,workers", _sets())
@pytest.mark.parametrize("with_update", [True, False])
@pytest.mark.parametrize("lag", [0, 1 << 20, 1 << 40])
def test_queue_order_and_completeness(pkg, name, layers, rank, workers, with_update, lag):
    q = pkg.psgd_plan_queue(layers, rank, workers, project_rows=8, lag_bytes=lag, with_update=with_update)
    mats = [(n, m) for n, m in layers if m]
    vecs = [n for n, m in layers if m == 0]
    pos = defaultdict(list)  # (phase, layer) -> queue positions
    seen = set()
    for i, (phase, li, a, b, c) in enumerate(q):
        key = (phase, li, a, b, c)
        assert key not in seen, key
        seen.add(key)
        if phase == DECOMP and c == 1:
            assert 0 <= li < len(vecs) and 0 <= a < math.ceil(vecs[li] / V_CHUNK)
            continue
        pos[(phase, li)].append(i)
    for li, (n, m) in enumerate(mats):
        S = math.ceil(math.ceil(m / 4) / 32)
        nrb = math.ceil(n / 8)
        proj = {(a, b) for (ph, l, a, b, c) in q if ph == PROJECT and l == li}
        assert proj == {(a, b) for a in range(nrb) for b in range(S)}
        orth = {a for (ph, l, a, b, c) in q if ph == ORTHO and l == li}
        assert orth == set(range(math.ceil(n / PH_ROWS)))
        back = {(a, b, c) for (ph, l, a, b, c) in q if ph == BACK and l == li}
        t3r = 1 + max(a for a, _, _ in back)
        assert back == {(a, b, c) for a in range(t3r) for b in range(S) for c in range(workers)}
        dec = {(a, b) for (ph, l, a, b, c) in q if ph == DECOMP and l == li and c == 0}
        if with_update:
            assert dec == {(a, b) for a in range(math.ceil(n / U_ROWS)) for b in range(S)}
        else:
            assert not dec
        # dependency order: project < orthonormalise < back-project < decompress
        assert max(pos[(PROJECT, li)]) < min(pos[(ORTHO, li)])
        assert max(pos[(ORTHO, li)]) < min(pos[(BACK, li)])
        if with_update:
            assert max(pos[(BACK, li)]) < min(pos[(DECOMP, li)])
    n_vec = sum(math.ceil(n / V_CHUNK) for n in vecs)
    assert sum(1 for t in q if t[0] == DECOMP and t[4] == 1) == (n_vec if with_update else 0)


def test_queue_lag_interleaves_layers(pkg):
    # with a lag, a layer's back-project tiles sit among later layers' project
    # tiles (that is what lets its error state stay in L2); with an infinite
    # lag every project tile comes first
    layers = workloads.c2_resnet18().layers
    q = pkg.psgd_plan_queue(layers, 2, 4, project_rows=32, lag_bytes=64 << 20)
    first_back = min(i for i, t in enumerate(q) if t[0] == BACK)
    last_proj = max(i for i, t in enumerate(q) if t[0] == PROJECT)
    assert first_back < last_proj
    q_inf = pkg.psgd_plan_queue(layers, 2, 4, project_rows=32, lag_bytes=1 << 50)
    assert max(i for i, t in enumerate(q_inf) if t[0] == PROJECT) < min(
        i for i, t in enumerate(q_inf) if t[0] in (ORTHO, BACK))


def test_queue_rejects_bad_arguments(pkg):
    with pytest.raises(pkg.PsgdError):
        pkg.psgd_plan_queue([(16, 8)], 0, 2)
    with pytest.raises(pkg.PsgdError):
        pkg.psgd_plan_queue([(16, 8)], 2, 2, project_rows=64)
