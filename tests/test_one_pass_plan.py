"""The one-pass project's persistent schedule (host only, no GPU).

The cluster kernel of the one-pass project runs one cluster per resident slot
over a fixed schedule, so its correctness and its balance rest on the plan.
Checked on the layer sets of the workloads and on ragged shapes:

* the column split: cw CTAs (a power of two, at most 8) of yfc float4 columns
  cover each row; a CTA's Y accumulators (its pairs, in whole rounds of 256,
  x RP float4) fit in 64 KB; no other cw within that bound has fewer pair
  rounds per row (ties go to the larger cw);
* the block height: 1 <= yr <= 16 / RP, and a CTA's block of M is at most
  64 KB unless the block is a single row;
* coverage: every block of every layer is in exactly one segment, a layer's
  segments are disjoint, and its slots 0 .. nys - 1 each appear once;
* balance: no run is longer than the mean by more than one round of its
  costliest layer.
"""
import pytest

import workloads

CLUSTER, THREADS, YSMEM, YBLOCK = 8, 256, 64 * 1024, 64 * 1024


@pytest.fixture(scope="module")
def pkg():
    import rank_gradient_compression_layer_gb300 as p
    p.build()
    return p


def _ceil(a, b):
    return -(-a // b)


def _padded(rank):
    return 1 << (rank - 1).bit_length()


def _smem(pairs, rp):
    return _ceil(pairs, THREADS) * THREADS * rp * 16


def _sets():
    ragged = [(7, 5), (33, 6), (100, 4100), (1000, 300), (64, 27), (513, 2305), (16, 0), (5, 9), (130, 130),
              (1, 1), (2049, 13)]
    return [
        ("resnet18", workloads.c2_resnet18().layers, 2, 4, 36),
        ("lstm", workloads.c3_lstm().layers, 4, 4, 36),
        ("square8192_r1_w8", [(8192, 8192)], 1, 8, 36),
        ("square8192_r2_w8", [(8192, 8192)], 2, 8, 36),
        ("ragged_r1_w3", ragged, 1, 3, 36),
        ("ragged_r2_w5_few_clusters", ragged, 2, 5, 3),
        ("ragged_r3_w2", [s for s in ragged if s[1] == 0 or min(s) >= 3], 3, 2, 19),
    ]


@pytest.mark.parametrize("name,shapes,rank,workers,clusters", _sets(), ids=[s[0] for s in _sets()])
def test_one_pass_schedule(pkg, name, shapes, rank, workers, clusters):
    rp = _padded(rank)
    layers, runs = pkg.psgd_plan_one_pass(shapes, rank, workers, clusters)
    mats = [(n, m) for n, m in shapes if m]
    assert len(layers) == len(mats) and len(runs) == clusters
    seen = [dict() for _ in mats]  # per layer: block -> segment
    slots = [set() for _ in mats]
    block_cost = []
    for li, ((n, m), (cw, yfc, yr, nys)) in enumerate(zip(mats, layers)):
        F = _ceil(m, 4)
        # the column split
        assert cw in (1, 2, 4, 8) and cw * yfc >= F and (cw - 1) * yfc < F
        pairs = yfc * workers
        assert _smem(pairs, rp) <= YSMEM
        rounds = cw * _ceil(pairs, THREADS)
        for other in (1, 2, 4, 8):
            p2 = _ceil(F, other) * workers
            if _smem(p2, rp) <= YSMEM:
                r2 = other * _ceil(p2, THREADS)
                assert r2 > rounds or (r2 == rounds and other <= cw), (li, cw, other)
        # the block height
        assert 1 <= yr <= 16 // rp
        assert yr == 1 or yr * pairs * 16 <= YBLOCK
        block_cost.append(cw * yr * _ceil(pairs, THREADS))
    for c, run in enumerate(runs):
        for (li, b0, b1, slot) in run:
            cw, yfc, yr, nys = layers[li]
            n = mats[li][0]
            assert 0 <= b0 < b1 <= _ceil(n, yr)
            assert 0 <= slot < nys and slot not in slots[li]
            slots[li].add(slot)
            for b in range(b0, b1):
                assert b not in seen[li], (li, b)
                seen[li][b] = (c, slot)
    for li, (n, m) in enumerate(mats):
        cw, yfc, yr, nys = layers[li]
        assert sorted(seen[li]) == list(range(_ceil(n, yr))), li
        assert slots[li] == set(range(nys)), li
    # balance: a segment of k blocks takes ceil(k / S) rounds of S blocks
    cost = []
    for run in runs:
        t = 0
        for (li, b0, b1, _) in run:
            S = CLUSTER // layers[li][0]
            t += _ceil(b1 - b0, S) * S * block_cost[li]
        cost.append(t)
    mean = sum(cost) / clusters
    worst_round = max((CLUSTER // layers[li][0]) * block_cost[li] for li in range(len(mats)))
    assert max(cost) <= mean + worst_round, (max(cost), mean, worst_round)


def test_one_pass_plan_rejects_what_it_cannot_run(pkg):
    from rank_gradient_compression_layer_gb300 import PSGD_ERR_INVALID, PsgdError

    with pytest.raises(PsgdError) as ei:  # rank above 4
        pkg.psgd_plan_one_pass([(64, 64)], 8, 2, 4)
    assert ei.value.code == PSGD_ERR_INVALID
    with pytest.raises(PsgdError) as ei:  # 8192 columns x 8 workers at r = 4: no split fits 64 KB of Y
        pkg.psgd_plan_one_pass([(8192, 8192)], 4, 8, 4)
    assert ei.value.code == PSGD_ERR_INVALID
    with pytest.raises(PsgdError) as ei:
        pkg.psgd_plan_one_pass([(64, 64)], 2, 2, 0)
    assert ei.value.code == PSGD_ERR_INVALID
