"""Host-side checks of libpsgd.so that need no GPU: build, exports, layout,
data-sent counters and argument validation."""
import ctypes
import os
import re

import pytest

import workloads
from oracle import powersgd as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    import rank_gradient_compression_layer_gb300 as p
    p.build()
    return p


def _declared():
    src = open(os.path.join(ROOT, "include", "psgd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(psgd_[A-Za-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(pkg):
    names = _declared()
    assert len(names) >= 15
    lib = pkg.lib()
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(pkg.EXPORTS) == names


def test_layout_alignment_and_padding(pkg):
    shapes = [(64, 27), (10, 0), (5, 6), (3, 4), (7, 0), (33278, 650)]
    off, ld, total = pkg.psgd_plan_layout(shapes)
    pos = 0
    for (n, m), o, l in zip(shapes, off, ld):
        assert o % 4 == 0 and o == pos
        if m:
            assert l == (m + 3) // 4 * 4
            pos += n * l
        else:
            assert l == 0
            pos += (n + 3) // 4 * 4
    assert total == pos


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4"])
def test_data_sent_counts_match_oracle(pkg, name):
    cfg = workloads.ALL[name]()
    for r in (1, 2, 4, cfg.rank):
        assert pkg.psgd_count_sent(cfg.layers, r) == O.data_sent_per_step(cfg.layers, r)


def test_data_sent_counts_rank_sweep(pkg):
    for r in (1, 2, 4, 8, 16, 32):
        cfg = workloads.c5_rank_sweep(r)
        assert pkg.psgd_count_sent(cfg.layers, r) == ((8192 + 8192) * r, 8192 * 8192)


def test_resnet18_message_matches_results_table(pkg):
    # 24 steps per epoch, 4-byte floats: 1023 / 4 / 8 / 14 MB (PowerSGD review page, results table)
    layers = workloads.resnet18_cifar_layers()
    mb = lambda f: round(f * 4 * 24 / 2 ** 20)
    assert mb(pkg.psgd_count_sent(layers, 1)[1]) == 1023
    assert [mb(pkg.psgd_count_sent(layers, r)[0]) for r in (1, 2, 4)] == [4, 8, 14]


def test_create_rejects_bad_arguments_before_touching_the_gpu(pkg):
    lib = pkg.lib()
    h = ctypes.c_void_p()
    n = (ctypes.c_int64 * 2)(16, 8)
    m = (ctypes.c_int64 * 2)(8, 0)
    cases = [
        (2, n, m, 0, 2),     # rank 0
        (2, n, m, 33, 2),    # rank > 32
        (2, n, m, 9, 2),     # rank > min(n, m) of layer 0
        (2, n, m, 2, 0),     # no workers
        (2, n, m, 2, 65),    # too many workers
        (0, n, m, 2, 2),     # no layers
    ]
    for L, nn, mm, r, W in cases:
        rc = lib.psgd_create(ctypes.byref(h), L, nn, mm, r, W, 0, None)
        assert rc == pkg.PSGD_ERR_INVALID, (L, r, W)
        assert lib.psgd_last_error()
    neg = (ctypes.c_int64 * 1)(-3)
    assert lib.psgd_create(ctypes.byref(h), 1, neg, (ctypes.c_int64 * 1)(4), 1, 1, 0, None) == pkg.PSGD_ERR_INVALID


def test_null_context_calls_fail_cleanly(pkg):
    lib = pkg.lib()
    assert lib.psgd_step(None, None, None) == pkg.PSGD_ERR_INVALID
    assert lib.psgd_sync(None) == pkg.PSGD_ERR_INVALID
    assert lib.psgd_get_PQ(None, 0, None, None) == pkg.PSGD_ERR_INVALID
    lib.psgd_destroy(None)
