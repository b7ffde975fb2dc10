"""Host logic of bench.py: byte accounting, workload names, source hashes.

No GPU: these check the numbers the bench line is built from against
independent counts (the oracle's data-sent formula, the layer tables).
"""
import pytest

import bench
import workloads
from oracle import powersgd as O


def test_rtopk_bytes_split_and_messages():
    cfg = workloads.c2_resnet18()
    ab = bench.rtopk_bytes(cfg, 100, 4)
    nm = sum(n * m for n, m in cfg.matrices)
    assert nm == 11164352  # the ResNet-18 layer table's matrix elements
    # pass 0: G and E read, M written per worker, U zeroed once
    assert ab["pass0"] == (3 * cfg.workers + 1) * nm * 4 == 580546304
    # every worker's message: the oracle's per-worker count of the matrix layers, in bytes
    per_worker = O.rtopk_data_sent(cfg.matrices, 100, 4)
    assert ab["messages"] == cfg.workers * per_worker * 4
    assert ab["total"] == ab["pass0"] + ab["messages"] + ab["vectors"]


def test_powersgd_bytes_include_factors_and_update():
    cfg = workloads.c2_resnet18()
    ab = bench.algorithmic_bytes(cfg, with_update=True)
    nm = sum(n * m for n, m in cfg.matrices)
    factors = sum(4 * (n + m) * cfg.rank for n, m in cfg.matrices)
    assert ab["core"] == cfg.workers * 3 * nm * 4 + factors
    assert ab["update"] == nm * 4
    assert bench.algorithmic_bytes(cfg, with_update=False)["vectors"] == 0


@pytest.mark.parametrize("name,shape,workers,rank", [
    ("c5r8", (8192, 8192), 8, 8),
    ("c5s32", (4096, 4096), 4, 32),
])
def test_rank_sweep_config_names(name, shape, workers, rank):
    cfg = bench.config_of(name)
    assert cfg.layers == (shape,) and cfg.workers == workers and cfg.rank == rank


def test_repeated_resnet_config():
    base = workloads.c2_resnet18()
    cfg = bench.config_of("c2x3")
    assert list(cfg.layers) == list(base.layers) * 3 and cfg.rank == base.rank


def test_source_hashes_per_variant_and_traffic_keys():
    # the rTop-k hash covers more files, so an rTop-k edit leaves PowerSGD's traffic valid
    assert bench.kernel_sources_hash() != bench.kernel_sources_hash(rtopk=True)
    for key, (h, nbytes) in bench.NCU_TRAFFIC.items():
        assert isinstance(key, tuple) and key[1] in ("powersgd", "rtopk")
        assert len(h) == 16 and nbytes > 0


def test_source_hash_ignores_comments_only():
    # comments and blank lines are left out; code, and a // inside it, is kept
    src = "int a; // note\n/* block\n   comment */\n\nint b = 2;  /* x */ int c;\n"
    assert bench._code_only(src) == "int a;\nint b = 2;   int c;"
    assert bench._code_only(src) == bench._code_only(src.replace("note", "another note"))
    assert bench._code_only(src) != bench._code_only(src.replace("b = 2", "b = 3"))
