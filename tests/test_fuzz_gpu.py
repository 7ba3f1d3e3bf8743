"""Seeded random shapes through the sparse and window paths, every row against
the oracle.

Each case draws KV groups, heads, page size, region size, region count,
query_len, cache dtype, gate, inactive rows, -1 padding and the split count
from a seeded generator, within what the library accepts (the piece
P = min(region, page, stage) must be a multiple of 8 dividing both region and
page), at sizes the float64 oracle finishes quickly."""
import numpy as np
import pytest

from gpu_util import check, oracle_rows, oracle_swa_rows, run, run_swa
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _piece_ok(fp8, block, rt):
    piece = min(rt, block, 64 if fp8 else 32)
    return piece % 8 == 0 and rt % piece == 0 and block % piece == 0


def sparse_case(seed):
    rng = np.random.default_rng(1000 + seed)
    fp8 = bool(rng.integers(0, 2))
    while True:
        block = int(rng.choice([8, 16, 24, 32, 48, 64, 128]))
        rt = int(rng.choice([8, 16, 24, 32, 64, 128, block, 2 * block]))
        if _piece_ok(fp8, block, rt):
            break
    groups = int(rng.choice([1, 2, 3, 4, 8]))
    cfg = inputs.scaled(
        "gqa", requests=int(rng.integers(1, 5)), query_len=int(rng.integers(1, 4)), groups=groups,
        heads=int(rng.integers(1, 17)), block=block, region_tokens=rt, num_regions=int(rng.integers(1, 49)),
        ctx=(int(rng.integers(1, 400)), int(rng.integers(400, 3000))), fp8=fp8, gate=bool(rng.integers(0, 2)),
        inactive_frac=float(rng.choice([0.0, 0.2])), pad_max=int(rng.choice([0, 0, 3])),
        short_frac=0.0, seed=seed)
    splits = [None, 1, 2, 3, 7][int(rng.integers(0, 5))]
    return cfg, splits


def window_case(seed):
    rng = np.random.default_rng(2000 + seed)
    fp8 = bool(rng.integers(0, 2))
    while True:
        block = int(rng.choice([8, 16, 24, 32, 48, 64]))
        if _piece_ok(fp8, block, block):
            break
    cfg = inputs.scaled(
        "swa", requests=int(rng.integers(1, 5)), query_len=int(rng.integers(1, 5)),
        groups=int(rng.choice([1, 2, 4])), heads=int(rng.integers(1, 17)), block=block,
        ctx=(int(rng.integers(1, 300)), int(rng.integers(300, 2500))), fp8=fp8,
        gate=bool(rng.integers(0, 2)), window=int(rng.integers(1, 3000)), seed=seed)
    splits = [None, 1, 2, 5][int(rng.integers(0, 4))]
    return cfg, splits


@pytest.mark.parametrize("seed", range(24))
def test_random_sparse_shapes(seed):
    cfg, splits = sparse_case(seed)
    w = inputs.make_workload(cfg, DEV, fill="all")
    rows = list(range(w.rows))
    out, flags = run(w, splits=splits)
    assert flags == 0
    check(w, out, oracle_rows(w, rows), rows)


@pytest.mark.parametrize("seed", range(8))
def test_random_window_shapes(seed):
    cfg, splits = window_case(seed)
    w = inputs.make_workload(cfg, DEV, fill="all")
    rows = list(range(w.rows))
    out, flags = run_swa(w, splits=splits)
    assert flags == 0
    check(w, out, oracle_swa_rows(w, rows), rows)
