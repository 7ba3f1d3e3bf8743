"""Seeded random shapes through every kernel, against the oracle: the sparse and
window paths row by row, the indexer score by score, the selection id by id.

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


def index_case(seed):
    rng = np.random.default_rng(3000 + seed)
    block = int(rng.choice([8, 16, 32, 64, 128, 256]))   # 64 and up: the tensor-core kernel
    lo = int(rng.integers(1, 3000))
    kw = dict(requests=int(rng.integers(1, 6)), groups=int(rng.integers(1, 9)),
              query_len=int(rng.integers(1, 5)), ctx=(lo, lo + int(rng.integers(0, 9000))), block=block,
              seed=seed)
    if rng.integers(0, 3) == 0:
        kw["n_cols"] = int(rng.integers(0, 600))
    return kw


@pytest.mark.parametrize("seed", range(24))
def test_random_indexer_shapes(seed):
    import torch
    import oracle
    w = inputs.make_index_workload(DEV, **index_case(seed))
    scores = torch.full((w.rows, w.n_cols), float("nan"), device=DEV)
    cur = torch.full((w.rows,), -7, dtype=torch.int32, device=DEV)
    lens = torch.full((w.rows,), -7, dtype=torch.int32, device=DEV)
    import sparse_decode_attention_02_gb300 as sda
    sda.sparse_decode_summary_scores(w.query, w.weights, w.summaries, w.block_table, w.seq_lens,
                                     block_size=w.block, query_len=w.query_len, scores=scores,
                                     current=cur, lengths=lens)
    torch.cuda.synchronize()
    q, m = w.query.cpu().view(torch.uint8), w.summaries.cpu().view(torch.uint8)
    args = (w.block_table.cpu(), w.seq_lens.cpu())
    kw = dict(block=w.block, n_cols=w.n_cols, query_len=w.query_len)
    rs, rc, rl = oracle.summary_scores(q, w.weights.cpu(), m, *args, **kw)
    scale, _, _ = oracle.summary_scores(q & 0x7F, w.weights.cpu().abs(), m & 0x7F, *args, **kw)
    gs = scores.cpu().numpy()
    assert np.array_equal(cur.cpu().numpy(), rc) and np.array_equal(lens.cpu().numpy(), rl)
    assert np.array_equal(np.isneginf(gs), np.isneginf(rs)) and not np.isnan(gs).any()
    fin = np.isfinite(rs)
    assert (np.abs(gs[fin] - rs[fin]) <= 4e-5 * scale[fin] + 1e-6).all()


@pytest.mark.parametrize("seed", range(10))
def test_random_selection_inputs(seed):
    import torch
    import oracle
    import sparse_decode_attention_02_gb300 as sda
    rng = np.random.default_rng(4000 + seed)
    rows, n = int(rng.integers(1, 40)), int(rng.integers(1, 40000))
    topk = int(rng.integers(1, min(5000, 2 * n + 2)))
    sc = rng.standard_normal((rows, n)).astype(np.float32)
    if rng.integers(0, 2):                                        # heavy ties
        sc = np.round(sc * 2) / 2
    sc[rng.random((rows, n)) < 0.01] = np.nan
    sc[rng.random((rows, n)) < 0.01] = -0.0
    lens = rng.integers(0, n + 1, size=rows).astype(np.int32)
    cur = np.array([int(rng.integers(-1, max(1, l + 1))) for l in lens], dtype=np.int32)
    t = lambda a: torch.as_tensor(a, device=DEV)
    got = sda.sparse_decode_select_regions(t(sc), t(cur), topk, topk_lengths=t(lens))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.select_regions(sc, cur, topk, lens))
