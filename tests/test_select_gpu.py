"""Region selection (CUDA kernel vs the oracle), and selection chained into
sparse decode attention.

Both sides keep the current region, take the best other scores, rank NaN
lowest and break ties by the lower id, so the selected ids are compared
exactly (the rule for ties is this library's reading: the page does not state
one)."""
import gc

import numpy as np
import pytest
import torch

import oracle
import sparse_decode_attention_02_gb300 as sda
from gpu_util import check, oracle_rows, run
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def select_both(scores, current, topk, lengths):
    got = sda.sparse_decode_select_regions(scores, current, topk, topk_lengths=lengths)
    torch.cuda.synchronize()
    ref = oracle.select_regions(scores.cpu(), current.cpu(), topk,
                                None if lengths is None else lengths.cpu())
    return got.cpu().numpy(), ref


@pytest.mark.parametrize("rows,n,topk", [(64, 300, 16), (33, 1000, 1000), (17, 5000, 1024),
                                         (8, 20000, 1), (5, 70000, 4096)])
@pytest.mark.parametrize("ties", [0.0, 0.3])
def test_select_matches_oracle(rows, n, topk, ties):
    g = torch.Generator(device=DEV).manual_seed(rows * 7 + n)
    scores = torch.randn(rows, n, generator=g, device=DEV)
    if ties:
        scores[torch.rand(rows, n, generator=g, device=DEV) < ties] = -0.75
    scores[0, :13] = float("nan")
    scores[1, :5] = float("-inf")
    scores[2, 10:20] = 0.0
    scores[2, 20:30] = -0.0
    lengths = torch.randint(0, n + 1, (rows,), generator=g, device=DEV, dtype=torch.int32)
    lengths[3] = n
    current = (torch.rand(rows, generator=g, device=DEV) * (lengths.float() + 1)).to(torch.int32) - 1
    got, ref = select_both(scores, current, topk, lengths)
    assert np.array_equal(got, ref)
    got, ref = select_both(scores, current, topk, None)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("topk", [1024, 2048])
def test_select_large_decode_rows(topk):
    sw = inputs.make_select_workload(DEV, topk=topk)
    got, ref = select_both(sw.scores, sw.current, sw.topk, sw.lengths)
    assert np.array_equal(got, ref)
    assert (got[:, 0] == sw.current.cpu().numpy()).all()


def test_select_then_sparse_decode():
    """Selection feeding the sparse path (8-token regions) equals the oracle chain."""
    cfg = inputs.scaled("fp8", requests=6, ctx=(3000, 9000), region_tokens=8, num_regions=64, gate=True)
    w = inputs.make_workload(cfg, DEV, fill="all")
    cur = (w.positions // 8).to(torch.int32)
    lengths = cur + 1
    scores = torch.randn(w.rows, int(lengths.max()), device=DEV)
    regions = sda.sparse_decode_select_regions(scores, cur, 64, topk_lengths=lengths)
    ref_regions = oracle.select_regions(scores.cpu(), cur.cpu(), 64, lengths.cpu())
    assert np.array_equal(regions.cpu().numpy(), ref_regions)
    w.regions = regions
    out, flags = run(w, splits=2)
    assert flags == 0
    rows = list(range(w.rows))
    check(w, out, oracle_rows(w, rows), rows)


# Bit patterns at every boundary of the float order the selection follows: denormals of both
# signs, both zeros, the infinities, NaN (both signs) and the largest finite values.
SPECIAL_BITS = [0x00000001, 0x00000002, 0x0000FFFF, 0x00010000, 0x007FFFFF, 0x00800000,
                0x80000001, 0x80000002, 0x8000FFFF, 0x80010000, 0x807FFFFF, 0x80800000,
                0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000,
                0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000, 0xBF800000]


@pytest.mark.parametrize("seed", range(8))
def test_select_special_floats(seed):
    """Rows longer than the shared-memory buffer, so the threshold comes from a sample, built
    from the special values above (some rows also from random denormal patterns of both signs);
    heavy ties on every value, so the lowest-id rule decides many slots."""
    rng = np.random.default_rng(900 + seed)
    rows, n = 12, int(rng.integers(4500, 30000))
    special = np.array(SPECIAL_BITS, dtype=np.uint32)
    bits = rng.choice(special, size=(rows, n), p=rng.dirichlet(np.full(len(special), 0.4)))
    denorm = rng.integers(1, 1 << 23, size=(rows, n), dtype=np.uint32) | \
        (rng.integers(0, 2, size=(rows, n), dtype=np.uint32) << 31)
    mix = (np.arange(rows) % 3 == 0)[:, None] & (rng.random((rows, n)) < 0.6)
    bits = np.where(mix, denorm, bits)
    sc = bits.view(np.float32)
    lens = rng.integers(n // 2, n + 1, size=rows).astype(np.int32)
    lens[0] = n
    cur = np.array([int(rng.integers(-1, l)) for l in lens], dtype=np.int32)
    t = lambda a: torch.as_tensor(a, device=DEV)
    for topk in (1, 97, 1024, 3000):
        got = sda.sparse_decode_select_regions(t(sc), t(cur), topk, topk_lengths=t(lens))
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), oracle.select_regions(sc, cur, topk, lens)), topk


def _keys(sc):
    """Order-preserving 32-bit keys of float32 scores (NaN lowest, -0 == +0)."""
    u = np.ascontiguousarray(sc, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = np.where((u & 0x7FFFFFFF) == 0, 0, u)
    k = np.where(u & 0x80000000, ~u & 0xFFFFFFFF, u | 0x80000000)
    return np.where(np.isnan(sc), 0, k).astype(np.uint64)


@pytest.mark.parametrize("case", ["spread", "ties", "wide"])
def test_select_threshold_in_buffer(case):
    """Rows long enough for the sampled bound, shaped so that the exact threshold among the
    buffered candidates is found each way the kernel has: by ranking the few keys that share
    the 16-bit prefix of rank topk (normal scores), by a radix select when more than 32 keys
    share it (scores on a 0.5 grid), and when that prefix lies 2047 or more prefixes above
    the bound's (log-normal scores over ~250 octaves)."""
    rng = np.random.default_rng({"spread": 11, "ties": 12, "wide": 13}[case])
    rows, n, topk = 6, 20000, 1024
    z = rng.standard_normal((rows, n))
    sc = {"spread": z, "ties": np.round(z * 2) / 2,
          "wide": np.exp(np.clip(z * 80 - 60, -87, 87))}[case]
    sc = sc.astype(np.float32)
    lens = np.full(rows, n, dtype=np.int32)
    cur = rng.integers(0, n, size=rows).astype(np.int32)
    for r in range(rows):                      # the branch each row reaches, from the keys alone
        keys = np.delete(_keys(sc[r]), cur[r])
        kth = np.sort(keys)[::-1][topk - 2]    # topk - 1 others besides the current region
        in_prefix = int(np.sum((keys >> 16) == (kth >> 16)))
        if case == "spread":
            assert in_prefix <= 32
        elif case == "ties":
            assert in_prefix > 32
        else:
            samp = np.sort(_keys(sc[r][(np.arange(2048) * n) // 2048]))[::-1]
            mu = np.float32(topk - 1) * 2048 / np.float32(n - 1)
            bound = samp[min(2048, int(mu + 5 * np.sqrt(mu)) + 17) - 1] >> 16
            assert (kth >> 16) - bound >= 2047
    t = lambda a: torch.as_tensor(a, device=DEV)
    got = sda.sparse_decode_select_regions(t(sc), t(cur), topk, topk_lengths=t(lens))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.select_regions(sc, cur, topk, lens))
