"""The seeded workload generators follow their stated recipe (no GPU).

Every parity test and every bench line is fed from inputs.py, so its recipe is
pinned here on small CPU builds of each workload (the properties do not depend
on the request count): context lengths in range, positions L - query_len + j,
a shuffled pool of exactly sum(ceil(L/B)) pages with each page used once,
region rows that hold distinct visible ids with the current region always in,
the -1 layout of each workload, the inactive fraction, the gate shape, the
FP8 scale (amax / 448), and determinism under the seed."""
import numpy as np
import pytest
import torch

from sparse_decode_attention_02_gb300 import inputs


def small(name, requests=8):
    cfg = inputs.CONFIGS[name]
    return inputs.scaled(cfg, requests=min(requests, cfg.requests))


@pytest.mark.parametrize("name", ["gqa", "fp8", "spec", "large", "swa"])
def test_positions_and_page_pool(name):
    cfg = small(name)
    w = inputs.make_workload(cfg, "cpu")
    L = w.seq_lens.numpy().astype(np.int64)
    assert ((L >= cfg.ctx[0]) & (L <= cfg.ctx[1])).all()
    ql, G = cfg.query_len, cfg.groups
    expect = np.repeat(np.concatenate([L[q] - ql + np.arange(ql) for q in range(cfg.requests)]), G)
    assert np.array_equal(w.positions.numpy(), expect)
    nblocks = -(-L // cfg.block)
    table = w.block_table.numpy()
    assert w.cache.shape[0] == nblocks.sum()                         # pool of exactly sum ceil(L/B)
    used = np.concatenate([table[q, :nblocks[q]] for q in range(cfg.requests)])
    assert np.array_equal(np.sort(used), np.arange(w.cache.shape[0]))  # each page once
    assert not np.array_equal(used, np.arange(len(used)))             # shuffled
    for q in range(cfg.requests):
        assert (table[q, nblocks[q]:] == -1).all()
    if cfg.gate:
        assert w.gate is not None and w.gate.shape == (cfg.tokens, G * cfg.heads)
        assert w.gate.dtype == torch.bfloat16
    else:
        assert w.gate is None


@pytest.mark.parametrize("name", ["gqa", "fp8", "spec", "large"])
def test_region_rows(name):
    cfg = small(name)
    w = inputs.make_workload(cfg, "cpu")
    reg, pos = w.regions.numpy(), w.positions.numpy()
    R, RT = cfg.num_regions, cfg.region_tokens
    assert reg.shape == (cfg.rows, R)
    short = 0
    for r in range(cfg.rows):
        live = reg[r][reg[r] >= 0]
        cur = pos[r] // RT
        assert cur in live                                            # current region always kept
        assert len(set(live.tolist())) == len(live)                   # distinct
        assert (live.astype(np.int64) * RT <= pos[r]).all()           # every id visible
        if cfg.pad_max:                                               # -1 at random slots
            assert R - cfg.pad_max <= len(live) <= R
        else:                                                         # -1 only at the tail
            assert (reg[r][:len(live)] >= 0).all() and (reg[r][len(live):] == -1).all()
        short += len(live) < R
        if cfg.selection == "recent_half":                            # half recent, half older
            recent = live[live >= max(0, cur - 511)]
            assert len(recent) == R // 2 and len(live) == R
        if len(live) >= 8:                                            # unsorted (a sorted shuffle
            assert not np.array_equal(live, np.sort(live))            # of 8 has odds 1/40320)
    if cfg.short_frac:
        assert short == int(round(cfg.short_frac * cfg.rows))
    elif not cfg.pad_max:
        assert short == 0


@pytest.mark.parametrize("name", ["fp8", "spec"])
def test_inactive_fraction(name):
    cfg = small(name, requests=64)
    w = inputs.make_workload(cfg, "cpu")
    assert int((w.active.numpy() == 0).sum()) == int(round(cfg.inactive_frac * cfg.rows))


def test_fp8_scales_map_amax_to_448():
    cfg = small("fp8", requests=2)
    w = inputs.make_workload(cfg, "cpu", fill="all")
    vals = w.cache.view(torch.float8_e4m3fn).float()
    assert not torch.isnan(vals).any()                                # saturated, never NaN
    assert float(vals[..., :192].abs().max()) == 448.0
    assert float(vals[..., 192:].abs().max()) == 448.0
    assert 0 < w.k_scale < 1 and 0 < w.v_scale < 1                   # N(0,1) amax over 448


def test_tiny_layout():
    w = inputs.make_workload("tiny", "cpu")
    pos = w.positions.numpy()
    assert ((pos >= 40) & (pos <= 500)).all()
    table = w.block_table.numpy()
    for q in range(table.shape[0]):                                   # each row a permutation of 32
        assert np.array_equal(np.sort(table[q]), np.arange(32))
    for r in range(w.rows):
        live = w.regions.numpy()[r]
        live = live[live >= 0]
        assert len(live) == min(4, pos[r] // 16 + 1)                  # -1 only when too few blocks


def test_seeded_and_deterministic():
    a = inputs.make_workload(small("spec", 4), "cpu")
    b = inputs.make_workload(small("spec", 4), "cpu")
    for name in ("query", "regions", "block_table", "positions", "active", "gate", "seq_lens"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert np.array_equal(a.filled_tiles, b.filled_tiles)
    t = torch.as_tensor(a.filled_tiles)
    assert torch.equal(a.cache[t[:, 0], t[:, 1]], b.cache[t[:, 0], t[:, 1]])


def test_window_workload_fills_exactly_the_windows():
    cfg = small("swa", 4)
    w = inputs.make_workload(cfg, "cpu")
    assert w.regions.shape == (cfg.rows, 0)
    table, pos = w.block_table.numpy(), w.positions.numpy()
    want = set()
    for r in range(cfg.rows):
        req, g = r // (cfg.groups * cfg.query_len), r % cfg.groups
        lo = max(0, int(pos[r]) - cfg.window + 1)
        for col in range(lo // cfg.block, int(pos[r]) // cfg.block + 1):
            want.add((int(table[req, col]), g))
    assert set(map(tuple, w.filled_tiles.tolist())) == want


def test_index_workload_recipe():
    iw = inputs.make_index_workload("cpu", requests=4, groups=2, query_len=2, ctx=(3000, 9000), block=64)
    L = iw.seq_lens.numpy().astype(np.int64)
    assert ((L >= 3000) & (L <= 9000)).all()
    nblocks = -(-L // 64)
    table = iw.block_table.numpy()
    used = np.concatenate([table[q, :nblocks[q]] for q in range(4)])
    assert len(np.unique(used)) == len(used)                          # each page once
    slots = iw.summaries.shape[0]
    assert slots == (nblocks.sum() + 64) * (64 // 8)                  # every pool page + 64 spare
    assert iw.query.shape == (8, 2, 8, 256) and iw.summaries.shape[1:] == (2, 256)
    w = iw.weights.numpy()
    assert w.shape == (8, 2, 8) and 0.03 < w.std() < 0.1              # N(0,1)/16
    q = iw.query.view(torch.float8_e4m3fn).float()
    assert not torch.isnan(q).any() and 1.5 < float(q.abs().max()) <= 448
