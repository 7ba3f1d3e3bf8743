"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Tolerance: max |gpu - oracle| <= 2e-2 (bf16 cache) / 5e-2 (FP8 cache) with
unit-variance V; inactive rows bit-exact +0.0; no NaN/Inf.  The five decode
workloads run at full size in the launch configuration the benchmark times;
the two largest are checked on sampled rows (the oracle computes them one by
one from host copies of exactly the pages they touch)."""
import gc

import numpy as np
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import check, oracle_all, oracle_rows, run, sample_rows, scales
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def mini(name, **changes):
    return inputs.make_workload(inputs.scaled(name, **changes), DEV, fill="all")


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def test_tiny_full():
    w = inputs.make_workload("tiny", DEV, fill="all")
    out, flags = run(w)
    assert flags == 0
    check(w, out, oracle_all(w))


@pytest.mark.parametrize("name", ["gqa", "fp8"])
def test_workload_all_rows(name):
    w = inputs.make_workload(name, DEV)
    out, flags = run(w)
    assert flags == 0
    rows = list(range(w.rows))
    check(w, out, oracle_rows(w, rows), rows)


@pytest.mark.parametrize("name,n", [("spec", 256), ("large", 64)])
def test_workload_sampled_rows(name, n):
    w = inputs.make_workload(name, DEV)
    out, flags = run(w)
    assert flags == 0
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(w, n)
    check(w, out, oracle_rows(w, rows), rows)


# ---------------------------------------------------------------------------
# Split-KV and the combine kernel
# ---------------------------------------------------------------------------

def test_split_counts_agree_with_oracle():
    w = mini("gqa", requests=12, ctx=(3000, 9000))
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    outs = {}
    for s in (1, 2, 3, 4, 8, 32, 64):
        out, flags = run(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)
        outs[s] = out.float()
    for s in outs:
        assert (outs[s] - outs[1]).abs().max().item() <= 2e-2


def test_split_partials_match_oracle():
    import oracle
    w = mini("gqa", requests=6, ctx=(2000, 7000))
    S = 3
    ws = torch.zeros(sda.workspace_bytes(w.rows, w.heads, S), dtype=torch.uint8, device=DEV)
    out, flags = run(w, splits=S, workspace=ws)
    assert flags == 0
    n = w.rows * S * w.heads
    part = ws[256:256 + n * 192 * 4].view(torch.float32).view(w.rows, S, w.heads, 192).cpu().numpy()
    lse = ws[256 + n * 192 * 4:256 + n * 192 * 4 + n * 4].view(torch.float32).view(w.rows, S, w.heads).cpu().numpy()
    hp = inputs.host_subset(w, range(w.rows))
    kw = dict(hp.kwargs)
    kw.pop("cache_fp8")
    rp, rl = oracle.split_partials(hp.query, hp.cache, hp.regions, hp.block_table, hp.positions,
                                   hp.active, splits=S, row_ids=hp.row_ids, cache_fp8=w.fp8, **kw)
    act = w.active.cpu().numpy().astype(bool)
    assert np.abs(part[act] - rp[act]).max() <= 2e-2
    fin = np.isfinite(rl[act])
    assert np.array_equal(fin, np.isfinite(lse[act]))
    assert np.abs(lse[act][fin] - rl[act][fin]).max() <= 1e-3


# ---------------------------------------------------------------------------
# Layout and shape variants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("changes", [
    dict(region_tokens=8, num_regions=96),                         # several regions per page
    dict(region_tokens=128, num_regions=16),                       # a region spans two pages
    dict(block=16, region_tokens=16, num_regions=40, heads=5),     # small pages, odd head count
    dict(heads=1, groups=1),
    dict(heads=8, groups=4, query_len=3),
    dict(num_regions=37, short_frac=0.5),                          # ragged region count
])
@pytest.mark.parametrize("fp8", [False, True])
def test_variants(changes, fp8):
    w = mini("gqa", requests=6, ctx=(1500, 6000), fp8=fp8, gate=True, inactive_frac=0.2, **changes)
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    for s in (1, 2):
        out, flags = run(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)


@pytest.mark.parametrize("changes", [
    dict(groups=8, heads=2),                                        # many KV groups, few heads
    dict(block=128, region_tokens=128, num_regions=12),             # a region = 2 FP8 / 4 bf16 pieces
    dict(block=32, region_tokens=64, num_regions=20, query_len=2),  # a region spans two blocks
    dict(block=64, region_tokens=16, num_regions=150, heads=12),    # four regions per page
    dict(block=24, region_tokens=24, num_regions=40),               # pieces that do not divide a stage
])
@pytest.mark.parametrize("fp8", [False, True])
def test_more_layouts(changes, fp8):
    w = mini("gqa", requests=4, ctx=(2000, 6000), fp8=fp8, gate=True, inactive_frac=0.1, **changes)
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    for s in (1, 3):
        out, flags = run(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)


def test_fp8_pages_of_48_tokens():
    """One 48-token piece per 64-slot FP8 stage."""
    w = mini("fp8", requests=4, ctx=(2000, 6000), block=48, region_tokens=48, num_regions=24)
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    for s in (1, 2):
        out, flags = run(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)


def test_region_slots_at_the_limit():
    """16,384 region slots per row (the most the entry point takes): every visible 8-token
    region selected, the rest -1; one slot more is refused."""
    w = mini("gqa", requests=2, ctx=(9000, 12000), region_tokens=8, num_regions=16384, fp8=True)
    rows = list(range(w.rows))
    out, flags = run(w, splits=1)
    assert flags == 0
    check(w, out, oracle_rows(w, rows), rows)
    wide = torch.full((w.rows, 16385), -1, dtype=torch.int32, device=DEV)
    wide[:, :16384] = w.regions
    w.regions = wide
    with pytest.raises(sda.SdaError) as e:
        run(w, splits=1)
    assert e.value.status == 2                        # SDA_ERR_UNSUPPORTED


def test_many_regions_per_row():
    w = mini("gqa", requests=3, ctx=(9000, 12000), region_tokens=8, num_regions=1024, fp8=True)
    rows = list(range(w.rows))
    out, flags = run(w, splits=1)
    assert flags == 0
    check(w, out, oracle_rows(w, rows), rows)


@pytest.mark.parametrize("fp8", [False, True])
def test_padded_page_stride(fp8):
    w = inputs.make_workload(inputs.scaled("gqa", requests=5, ctx=(1000, 5000), fp8=fp8), DEV,
                             fill="all", page_stride_pad=64)
    assert w.cache.stride(0) != w.cache.shape[1] * w.cache.shape[2] * 384
    rows = list(range(w.rows))
    out, flags = run(w)
    assert flags == 0
    check(w, out, oracle_rows(w, rows), rows)


def test_strided_query_output_gate():
    w = mini("gqa", requests=4, ctx=(1000, 4000), gate=True)
    H = w.heads
    qbig = torch.zeros(w.rows, H + 3, 192, dtype=torch.bfloat16, device=DEV)
    qbig[:, 2:H + 2] = w.query
    w.query = qbig[:, 2:H + 2]
    gbig = torch.zeros(w.gate.shape[0], w.gate.shape[1] * 2, dtype=torch.bfloat16, device=DEV)
    gbig[:, ::2] = w.gate
    w.gate = gbig[:, ::2]
    obig = torch.full((w.rows, H + 1, 192), 3.0, dtype=torch.bfloat16, device=DEV)
    out = obig[:, 1:]
    run(w, out=out)
    rows = list(range(w.rows))
    check(w, out, oracle_rows(w, rows), rows)
    assert (obig[:, 0] == 3.0).all()


def test_fp8_cache_as_uint8_or_e4m3():
    w = mini("fp8", requests=4, ctx=(1000, 4000))
    a, _ = run(w)
    b, _ = run(w, cache=w.cache.view(torch.float8_e4m3fn))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------------------
# Edge cases and the method's degenerate cases
# ---------------------------------------------------------------------------

def test_zero_rows_is_a_no_op():
    w = mini("gqa", requests=2, ctx=(500, 900))
    q = w.query[:0]
    out = torch.empty_like(q)
    sda.sparse_decode_attention(q, w.cache, w.regions[:0], w.block_table, w.positions[:0],
                                w.active[:0], out, scale=w.scale, splits=1)
    torch.cuda.synchronize()


def test_single_visible_token_returns_v_exactly():
    w = mini("gqa", requests=4, ctx=(1000, 3000))
    pos = w.positions.clone()
    regions = torch.full_like(w.regions, -1)
    RT = w.region_tokens
    cur = pos // RT
    pos = (cur * RT).to(torch.int32)
    regions[:, 5] = cur.to(torch.int32)
    w.positions, w.regions = pos, regions
    out, flags = run(w, splits=1)
    assert flags == 0
    # expected: V row of token cur*RT for every head, exactly (bf16 in, bf16 out)
    G, ql, B = w.groups, w.query_len, w.block
    for r in range(w.rows):
        req, g = r // (G * ql), r % G
        t = int(pos[r])
        page = int(w.block_table[req, t // B])
        v = w.cache[page, g, t % B, 192:]
        assert torch.equal(out[r].view(torch.int16), v.expand(w.heads, 192).contiguous().view(torch.int16))


def test_rows_without_visible_tokens_are_zero():
    w = mini("gqa", requests=4, ctx=(1000, 3000), gate=True)
    w.regions[0] = -1
    w.regions[1] = -1
    w.regions[1, 3] = int(w.positions[1]) // w.region_tokens + 2      # starts past the position
    w.positions[2] = -1
    for s in (1, 4):
        out, flags = run(w, splits=s)
        assert flags == 0
        assert (out[:3].view(torch.int16) == 0).all()


@pytest.mark.parametrize("splits", [1, 2])
def test_clear_inactive_false_leaves_rows(splits):
    w = mini("gqa", requests=4, ctx=(1000, 3000), inactive_frac=0.25)
    out = torch.full_like(w.query, 7.0)
    out, _ = run(w, splits=splits, out=out, clear_inactive=False)
    act = w.active.bool()
    assert (out[~act] == 7.0).all()
    rows = torch.nonzero(act).flatten().tolist()
    ref = oracle_rows(w, rows)
    assert np.abs(out[act].float().cpu().numpy() - ref).max() <= 2e-2


def test_garbage_past_position_is_ignored():
    """Slots of the current block past the position may hold anything (NaN here)."""
    w = mini("gqa", requests=6, ctx=(1000, 5000))
    G, B = w.groups, w.block
    for r in range(w.rows):
        req, g = r // G, r % G
        pos = int(w.positions[r])
        page = int(w.block_table[req, pos // B])
        w.cache[page, g, pos % B + 1:] = float("nan")
    rows = list(range(w.rows))
    for s in (1, 3):
        out, flags = run(w, splits=s)
        assert flags == 0
        check(w, out, oracle_rows(w, rows), rows)


def test_region_order_and_padding_invariance():
    w = mini("gqa", requests=4, ctx=(1000, 3000), fp8=True)
    a, _ = run(w, splits=1)
    perm = torch.stack([torch.randperm(w.regions.shape[1], device=DEV) for _ in range(w.rows)])
    reg = torch.gather(w.regions, 1, perm)
    w.regions = torch.cat([torch.full((w.rows, 5), -1, dtype=torch.int32, device=DEV), reg], 1).contiguous()
    b, _ = run(w, splits=1)
    assert (a.float() - b.float()).abs().max().item() <= 1e-2


def test_bad_indices_are_flagged_not_faulted():
    w = mini("gqa", requests=4, ctx=(1000, 3000))
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    w.regions[1, 0] = -5
    out, flags = run(w, splits=1)
    assert flags & sda.FLAG_BOUNDS
    keep = [r for r in rows if r != 1]
    check(w, out, ref[keep], keep)
    w2 = mini("gqa", requests=4, ctx=(1000, 3000))
    r0 = int(w2.positions[0]) // w2.block
    w2.block_table[0, r0] = w2.cache.shape[0] + 5
    out, flags = run(w2, splits=2)
    assert flags & sda.FLAG_BOUNDS
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("splits", [1, 2])
def test_fp8_query_of_any_bf16_magnitude(splits):
    """The FP8 path multiplies in fp16, whose range bf16 queries exceed: rows whose q sits
    around 1e5 (past fp16's 65504), around 1e-6 (below fp16's normal range), or mixes 3e4
    with 1e-3 inside one head must still match the oracle, with no NaN or Inf."""
    w = mini("fp8", requests=6, ctx=(2000, 6000), gate=True)
    q = w.query.float()
    q[0::4] *= 1e5
    q[1::4] *= 1e-6
    q[2::4, :, :96] *= 3e4
    q[2::4, :, 96:] *= 1e-3
    w.query.copy_(q.to(torch.bfloat16))
    assert w.query[0::4].float().abs().max().item() > 65504
    out, flags = run(w, splits=splits)
    assert flags == 0
    rows = list(range(w.rows))
    check(w, out, oracle_rows(w, rows), rows)


def test_deterministic_and_graph_capturable():
    w = mini("fp8", requests=8, ctx=(2000, 6000))
    S = sda.sparse_decode_splits(w.rows)
    ws = torch.zeros(sda.workspace_bytes(w.rows, w.heads, S), dtype=torch.uint8, device=DEV)
    ks, vs = scales(w)
    eager = torch.empty_like(w.query)
    args = (w.query, w.cache, w.regions, w.block_table, w.positions, w.active)
    kw = dict(scale=w.scale, splits=S, k_scale=ks, v_scale=vs, gate=w.gate, workspace=ws)
    sda.sparse_decode_attention(*args, eager, **kw)
    again = torch.empty_like(w.query)
    sda.sparse_decode_attention(*args, again, **kw)
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), again.view(torch.int16))
    out = torch.empty_like(w.query)
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sda.sparse_decode_attention(*args, out, **kw)      # warm-up on the capture stream
        stream.synchronize()
        out.zero_()
        with torch.cuda.graph(g, stream=stream):
            sda.sparse_decode_attention(*args, out, **kw, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert sda.read_errors(ws) == 0


def test_default_workspaces_are_per_stream():
    """Split calls on two streams at once, without explicit workspaces: each stream's
    default workspace is its own, so the partials do not race."""
    w = mini("gqa", requests=8, ctx=(4000, 9000))
    rows = list(range(w.rows))
    ref = oracle_rows(w, rows)
    ks, vs = scales(w)
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    outs = [torch.full_like(w.query, float("nan")) for _ in streams]
    torch.cuda.synchronize()
    for _ in range(20):
        for s, o in zip(streams, outs):
            with torch.cuda.stream(s):
                sda.sparse_decode_attention(w.query, w.cache, w.regions, w.block_table, w.positions, w.active, o,
                                            scale=w.scale, splits=4, k_scale=ks, v_scale=vs, gate=w.gate,
                                            region_tokens=w.region_tokens, stream=s)
    torch.cuda.synchronize()
    for o in outs:
        check(w, o, ref, rows)
