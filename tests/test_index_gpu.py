"""Indexer decode scores (CUDA kernel vs the oracle), and the whole decode chain
scores -> region selection -> sparse attention.

Tolerance.  Both sides decode the same E4M3 bytes exactly; each product of two
E4M3 values is exact in fp32.  The GPU accumulates the 256-term dot products in
fp32 (the MMA's adds may truncate: at most 2^-23 relative each), then weights
and sums 8 heads in fp32, so |gpu - oracle| <= (256 + 8) * 2^-23 * A with
A = sum_h |w_h| sum_d |q_hd| |m_jd|.  The tests use TOL_REL = 4e-5 >= 264 *
2^-23 of A, with A computed by the oracle on the absolute values (clearing the
E4M3 sign bits and taking |w|).  The -inf pattern, `current` and `lengths` are
compared exactly."""
import gc

import numpy as np
import pytest
import torch

import oracle
import sparse_decode_attention_02_gb300 as sda
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL_REL = 4e-5


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def run_gpu(w, *, query=None, weights=None, table=None, workspace=None, n_cols=None):
    n_cols = w.n_cols if n_cols is None else n_cols
    scores = torch.full((w.rows, n_cols), float("nan"), device=DEV)
    cur = torch.full((w.rows,), -7, dtype=torch.int32, device=DEV)
    lens = torch.full((w.rows,), -7, dtype=torch.int32, device=DEV)
    sda.sparse_decode_summary_scores(w.query if query is None else query,
                                     w.weights if weights is None else weights, w.summaries,
                                     w.block_table if table is None else table, w.seq_lens,
                                     block_size=w.block, query_len=w.query_len, scores=scores,
                                     current=cur, lengths=lens, workspace=workspace)
    torch.cuda.synchronize()
    return scores.cpu().numpy(), cur.cpu().numpy(), lens.cpu().numpy()


def run_oracle(h, *, n_cols=None, absolute=False):
    """The oracle on host workload `h`; with `absolute`, on |q|, |w|, |m| (the error scale)."""
    q, w, m = h.query.view(torch.uint8), h.weights, h.summaries.view(torch.uint8)
    if absolute:
        q, w, m = q & 0x7F, w.abs(), m & 0x7F
    return oracle.summary_scores(q, w, m, h.block_table, h.seq_lens, block=h.block,
                                 n_cols=h.n_cols if n_cols is None else n_cols, query_len=h.query_len)


def host(w):
    return inputs.IndexWorkload(w.query.cpu(), w.weights.cpu(), w.summaries.cpu(), w.block_table.cpu(),
                                w.seq_lens.cpu(), w.block, w.query_len, w.n_cols)


def check(got, ref, scale):
    gs, gc_, gl = got
    rs, rc, rl = ref
    assert np.array_equal(gc_, rc) and np.array_equal(gl, rl)
    assert not np.isnan(gs).any()
    assert np.array_equal(np.isneginf(gs), np.isneginf(rs))
    fin = np.isfinite(rs)
    assert np.isfinite(gs[fin]).all()
    err = np.abs(gs[fin] - rs[fin])
    bound = TOL_REL * scale[fin] + 1e-6
    assert (err <= bound).all(), float(np.max(err / bound))


CASES = {
    "block8_g1": dict(requests=3, groups=1, query_len=1, ctx=(1, 700), block=8),
    "chunks_g2_ql2": dict(requests=5, groups=2, query_len=2, ctx=(100, 9000), block=16),
    "g4_ql1": dict(requests=4, groups=4, query_len=1, ctx=(4000, 20000), block=64),
    "g8_ql3_capped": dict(requests=3, groups=8, query_len=3, ctx=(10, 5000), block=64, n_cols=300),
    "short_ql4": dict(requests=4, groups=2, query_len=4, ctx=(1, 3), block=16),
    "g4_ql4_long": dict(requests=2, groups=4, query_len=4, ctx=(30000, 40000), block=32),
    "g2_ql1_ragged": dict(requests=7, groups=2, query_len=1, ctx=(511 * 8, 513 * 8 + 7), block=64),
    "g3_ql2": dict(requests=3, groups=3, query_len=2, ctx=(700, 6000), block=32),
    "g6_ql1": dict(requests=3, groups=6, query_len=1, ctx=(3000, 9000), block=64),
    # pages of 64 tokens or more take the tensor-core variant (128-region tiles)
    "tc_block128_g2_ql2": dict(requests=3, groups=2, query_len=2, ctx=(5000, 20000), block=128),
    "tc_block2048_g1_ql3": dict(requests=2, groups=1, query_len=3, ctx=(9000, 40000), block=2048),
    "tc_block64_g4_ql4": dict(requests=3, groups=4, query_len=4, ctx=(20000, 40000), block=64),
    "tc_block64_g1_ql3_short": dict(requests=5, groups=1, query_len=3, ctx=(1, 200), block=64),
    "tc_block64_g2_ql1_capped": dict(requests=3, groups=2, query_len=1, ctx=(3000, 30000), block=64,
                                     n_cols=2500),
    # one group per block (N = 16 with 8 padding rows at query_len 1, 32 with 8 at query_len 3)
    "tc_block64_g3_ql1": dict(requests=4, groups=3, query_len=1, ctx=(2000, 12000), block=64),
    "tc_block64_g5_ql3": dict(requests=3, groups=5, query_len=3, ctx=(500, 9000), block=64),
    "tc_block256_g2_ql4_short": dict(requests=6, groups=2, query_len=4, ctx=(1, 2100), block=256),
}


@pytest.mark.parametrize("name", list(CASES))
def test_summary_scores_match_oracle(name):
    w = inputs.make_index_workload(DEV, seed=11, **CASES[name])
    h = host(w)
    got = run_gpu(w)
    check(got, run_oracle(h), run_oracle(h, absolute=True)[0])


def test_group_major_strides():
    """Indexer outputs may be group-major: queries and weights as [G, tokens] views."""
    w = inputs.make_index_workload(DEV, requests=4, groups=4, query_len=2, ctx=(900, 4000), block=64, seed=5)
    qg = w.query.permute(1, 0, 2, 3).contiguous().permute(1, 0, 2, 3)
    wg = w.weights.permute(1, 0, 2).contiguous().permute(1, 0, 2)
    assert qg.stride(1) > qg.stride(0) and wg.stride(1) > wg.stride(0)
    h = host(w)
    check(run_gpu(w, query=qg, weights=wg), run_oracle(h), run_oracle(h, absolute=True)[0])


def test_bad_page_flags_and_scores_minus_inf():
    w = inputs.make_index_workload(DEV, requests=3, groups=2, query_len=1, ctx=(2000, 3000), block=16, seed=9)
    h = host(w)
    ref = run_oracle(h)
    scale = run_oracle(h, absolute=True)[0]
    bad = w.block_table.clone()
    bad[1, 3] = w.summaries.shape[0] // 2          # page ids start past the summary buffer
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    got = run_gpu(w, table=bad, workspace=ws)
    assert sda.read_errors(ws) & sda.FLAG_BOUNDS
    rows = [2, 3]                                   # request 1's rows (G = 2)
    cols = slice(3 * 2, 4 * 2)                      # column 3 of 16-token pages = regions 6, 7
    assert np.all(got[0][rows, cols] == -np.inf)
    keep = np.ones_like(ref[0], dtype=bool)
    keep[rows, cols] = False
    gs = np.where(keep, got[0], ref[0])
    check((gs, got[1], got[2]), ref, scale)
    ws.zero_()
    run_gpu(w, workspace=ws)
    assert sda.read_errors(ws) == 0


def test_bad_page_tensor_core_path():
    """A page id past the summaries on the 128-region-tile path (64-token pages): flagged, and
    exactly that page's regions score -inf."""
    w = inputs.make_index_workload(DEV, requests=3, groups=2, query_len=2, ctx=(6000, 9000), block=64, seed=19)
    h = host(w)
    ref = run_oracle(h)
    scale = run_oracle(h, absolute=True)[0]
    bad = w.block_table.clone()
    bad[2, 5] = w.summaries.shape[0]                # past the last page (8 slots per page)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    got = run_gpu(w, table=bad, workspace=ws)
    assert sda.read_errors(ws) & sda.FLAG_BOUNDS
    rows = list(range(2 * 2 * 2, 3 * 2 * 2))        # request 2's rows (query_len 2, G = 2)
    cols = slice(5 * 8, 6 * 8)                      # column 5 of 64-token pages = regions 40..47
    assert np.all(got[0][rows, cols] == -np.inf)
    keep = np.ones_like(ref[0], dtype=bool)
    keep[rows, cols] = False
    gs = np.where(keep, got[0], ref[0])
    check((gs, got[1], got[2]), ref, scale)


def test_wait_timeout_is_flagged_and_recoverable():
    """The tensor-core path's pipeline waits honour the process-wide limit: at 0 they run
    out, the kernel flags SDA_FLAG_TIMEOUT, lets its copies and MMAs finish, releases its
    tensor memory and returns; the next call with the normal limit is correct."""
    w = inputs.make_index_workload(DEV, requests=4, groups=4, query_len=2, ctx=(20000, 30000), block=64, seed=23)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    sda.set_wait_limit_ns(0)
    try:
        run_gpu(w, workspace=ws)
    finally:
        sda.set_wait_limit_ns(10 ** 9)
    assert sda.read_errors(ws, clear=True) & sda.FLAG_TIMEOUT
    h = host(w)
    got = run_gpu(w, workspace=ws)
    assert sda.read_errors(ws) == 0
    check(got, run_oracle(h), run_oracle(h, absolute=True)[0])


def test_no_columns_still_writes_current_and_lengths():
    w = inputs.make_index_workload(DEV, requests=2, groups=2, query_len=2, ctx=(50, 90), block=16, seed=1)
    s, c, l = run_gpu(w, n_cols=0)
    _, rc, rl = run_oracle(host(w), n_cols=0)
    assert s.shape == (w.rows, 0) and np.array_equal(c, rc) and np.array_equal(l, rl)


def test_full_size_sampled_rows():
    """The decode-row workload at full size (512 requests x 4 groups, contexts
    128K-256K, 32K columns): sampled requests against the oracle, and the
    -inf / current / lengths pattern of every row."""
    w = inputs.make_index_workload(DEV)
    got = run_gpu(w)
    seq = w.seq_lens.cpu().numpy().astype(np.int64)
    pos = np.repeat(seq - 1, w.groups)
    n = np.minimum(pos // 8 + 1, w.n_cols)
    assert np.array_equal(got[1], pos // 8) and np.array_equal(got[2], n)
    cols = np.arange(w.n_cols)
    assert np.array_equal(np.isneginf(got[0]), cols[None, :] >= n[:, None])
    assert np.isfinite(got[0][cols[None, :] < n[:, None]]).all()
    reqs = [0, 217, 511]
    sub = inputs.index_host_subset(w, reqs)
    rows = [r * w.groups + g for r in reqs for g in range(w.groups)]
    check(tuple(x[rows] for x in got), run_oracle(sub), run_oracle(sub, absolute=True)[0])


def test_decode_chain_scores_select_attention():
    """scores -> select_regions -> sparse_decode_attention with 8-token regions,
    every step on the GPU; each step checked against the oracle on the previous
    step's GPU output (scores within tolerance, ids exactly, attention within
    the bf16 tolerance)."""
    w = inputs.make_index_workload(DEV, requests=6, groups=2, query_len=2, ctx=(3000, 12000), block=64, seed=4)
    h = host(w)
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    scores = torch.empty((w.rows, w.n_cols), device=DEV)
    cur = torch.empty(w.rows, dtype=torch.int32, device=DEV)
    lens = torch.empty(w.rows, dtype=torch.int32, device=DEV)
    sda.sparse_decode_summary_scores(w.query, w.weights, w.summaries, w.block_table, w.seq_lens,
                                     block_size=w.block, query_len=w.query_len, scores=scores,
                                     current=cur, lengths=lens, workspace=ws)
    topk = 64
    regions = sda.sparse_decode_select_regions(scores, cur, topk, topk_lengths=lens)
    g = torch.Generator(device=DEV).manual_seed(3)
    pages = w.summaries.shape[0] // (w.block // 8)
    cache = torch.randn((pages, w.groups, w.block, 384), generator=g, device=DEV).to(torch.bfloat16)
    query = torch.randn((w.rows, 16, 192), generator=g, device=DEV).to(torch.bfloat16)
    seq = w.seq_lens.long()
    tok = torch.arange(w.tokens, device=DEV)
    positions = (seq[tok // w.query_len] - w.query_len + tok % w.query_len).repeat_interleave(w.groups)
    positions = positions.to(torch.int32)
    active = torch.ones(w.rows, dtype=torch.bool, device=DEV)
    out = torch.empty_like(query)
    sda.sparse_decode_attention(query, cache, regions, w.block_table, positions, active, out,
                                scale=192 ** -0.5, query_len=w.query_len, region_tokens=8)
    torch.cuda.synchronize()
    assert sda.read_errors(ws) == 0
    check((scores.cpu().numpy(), cur.cpu().numpy(), lens.cpu().numpy()), run_oracle(h),
          run_oracle(h, absolute=True)[0])
    ref_ids = oracle.select_regions(scores.cpu(), cur.cpu(), topk, lens.cpu())
    assert np.array_equal(regions.cpu().numpy(), ref_ids)
    ref = oracle.sparse_decode_attention(query.cpu(), cache.cpu(), regions.cpu(), w.block_table.cpu(),
                                         positions.cpu(), active.cpu(), scale=192 ** -0.5,
                                         query_len=w.query_len, region_tokens=8)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= 2e-2, err


@pytest.mark.parametrize("query_len", [1, 2])    # 2: speculative decode, two tokens per request
def test_decode_chain_full_size_sampled(query_len):
    """The whole decode step at full size (512 requests x 4 groups, contexts
    128K-256K, top-1024 of 8-token regions, FP8 cache) in the launch
    configuration the benchmark times; sampled requests checked step by step."""
    ch = inputs.make_decode_chain(DEV, query_len=query_len)
    iw = ch.index
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    scores = torch.empty((iw.rows, iw.n_cols), device=DEV)
    cur = torch.empty(iw.rows, dtype=torch.int32, device=DEV)
    lens = torch.empty(iw.rows, dtype=torch.int32, device=DEV)
    sda.sparse_decode_summary_scores(iw.query, iw.weights, iw.summaries, iw.block_table, iw.seq_lens,
                                     block_size=iw.block, query_len=iw.query_len, scores=scores,
                                     current=cur, lengths=lens, workspace=ws)
    regions = sda.sparse_decode_select_regions(scores, cur, ch.topk, topk_lengths=lens)
    out = torch.empty_like(ch.query)
    ks = torch.tensor([ch.k_scale], device=DEV)
    vs = torch.tensor([ch.v_scale], device=DEV)
    sda.sparse_decode_attention(ch.query, ch.cache, regions, iw.block_table, ch.positions, ch.active, out,
                                scale=ch.scale, query_len=iw.query_len, splits=1, k_scale=ks, v_scale=vs,
                                region_tokens=8, workspace=ws)
    torch.cuda.synchronize()
    assert sda.read_errors(ws) == 0
    reqs = [5, 300]
    ql, G = iw.query_len, iw.groups
    rows = [(r * ql + t) * G + g for r in reqs for t in range(ql) for g in range(G)]
    sub = inputs.index_host_subset(iw, reqs)
    check((scores[rows].cpu().numpy(), cur[rows].cpu().numpy(), lens[rows].cpu().numpy()),
          run_oracle(sub), run_oracle(sub, absolute=True)[0])
    sel = regions[rows].cpu().numpy()
    assert np.array_equal(sel, oracle.select_regions(scores[rows].cpu(), cur[rows].cpu(), ch.topk,
                                                     lens[rows].cpu()))
    assert (sel >= 0).all()                          # every row has > 1024 regions to choose from
    # attention of the sampled rows over their own selected regions, on the requests' pages
    table = iw.block_table.cpu().numpy()
    used = sorted({int(p) for r in reqs for p in table[r] if p >= 0})
    remap = np.full(int(table.max()) + 1, -1, np.int64)
    remap[used] = np.arange(len(used))
    sub_table = np.where(table[reqs] >= 0, remap[np.maximum(table[reqs], 0)], -1).astype(np.int32)
    cache = ch.cache[torch.as_tensor(used, device=DEV)].cpu()
    ref = oracle.sparse_decode_attention(ch.query[rows].cpu(), cache, regions[rows].cpu(), sub_table,
                                         ch.positions[rows].cpu(), ch.active[rows].cpu(), scale=ch.scale,
                                         query_len=iw.query_len, region_tokens=8, k_scale=ch.k_scale,
                                         v_scale=ch.v_scale, cache_fp8=True)
    err = np.abs(out[rows].float().cpu().numpy() - ref).max()
    assert err <= 5e-2, err


def test_padded_summary_slots():
    """Summary slots with a padded stride (the slot's G x 256 bytes followed by 64 unused)."""
    w = inputs.make_index_workload(DEV, requests=4, groups=2, query_len=1, ctx=(900, 5000), block=32, seed=12)
    slots = w.summaries.shape[0]
    big = torch.zeros((slots, w.groups * 256 + 64), dtype=torch.uint8, device=DEV)
    big[:, :w.groups * 256] = w.summaries.view(torch.uint8).reshape(slots, -1)
    big[:, w.groups * 256:] = 0x7F                              # NaN codes in the padding
    padded = big[:, :w.groups * 256].view(slots, w.groups, 256)
    assert padded.stride(0) == w.groups * 256 + 64
    h = host(w)
    w.summaries = padded
    check(run_gpu(w), run_oracle(h), run_oracle(h, absolute=True)[0])


def test_padded_summary_slots_tensor_core_path():
    """The same padded slot stride on the 128-region-tile path (64-token pages)."""
    w = inputs.make_index_workload(DEV, requests=3, groups=4, query_len=3, ctx=(9000, 15000), block=64, seed=13)
    slots = w.summaries.shape[0]
    big = torch.zeros((slots, w.groups * 256 + 64), dtype=torch.uint8, device=DEV)
    big[:, :w.groups * 256] = w.summaries.view(torch.uint8).reshape(slots, -1)
    big[:, w.groups * 256:] = 0x7F                              # NaN codes in the padding
    padded = big[:, :w.groups * 256].view(slots, w.groups, 256)
    h = host(w)
    w.summaries = padded
    check(run_gpu(w), run_oracle(h), run_oracle(h, absolute=True)[0])


def _chain_step(w, cache, query, positions, active, topk, bufs, stream):
    """One decode step (scores -> selection -> attention) into the tensors of `bufs`."""
    scores, cur, lens, regions, out, ws = bufs
    sda.sparse_decode_summary_scores(w.query, w.weights, w.summaries, w.block_table, w.seq_lens,
                                     block_size=w.block, query_len=w.query_len, scores=scores,
                                     current=cur, lengths=lens, workspace=ws, stream=stream)
    sda.sparse_decode_select_regions(scores, cur, topk, regions, topk_lengths=lens, stream=stream)
    sda.sparse_decode_attention(query, cache, regions, w.block_table, positions, active, out,
                                scale=192 ** -0.5, query_len=w.query_len, splits=2, region_tokens=8,
                                workspace=ws, stream=stream)


def _chain_inputs(w, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    pages = w.summaries.shape[0] // (w.block // 8)
    cache = torch.randn((pages, w.groups, w.block, 384), generator=g, device=DEV).to(torch.bfloat16)
    query = torch.randn((w.rows, 16, 192), generator=g, device=DEV).to(torch.bfloat16)
    seq = w.seq_lens.long()
    tok = torch.arange(w.tokens, device=DEV)
    positions = (seq[tok // w.query_len] - w.query_len + tok % w.query_len).repeat_interleave(w.groups)
    return cache, query, positions.to(torch.int32), torch.ones(w.rows, dtype=torch.bool, device=DEV)


def _chain_bufs(w, topk):
    return (torch.full((w.rows, w.n_cols), float("nan"), device=DEV),
            torch.full((w.rows,), -7, dtype=torch.int32, device=DEV),
            torch.full((w.rows,), -7, dtype=torch.int32, device=DEV),
            torch.full((w.rows, topk), -7, dtype=torch.int32, device=DEV),
            torch.full((w.rows, 16, 192), float("nan"), dtype=torch.bfloat16, device=DEV),
            torch.zeros(sda.workspace_bytes(w.rows, 16, 2), dtype=torch.uint8, device=DEV))


def _same(a, b):
    return all(torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else
                           x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
               for x, y in zip(a[:5], b[:5]))


def test_decode_chain_graph_replay_matches_eager():
    """The whole decode step (tensor-core indexer, selection, split attention + combine)
    captured in one CUDA graph: its replays write the eager step's bits (scores, metadata,
    ids, output), so no kernel of the chain depends on host state or on a previous call."""
    w = inputs.make_index_workload(DEV, requests=5, groups=4, query_len=2, ctx=(9000, 30000), block=64, seed=21)
    cache, query, positions, active = _chain_inputs(w, 22)
    topk = 256
    eager = _chain_bufs(w, topk)
    _chain_step(w, cache, query, positions, active, topk, eager, torch.cuda.current_stream())
    torch.cuda.synchronize()
    graphed = _chain_bufs(w, topk)
    stream = torch.cuda.Stream(DEV)
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        _chain_step(w, cache, query, positions, active, topk, graphed, stream)   # warm-up
        stream.synchronize()
        for t in graphed[:5]:
            t.fill_(0)
        with torch.cuda.graph(g, stream=stream):
            _chain_step(w, cache, query, positions, active, topk, graphed, stream)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert _same(graphed, eager)
    assert sda.read_errors(eager[5]) == 0 and sda.read_errors(graphed[5]) == 0
    ids = graphed[3].cpu().numpy()
    assert np.array_equal(ids, oracle.select_regions(eager[0].cpu(), eager[1].cpu(), topk, eager[2].cpu()))


def test_decode_chains_on_two_streams_at_once():
    """Two decode steps on different inputs, interleaved on two streams with their own
    buffers: each stream's results equal its step run alone (the library keeps no state
    between calls that two streams could share)."""
    ws_ = [inputs.make_index_workload(DEV, requests=4, groups=4, query_len=q, ctx=(6000, 20000), block=64,
                                      seed=31 + q) for q in (1, 2)]
    ins = [_chain_inputs(w, 40 + i) for i, w in enumerate(ws_)]
    topk = 128
    alone = []
    for w, (cache, query, pos, act) in zip(ws_, ins):
        b = _chain_bufs(w, topk)
        _chain_step(w, cache, query, pos, act, topk, b, torch.cuda.current_stream())
        torch.cuda.synchronize()
        alone.append(b)
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    bufs = [_chain_bufs(w, topk) for w in ws_]
    torch.cuda.synchronize()
    for _ in range(10):
        for w, (cache, query, pos, act), b, s in zip(ws_, ins, bufs, streams):
            _chain_step(w, cache, query, pos, act, topk, b, s)
    torch.cuda.synchronize()
    for b, a in zip(bufs, alone):
        assert _same(b, a)
        assert sda.read_errors(b[5]) == 0
