"""The allocation-free entry point against the regular one (GPU).

sparse_decode_attention_no_alloc serves callers that cannot allocate device
memory: plugin or FFI hosts handed tensor pointers but no allocator, and code
that must not call cudaMalloc while other work is in flight.  Its split-KV
scratch is a static 8 MiB device array inside the library.  Two calls in a
row, on different workloads and split counts, must each match the regular
entry point (caller-supplied workspace) within the parity tolerance, also
when a call with more rows and splits has left its partials in the array; a
call whose scratch would not fit is refused before anything is enqueued,
arguments outside the contract get the regular entry point's statuses, and
device flags collect in the array until read.  Collected last so a failure
here cannot hide failures of the other tests.
"""
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import TOL_BF16, TOL_FP8, check, oracle_all, run, scales
from sparse_decode_attention_02_gb300 import _binding as B
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def no_alloc(w, splits, **kw):
    out = torch.full_like(w.query, float("nan"))
    ks, vs = scales(w)
    B.sparse_decode_attention_no_alloc(w.query, w.cache, w.regions, w.block_table, w.positions,
                                       w.active, out, scale=w.scale, query_len=w.query_len,
                                       splits=splits, k_scale=ks, v_scale=vs, gate=w.gate,
                                       region_tokens=w.region_tokens, **kw)
    torch.cuda.synchronize()
    return out


def test_no_alloc_matches_regular_entry_point_twice():
    sda.no_alloc_read_errors(clear=True)
    cases = [
        (inputs.scaled("gqa", requests=16, ctx=(3000, 9000), inactive_frac=0.1, gate=True), 4),
        (inputs.scaled("fp8", requests=8, ctx=(2000, 6000)), 2),
        (inputs.scaled("gqa", requests=6, ctx=(1000, 4000)), 1),
    ]
    for cfg, splits in cases:
        w = inputs.make_workload(cfg, DEV, fill="all")
        first = no_alloc(w, splits)
        second = no_alloc(w, splits)
        ref, flags = run(w, splits=splits)
        assert flags == 0
        tol = TOL_FP8 if w.fp8 else TOL_BF16
        for got in (first, second):
            assert torch.isfinite(got.float()).all()
            assert (got.float() - ref.float()).abs().max().item() <= tol
            inactive = ~w.active.bool()
            assert (got[inactive].view(torch.int16) == 0).all()
    assert sda.no_alloc_read_errors() == 0


def test_no_alloc_after_a_larger_call_matches_the_oracle():
    """A call with more rows and splits leaves its partials in the shared array; a
    smaller call after it must not read any of them."""
    big = inputs.make_workload(inputs.scaled("gqa", requests=40, ctx=(2000, 5000)), DEV, fill="all")
    small = inputs.make_workload(inputs.scaled("gqa", requests=5, ctx=(1500, 3000), inactive_frac=0.2),
                                 DEV, fill="all")
    no_alloc(big, 4)
    got = no_alloc(small, 2)
    check(small, got, oracle_all(small))
    assert sda.no_alloc_read_errors() == 0


def test_no_alloc_reports_device_flags_until_cleared():
    w = inputs.make_workload(inputs.scaled("gqa", requests=4, ctx=(1000, 3000)), DEV, fill="all")
    sda.no_alloc_read_errors(clear=True)
    good = no_alloc(w, 2)
    assert sda.no_alloc_read_errors() == 0
    col = int(w.positions[0]) // w.block
    saved = int(w.block_table[0, col])
    w.block_table[0, col] = w.cache.shape[0] + 5              # a page past the pool
    bad = no_alloc(w, 2)
    assert torch.isfinite(bad.float()).all()
    # the flag survives later clean calls until it is read with clear
    w.block_table[0, col] = saved
    again = no_alloc(w, 2)
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
    assert sda.no_alloc_read_errors() & sda.FLAG_BOUNDS
    assert sda.no_alloc_read_errors(clear=True) & sda.FLAG_BOUNDS
    assert sda.no_alloc_read_errors() == 0
    no_alloc(w, 1)
    assert sda.no_alloc_read_errors() == 0


def test_no_alloc_refuses_scratch_beyond_its_limit():
    w = inputs.make_workload(inputs.scaled("gqa", requests=4, ctx=(1000, 2000)), DEV, fill="all")
    rows = 704                                          # 704 rows x 16 heads x 2 splits > 8 MiB
    q = torch.zeros(rows, 16, 192, dtype=torch.bfloat16, device=DEV)
    reg = torch.full((rows, w.regions.shape[1]), -1, dtype=torch.int32, device=DEV)
    pos = torch.zeros(rows, dtype=torch.int32, device=DEV)
    act = torch.ones(rows, dtype=torch.uint8, device=DEV)
    table = torch.zeros(rows // 2, w.block_table.shape[1], dtype=torch.int32, device=DEV)
    out = torch.full_like(q, 5.0)
    assert sda.workspace_bytes(rows, 16, 2) > (8 << 20)
    with pytest.raises(sda.SdaError) as e:
        B.sparse_decode_attention_no_alloc(q, w.cache, reg, table, pos, act, out, scale=w.scale, splits=2)
    assert e.value.status == B.SDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 5.0).all()
    # splits = 1 needs only the flag header: the same rows are accepted
    B.sparse_decode_attention_no_alloc(q, w.cache, reg, table, pos, act, out, scale=w.scale, splits=1)
    torch.cuda.synchronize()
    assert (out.view(torch.int16) == 0).all()            # no visible token -> zeros


def test_no_alloc_argument_errors_match_the_regular_entry_point():
    w = inputs.make_workload(inputs.scaled("gqa", requests=2, ctx=(1000, 2000)), DEV, fill="all")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    q17 = torch.zeros(w.rows, 17, 192, dtype=torch.bfloat16, device=DEV)
    out17 = torch.zeros_like(q17)
    cases = [
        (dict(query=q17, output=out17, splits=1), B.SDA_ERR_UNSUPPORTED),     # more than 16 heads
        (dict(splits=65), B.SDA_ERR_INVALID),                                # more than 64 splits
        (dict(splits=0), B.SDA_ERR_INVALID),
        (dict(query_len=0, splits=1), B.SDA_ERR_INVALID),
    ]
    for change, status in cases:
        args = dict(query=w.query, output=torch.empty_like(w.query), splits=2, query_len=1)
        args.update(change)
        common = (args["query"], w.cache, w.regions, w.block_table, w.positions, w.active, args["output"])
        with pytest.raises(sda.SdaError) as regular:
            sda.sparse_decode_attention(*common, scale=w.scale, query_len=args["query_len"],
                                        splits=args["splits"], workspace=ws)
        with pytest.raises(sda.SdaError) as free:
            B.sparse_decode_attention_no_alloc(*common, scale=w.scale, query_len=args["query_len"],
                                               splits=args["splits"])
        assert regular.value.status == free.value.status == status
