"""The allocation-free entry point against the regular one (GPU).

sparse_decode_attention_no_alloc serves callers that cannot allocate device
memory (plugin or FFI hosts handed tensor pointers but no allocator, code that
must not cudaMalloc in the middle of a capture); its split-KV scratch is a
static 8 MiB device array inside the library.  Two calls in a row, on
different workloads and split counts, must each match the regular entry point
(caller-supplied workspace) within the parity tolerance; a call whose scratch
would not fit is refused before anything is enqueued.  Collected last so a
failure here cannot hide failures of the other tests.
"""
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import TOL_BF16, TOL_FP8, run, scales
from sparse_decode_attention_02_gb300 import _binding as B
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def no_alloc(w, splits):
    out = torch.full_like(w.query, float("nan"))
    ks, vs = scales(w)
    B.sparse_decode_attention_no_alloc(w.query, w.cache, w.regions, w.block_table, w.positions,
                                       w.active, out, scale=w.scale, query_len=w.query_len,
                                       splits=splits, k_scale=ks, v_scale=vs, gate=w.gate,
                                       region_tokens=w.region_tokens)
    torch.cuda.synchronize()
    return out


def test_no_alloc_matches_regular_entry_point_twice():
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
