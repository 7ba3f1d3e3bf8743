"""Gated sliding-window decode (CUDA path vs the float64 oracle).

The non-DSA layers' fused decode (page "vllm.models.step5.nvidia.
sparse_attention", forward_with_headwise_gate -> swa_decode_gated): token j
of request q at p = seq_lens[q] - query_len + j attends over
[max(0, p - window + 1), p], then the headwise gate.  Same tolerances as the
sparse path."""
import gc

import numpy as np
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import check, oracle_swa_rows, run_swa, sample_rows
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def mini(**changes):
    return inputs.make_workload(inputs.scaled("swa", **changes), DEV, fill="all")


@pytest.mark.parametrize("splits", [None, 2])    # the policy (one split), and token pairs with partials
def test_swa_workload_sampled_rows(splits):
    w = inputs.make_workload("swa", DEV)
    out, flags = run_swa(w, splits=splits)
    assert flags == 0
    assert torch.isfinite(out.float()).all()
    rows = sample_rows(w, 128)
    check(w, out, oracle_swa_rows(w, rows), rows)


@pytest.mark.parametrize("window", [1, 37, 700, 100_000])
@pytest.mark.parametrize("fp8", [False, True])
def test_swa_windows(window, fp8):
    w = mini(requests=5, ctx=(1500, 5000), window=window, fp8=fp8)
    rows = list(range(w.rows))
    ref = oracle_swa_rows(w, rows)
    for s in (1, 2, 3):
        out, flags = run_swa(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)


@pytest.mark.parametrize("changes", [
    dict(query_len=1, groups=1, heads=1),
    dict(query_len=3, groups=2, heads=5),
    dict(query_len=4, groups=4, heads=16, block=16),
    dict(query_len=2, groups=2, heads=8, block=32, gate=False),
    dict(query_len=2, groups=2, heads=8, block=24),                 # 24-token pieces
    dict(query_len=1, groups=2, heads=4, block=48, fp8=True),       # one 48-token piece per stage
])
def test_swa_shapes(changes):
    w = mini(requests=4, ctx=(900, 3000), window=513, **changes)
    rows = list(range(w.rows))
    ref = oracle_swa_rows(w, rows)
    for s in (1, 4):
        out, flags = run_swa(w, splits=s)
        assert flags == 0
        check(w, out, ref, rows)


def test_swa_window_one_returns_v():
    w = mini(requests=4, ctx=(900, 3000), window=1, gate=False)
    out, flags = run_swa(w, splits=1)
    assert flags == 0
    G, ql, B = w.groups, w.query_len, w.block
    for r in range(w.rows):
        req, g = r // (G * ql), r % G
        t = int(w.positions[r])
        v = w.cache[int(w.block_table[req, t // B]), g, t % B, 192:]
        assert torch.equal(out[r].view(torch.int16), v.expand(w.heads, 192).contiguous().view(torch.int16))


@pytest.mark.parametrize("splits", [1, 2])       # 1: token pairs share a CTA
def test_swa_rows_before_the_sequence_start_are_zero(splits):
    w = mini(requests=4, ctx=(900, 3000), window=64, query_len=2)
    w.seq_lens[0] = 1          # token 0 of request 0 would sit at position -1
    w.seq_lens[1] = 2          # request 1's tokens sit at positions 0 and 1
    ql = w.query_len
    tok = torch.arange(w.rows // w.groups, device=w.seq_lens.device)
    w.positions = (w.seq_lens.long()[tok // ql] - ql + tok % ql).repeat_interleave(w.groups).to(torch.int32)
    out, flags = run_swa(w, splits=splits)
    assert flags == 0
    G = w.groups
    assert (out[:G].view(torch.int16) == 0).all()        # request 0, token 0: every group
    rows = list(range(w.rows))
    check(w, out, oracle_swa_rows(w, rows), rows)
