"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the float64 oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_decode_attention_02_gb300 as sda
from sparse_decode_attention_02_gb300 import inputs

TOL_BF16 = 2e-2      # max |gpu - oracle| with a bf16 cache, unit-variance V
TOL_FP8 = 5e-2       # with an FP8 E4M3 cache


def tol(w) -> float:
    return TOL_FP8 if w.fp8 else TOL_BF16


def scales(w):
    if not w.fp8:
        return None, None
    dev = w.query.device
    return (torch.tensor([w.k_scale], dtype=torch.float32, device=dev),
            torch.tensor([w.v_scale], dtype=torch.float32, device=dev))


def run(w, *, splits=None, out=None, clear_inactive=True, workspace=None, cache=None, **kw):
    """The CUDA path on workload `w`; returns (output bf16 tensor, device flags)."""
    splits = splits or w.splits or sda.sparse_decode_splits(w.rows)
    if out is None:
        out = torch.full_like(w.query, float("nan"))
    if workspace is None:
        workspace = torch.zeros(sda.workspace_bytes(w.rows, w.heads, splits), dtype=torch.uint8,
                                device=w.query.device)
    ks, vs = scales(w)
    sda.sparse_decode_attention(w.query, w.cache if cache is None else cache, w.regions, w.block_table,
                                w.positions, w.active, out, scale=w.scale, query_len=w.query_len,
                                splits=splits, clear_inactive=clear_inactive, k_scale=ks, v_scale=vs,
                                gate=w.gate, region_tokens=w.region_tokens, workspace=workspace, **kw)
    torch.cuda.synchronize()
    return out, sda.read_errors(workspace)


def run_swa(w, *, splits=None, out=None, workspace=None):
    """The window path on a window workload; returns (output, device flags)."""
    splits = splits or sda.sparse_decode_swa_splits(w.rows, w.window)
    if out is None:
        out = torch.full_like(w.query, float("nan"))
    if workspace is None:
        workspace = torch.zeros(sda.workspace_bytes(w.rows, w.heads, splits), dtype=torch.uint8,
                                device=w.query.device)
    ks, vs = scales(w)
    sda.sparse_decode_swa_attention(w.query, w.cache, w.block_table, w.seq_lens, out, scale=w.scale,
                                    window=w.window, query_len=w.query_len, splits=splits, k_scale=ks,
                                    v_scale=vs, gate=w.gate, workspace=workspace)
    torch.cuda.synchronize()
    return out, sda.read_errors(workspace)


def oracle_swa_rows(w, rows) -> np.ndarray:
    hp = inputs.host_subset(w, rows)
    return oracle.swa_decode(hp.query, hp.cache, hp.block_table, hp.seq_lens, scale=w.scale,
                             window=w.window, query_len=w.query_len, k_scale=w.k_scale,
                             v_scale=w.v_scale, cache_fp8=w.fp8, gate=hp.gate, row_ids=hp.row_ids)


def oracle_all(w) -> np.ndarray:
    return oracle.sparse_decode_attention(
        w.query.cpu(), w.cache.cpu(), w.regions.cpu(), w.block_table.cpu(), w.positions.cpu(),
        w.active.cpu(), gate=None if w.gate is None else w.gate.cpu(), scale=w.scale,
        query_len=w.query_len, region_tokens=w.region_tokens, k_scale=w.k_scale,
        v_scale=w.v_scale, cache_fp8=w.fp8)


def oracle_rows(w, rows) -> np.ndarray:
    hp = inputs.host_subset(w, rows)
    return oracle.sparse_decode_attention(hp.query, hp.cache, hp.regions, hp.block_table, hp.positions,
                                          hp.active, gate=hp.gate, row_ids=hp.row_ids, **hp.kwargs)


def check(w, got: torch.Tensor, ref: np.ndarray, rows=None, tolerance=None):
    """Element-wise comparison; inactive rows must be +0.0 bit-exactly."""
    g = got if rows is None else got[torch.as_tensor(np.asarray(rows), device=got.device)]
    act = w.active.cpu().numpy().astype(bool)
    if rows is not None:
        act = act[np.asarray(rows)]
    gf = g.float().cpu().numpy()
    assert np.isfinite(gf).all(), "non-finite output"
    bits = g.view(torch.int16).cpu().numpy()
    assert (bits[~act] == 0).all(), "inactive rows must be +0.0"
    err = np.abs(gf - ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= (tolerance or tol(w)), f"max abs err {worst:.4g} (tol {tolerance or tol(w)})"
    return worst


def sample_rows(w, n, seed=0):
    """n rows spread over the batch, always including inactive rows and the
    rows with the fewest live regions."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(w.rows, size=min(n, w.rows), replace=False).tolist())
    act = w.active.cpu().numpy()
    rows.update(np.nonzero(act == 0)[0][:4].tolist())
    live = (w.regions >= 0).sum(1).cpu().numpy()
    rows.update(np.argsort(live)[:4].tolist())
    rows.update([0, w.rows - 1])
    return sorted(rows)
