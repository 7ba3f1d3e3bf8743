"""CPU float64 oracle for DSA sparse decode attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It wraps ``sda_oracle.c`` (plain C, float64,
built with gcc on first use) through ctypes and shares nothing with the CUDA
library.  Inputs are numpy arrays or CPU torch tensors holding the same bytes
the GPU path receives: bf16 as raw 16-bit patterns, FP8 E4M3 as raw bytes.

The definition it computes is the one of the vLLM API page
"vllm.models.step5.nvidia.ops.sparse_decode_attention" (functions
``sparse_decode_attention``, ``_gate`` and ``sparse_decode_splits``), plus the
steps around it on the neighbouring pages (sliding-window decode, region
selection, indexer decode scores); the C file's header lists the readings
taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_sda.so")
_lock = threading.Lock()
_lib = None


def build(out_path: str = _LIB_PATH, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with one planted mistake) and return the .so path."""
    if (not force and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= os.path.getmtime(_SRC)):
        return out_path
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _declare(lib):
    i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    common = [vp, i64, i64, i32, i32,            # query, q_s0, q_s1, rows, heads
              vp, i32, i64, i32, i32,            # cache, fp8, pages, groups, block
              i64, i64, i64,                     # c_s0, c_s1, c_s2
              vp, i64, i32,                      # regions, reg_s0, R
              vp, i64, i32, i32,                 # block_table, bt_s0, table rows, cols
              vp, vp,                            # positions, active
              dbl, i32, i32, dbl, dbl]           # scale, query_len, RT, k_scale, v_scale
    lib.oracle_sparse_decode_attention.argtypes = common + [vp, i64, i64, vp, i32, vp]
    lib.oracle_sparse_decode_attention.restype = i32
    lib.oracle_split_partials.argtypes = common + [i32, vp, i32, vp, vp]
    lib.oracle_split_partials.restype = i32
    lib.oracle_swa_decode.argtypes = [vp, i64, i64, i32, i32, vp, i32, i64, i32, i32, i64, i64, i64,
                                      vp, i64, i32, i32, vp, i32, dbl, i32, i32, dbl, dbl,
                                      vp, i64, i64, vp, i32, vp]
    lib.oracle_swa_decode.restype = i32
    lib.oracle_select_regions.argtypes = [vp, i64, i32, i32, vp, vp, i32, vp]
    lib.oracle_select_regions.restype = i32
    lib.oracle_summary_scores.argtypes = [vp, i64, i64, i32, i32, vp, i64, i64, vp, i64, i64,
                                          vp, i64, i32, i32, vp, i32, i32, i32, vp, i32, vp, vp, vp]
    lib.oracle_summary_scores.restype = i32
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = dbl
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = dbl
    lib.oracle_bf16_round.argtypes = [ctypes.c_float]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_gate_factor.argtypes = [ctypes.c_uint16]
    lib.oracle_gate_factor.restype = dbl
    lib.oracle_sparse_decode_splits.argtypes = [i32]
    lib.oracle_sparse_decode_splits.restype = i32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_num_threads.argtypes = [i32]
    lib.oracle_set_num_threads.restype = None
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use).  ``path`` loads another build, e.g. a mutant."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


class OracleError(RuntimeError):
    pass


_ERRORS = {-1: "bad arguments", -2: "region id below -1", -3: "token past the block-table width",
           -4: "block-table entry is not a page of the cache", -5: "out of host memory"}


def _np(x, dtype):
    """A numpy view of x's bytes as ``dtype`` (torch CPU tensors are reinterpreted, not converted)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("the oracle takes host tensors")
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.view(torch.int16)
            elif x.dtype in (torch.float8_e4m3fn, torch.bool):
                x = x.view(torch.uint8)
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype.itemsize != np.dtype(dtype).itemsize:
        raise ValueError(f"expected {np.dtype(dtype)}-sized elements, got {x.dtype}")
    return x.view(dtype)


def _estrides(a):
    return [s // a.itemsize for s in a.strides]


class Problem:
    """The arguments of one call, as host arrays plus the C argument list."""

    def __init__(self, query, cache, regions, block_table, positions, active, *, scale,
                 query_len=1, region_tokens=None, k_scale=None, v_scale=None, cache_fp8=None):
        self.query = _np(query, np.uint16)
        if cache_fp8 is None:
            cache_fp8 = _itemsize(cache) == 1
        self.fp8 = bool(cache_fp8)
        self.cache = _np(cache, np.uint8 if self.fp8 else np.uint16)
        self.regions = _np(regions, np.int32)
        self.block_table = _np(block_table, np.int32)
        self.positions = np.ascontiguousarray(_np(positions, np.int32))
        self.active = np.ascontiguousarray(_np(active, np.uint8))
        rows, heads, dim = self.query.shape
        pages, groups, block, width = self.cache.shape
        if dim != 192 or width != 384:
            raise ValueError("query dim must be 192 and cache rows 384 wide")
        if self.fp8 and (k_scale is None or v_scale is None):
            raise ValueError("an FP8 cache needs k_scale and v_scale")
        self.rows, self.heads, self.groups, self.block = rows, heads, groups, block
        self.query_len = int(query_len)
        self.region_tokens = int(region_tokens or block)
        qs, cs = _estrides(self.query), _estrides(self.cache)
        if qs[2] != 1 or cs[3] != 1:
            raise ValueError("inner strides must be 1")
        rs, bs = _estrides(self.regions), _estrides(self.block_table)
        if rows and rs[1] != 1 or bs[1] != 1:
            raise ValueError("regions / block_table rows must be contiguous")
        self.args = [
            self.query.ctypes.data, qs[0], qs[1], rows, heads,
            self.cache.ctypes.data, int(self.fp8), pages, groups, block, cs[0], cs[1], cs[2],
            self.regions.ctypes.data, rs[0], self.regions.shape[1],
            self.block_table.ctypes.data, bs[0], self.block_table.shape[0], self.block_table.shape[1],
            self.positions.ctypes.data, self.active.ctypes.data,
            float(scale), self.query_len, self.region_tokens,
            float(k_scale if k_scale is not None else 1.0), float(v_scale if v_scale is not None else 1.0),
        ]


def _itemsize(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.element_size()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x).itemsize


def _rows_arg(row_ids, rows):
    if row_ids is None:
        return None, rows
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int32))
    return ids, len(ids)


def sparse_decode_attention(query, cache, regions, block_table, positions, active, *, scale,
                            query_len=1, region_tokens=None, k_scale=None, v_scale=None,
                            gate=None, cache_fp8=None, row_ids=None, lib=None) -> np.ndarray:
    """float64 output [n, heads, 192] for ``row_ids`` (default: every row).

    ``cache_fp8`` defaults to "the cache has 1-byte elements".  ``gate`` is the
    bf16 [tokens, G * heads] headwise gate or None.  ``lib`` selects another
    oracle build (used by the pin-strength test)."""
    lib = lib or load()
    p = Problem(query, cache, regions, block_table, positions, active, scale=scale,
                query_len=query_len, region_tokens=region_tokens, k_scale=k_scale,
                v_scale=v_scale, cache_fp8=cache_fp8)
    ids, n = _rows_arg(row_ids, p.rows)
    out = np.zeros((n, p.heads, 192), dtype=np.float64)
    if gate is not None:
        g = _np(gate, np.uint16)
        gs = _estrides(g)
        gate_args = [g.ctypes.data, gs[0], gs[1]]
    else:
        g = None
        gate_args = [None, 0, 0]
    rc = lib.oracle_sparse_decode_attention(
        *p.args, *gate_args, ids.ctypes.data if ids is not None else None, n, out.ctypes.data)
    if rc:
        raise OracleError(_ERRORS.get(rc, str(rc)))
    return out


def split_partials(query, cache, regions, block_table, positions, active, *, scale, splits,
                   query_len=1, region_tokens=None, k_scale=None, v_scale=None,
                   cache_fp8=None, row_ids=None, lib=None):
    """(partial [n, S, heads, 192], lse [n, S, heads]) float64 for split-KV chunk s of S."""
    lib = lib or load()
    p = Problem(query, cache, regions, block_table, positions, active, scale=scale,
                query_len=query_len, region_tokens=region_tokens, k_scale=k_scale,
                v_scale=v_scale, cache_fp8=cache_fp8)
    ids, n = _rows_arg(row_ids, p.rows)
    partial = np.zeros((n, splits, p.heads, 192), dtype=np.float64)
    lse = np.zeros((n, splits, p.heads), dtype=np.float64)
    rc = lib.oracle_split_partials(*p.args, int(splits), ids.ctypes.data if ids is not None else None,
                                   n, partial.ctypes.data, lse.ctypes.data)
    if rc:
        raise OracleError(_ERRORS.get(rc, str(rc)))
    return partial, lse


def swa_decode(query, cache, block_table, seq_lens, *, scale, window, query_len=1, k_scale=None,
               v_scale=None, gate=None, cache_fp8=None, row_ids=None, lib=None) -> np.ndarray:
    """Gated sliding-window decode: float64 output [n, heads, 192] for ``row_ids``.

    Token j of request q sits at seq_lens[q] - query_len + j and attends over the
    ``window`` tokens ending at it (the non-DSA layers' fused decode)."""
    lib = lib or load()
    q = _np(query, np.uint16)
    if cache_fp8 is None:
        cache_fp8 = _itemsize(cache) == 1
    c = _np(cache, np.uint8 if cache_fp8 else np.uint16)
    bt = _np(block_table, np.int32)
    sl = np.ascontiguousarray(_np(seq_lens, np.int32))
    rows, heads, dim = q.shape
    pages, groups, block, width = c.shape
    if dim != 192 or width != 384:
        raise ValueError("query dim must be 192 and cache rows 384 wide")
    if cache_fp8 and (k_scale is None or v_scale is None):
        raise ValueError("an FP8 cache needs k_scale and v_scale")
    qs, cs, bs = _estrides(q), _estrides(c), _estrides(bt)
    ids, n = _rows_arg(row_ids, rows)
    out = np.zeros((n, heads, 192), dtype=np.float64)
    if gate is not None:
        g = _np(gate, np.uint16)
        gs = _estrides(g)
        gate_args = [g.ctypes.data, gs[0], gs[1]]
    else:
        gate_args = [None, 0, 0]
    rc = lib.oracle_swa_decode(
        q.ctypes.data, qs[0], qs[1], rows, heads, c.ctypes.data, int(bool(cache_fp8)), pages, groups,
        block, cs[0], cs[1], cs[2], bt.ctypes.data, bs[0], bt.shape[0], bt.shape[1], sl.ctypes.data,
        len(sl), float(scale), int(query_len), int(window),
        float(k_scale if k_scale is not None else 1.0), float(v_scale if v_scale is not None else 1.0),
        *gate_args, ids.ctypes.data if ids is not None else None, n, out.ctypes.data)
    if rc:
        raise OracleError(_ERRORS.get(rc, str(rc)))
    return out


def select_regions(scores, current, topk, topk_lengths=None, lib=None) -> np.ndarray:
    """Region selection: int32 [rows, topk], the current region first, then the
    topk - 1 best-scoring other candidates among ids [0, topk_lengths[r]) in
    ascending id order, padded with -1 (ties go to the lower id)."""
    lib = lib or load()
    sc = _np(scores, np.float32)
    if sc.ndim != 2:
        raise ValueError("scores must be [rows, N]")
    if sc.shape[1] and _estrides(sc)[1] != 1:
        sc = np.ascontiguousarray(sc)
    cur = np.ascontiguousarray(_np(current, np.int32))
    ln = None if topk_lengths is None else np.ascontiguousarray(_np(topk_lengths, np.int32))
    rows, n_cols = sc.shape
    out = np.zeros((rows, topk), dtype=np.int32)
    rc = lib.oracle_select_regions(sc.ctypes.data, _estrides(sc)[0], rows, n_cols, cur.ctypes.data,
                                   ln.ctypes.data if ln is not None else None, int(topk), out.ctypes.data)
    if rc:
        raise OracleError(_ERRORS.get(rc, str(rc)))
    return out


def summary_scores(query, weights, summaries, block_table, seq_lens, *, block, n_cols,
                   query_len=1, row_ids=None, lib=None):
    """Indexer decode scores: (scores float64 [n, n_cols], current int32 [n],
    lengths int32 [n]) for the rows (token, g) in ``row_ids`` (all rows when None).

    query [tokens, G, 8, 256] E4M3 bytes (heads and dims contiguous), weights
    [tokens, G, 8] fp32, summaries [slots, G, 256] E4M3 bytes (one slot per
    8-token region of every page, slot = page * (block / 8) + offset / 8)."""
    lib = lib or load()
    q = _np(query, np.uint8)
    w = _np(weights, np.float32)
    m = _np(summaries, np.uint8)
    bt = _np(block_table, np.int32)
    sl = np.ascontiguousarray(_np(seq_lens, np.int32))
    if q.ndim != 4 or q.shape[2:] != (8, 256) or _estrides(q)[2:] != [256, 1]:
        raise ValueError("query must be [tokens, G, 8, 256] with heads and dims contiguous")
    tokens, groups = q.shape[:2]
    if w.shape != (tokens, groups, 8) or _estrides(w)[2] != 1:
        raise ValueError("weights must be [tokens, G, 8] with unit head stride")
    if m.ndim != 3 or m.shape[1:] != (groups, 256) or _estrides(m)[1:] != [256, 1]:
        raise ValueError("summaries must be [slots, G, 256] with groups and dims contiguous")
    if bt.shape[1] and _estrides(bt)[1] != 1:
        bt = np.ascontiguousarray(bt)
    ids, n = _rows_arg(row_ids, tokens * groups)
    out = np.zeros((n, n_cols), dtype=np.float64)
    cur = np.zeros(n, dtype=np.int32)
    lens = np.zeros(n, dtype=np.int32)
    qs, ws, ms = _estrides(q), _estrides(w), _estrides(m)
    rc = lib.oracle_summary_scores(
        q.ctypes.data, qs[0], qs[1], tokens, groups, w.ctypes.data, ws[0], ws[1], m.ctypes.data,
        ms[0], m.shape[0], bt.ctypes.data, _estrides(bt)[0], bt.shape[0], bt.shape[1], sl.ctypes.data,
        int(block), int(query_len), int(n_cols), ids.ctypes.data if ids is not None else None, n,
        out.ctypes.data, cur.ctypes.data, lens.ctypes.data)
    if rc:
        raise OracleError(_ERRORS.get(rc, str(rc)))
    return out, cur, lens


def e4m3_decode(code: int, lib=None) -> float:
    return (lib or load()).oracle_e4m3_decode(code)


def bf16_decode(bits: int, lib=None) -> float:
    return (lib or load()).oracle_bf16_decode(bits)


def bf16_round(x: float, lib=None) -> int:
    return (lib or load()).oracle_bf16_round(x)


def gate_factor(bits: int, lib=None) -> float:
    return (lib or load()).oracle_gate_factor(bits)


def sparse_decode_splits(rows: int, lib=None) -> int:
    return (lib or load()).oracle_sparse_decode_splits(rows)


def num_threads() -> int:
    return load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    load().oracle_set_num_threads(int(n))
