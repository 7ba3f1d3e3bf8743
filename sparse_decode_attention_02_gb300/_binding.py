"""ctypes binding of libsdattn.so (argument marshalling only).

Every function here turns torch tensors into the C ABI's `sda_tensor`
descriptors and calls the library; all computation happens in the CUDA
kernels behind include/sdattn.h.  There is no fallback: if the library is
missing or fails to load, the call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsdattn.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "sdattn.h")

SDA_OK, SDA_ERR_INVALID, SDA_ERR_UNSUPPORTED, SDA_ERR_WORKSPACE, SDA_ERR_CUDA, SDA_ERR_TIMEOUT, SDA_ERR_BOUNDS = range(7)
FLAG_BOUNDS = 0x1
FLAG_TIMEOUT = 0x2

_DTYPES = {
    torch.bfloat16: 1,
    torch.float8_e4m3fn: 2,
    torch.uint8: 3,
    torch.int32: 4,
    torch.bool: 5,
    torch.float32: 6,
}


class SdaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class SdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"sparse_decode_attention: {message} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P = ctypes.POINTER(SdaTensor)
    lib.sparse_decode_splits.argtypes = [ctypes.c_int]
    lib.sparse_decode_splits.restype = ctypes.c_int
    lib.sparse_decode_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.sparse_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.sparse_decode_attention.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, P,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_size_t, ctypes.c_void_p]
    lib.sparse_decode_attention.restype = ctypes.c_int
    lib.sparse_decode_swa_splits.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.sparse_decode_swa_splits.restype = ctypes.c_int
    lib.sparse_decode_swa_attention.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, P,
                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.sparse_decode_swa_attention.restype = ctypes.c_int
    lib.sparse_decode_select_regions.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_void_p]
    lib.sparse_decode_select_regions.restype = ctypes.c_int
    lib.sparse_decode_summary_scores.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, P, P, P,
                                                 ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.sparse_decode_summary_scores.restype = ctypes.c_int
    lib.sparse_decode_read_errors.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32),
                                              ctypes.c_int, ctypes.c_void_p]
    lib.sparse_decode_read_errors.restype = ctypes.c_int
    lib.sparse_decode_attention_no_alloc.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, P,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.sparse_decode_attention_no_alloc.restype = ctypes.c_int
    lib.sparse_decode_no_alloc_read_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int,
                                                       ctypes.c_void_p]
    lib.sparse_decode_no_alloc_read_errors.restype = ctypes.c_int
    lib.sparse_decode_timeline_buffer.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    lib.sparse_decode_timeline_buffer.restype = ctypes.c_int
    lib.sparse_decode_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.sparse_decode_set_wait_limit_ns.restype = None
    lib.sparse_decode_status_string.argtypes = [ctypes.c_int]
    lib.sparse_decode_status_string.restype = ctypes.c_char_p
    return lib


def load(path: str | None = None):
    """The loaded library.  Raises if it has not been built (see build.py)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def use_library(path: str):
    """Makes every later call of this module go to the library at `path` (a
    diagnostic build of the same sources, e.g. one compiled with SDA_TIMELINE);
    returns it."""
    global _lib
    with _lock:
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def declared_functions() -> list[str]:
    """Names of the entry points include/sdattn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sparse_decode_\w+)\s*\(", text)))


def describe(t: torch.Tensor | None) -> SdaTensor | None:
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("at most 4 dimensions")
    d = SdaTensor()
    d.data = t.data_ptr() if t.numel() else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _device_of(*tensors, stream: torch.cuda.Stream | None = None) -> torch.device:
    """The one CUDA device that every given tensor (None entries skipped) and
    the stream belong to.  Raises ValueError for a CPU tensor or mixed devices,
    before anything is allocated or launched: the kernels dereference every
    pointer on that device."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"sparse_decode: every tensor must be a CUDA tensor (got one on {t.device})")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"sparse_decode: tensors on {dev} and {t.device}; pass them all on one device")
    if dev is None:
        raise ValueError("sparse_decode: no tensor arguments")
    if stream is not None and stream.device != dev:
        raise ValueError(f"sparse_decode: stream of {stream.device} for tensors on {dev}")
    return dev


def _current(dev: torch.device):
    """Makes `dev` the current device for a library call (the library launches
    on the current device)."""
    return contextlib.nullcontext() if torch.cuda.current_device() == dev.index else torch.cuda.device(dev)


def sparse_decode_splits(rows: int) -> int:
    return load().sparse_decode_splits(int(rows))


def workspace_bytes(rows: int, heads: int, splits: int) -> int:
    return load().sparse_decode_workspace_bytes(int(rows), int(heads), int(splits))


_workspaces: dict = {}


def default_workspace(device: torch.device, nbytes: int, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """A zero-initialised workspace per (device, stream), grown on demand: calls
    on one stream are ordered, so they can share it; another stream gets its own."""
    device = torch.device(device)
    handle = stream.cuda_stream if stream is not None else torch.cuda.current_stream(device).cuda_stream
    key = (device, handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 12), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _scale_ptr(x, device):
    if x is None:
        return None, None
    if not isinstance(x, torch.Tensor):
        x = torch.tensor([float(x)], dtype=torch.float32, device=device)
    if x.dtype != torch.float32 or x.device != device or x.numel() != 1:
        raise ValueError("k_scale / v_scale must be one-element float32 tensors on the query's device")
    return x.data_ptr(), x


def sparse_decode_attention(query, cache, regions, block_table, positions, active, output, *,
                            scale: float, query_len: int = 1, splits: int | None = None,
                            clear_inactive: bool = True, k_scale=None, v_scale=None, gate=None,
                            region_tokens: int = 0, workspace: torch.Tensor | None = None,
                            stream: torch.cuda.Stream | None = None) -> None:
    """Sparse decode attention into `output` (see include/sdattn.h for the contract).

    `splits=None` uses the library's split policy.  `k_scale`/`v_scale` are
    one-element float32 device tensors (python floats are uploaded)."""
    lib = load()
    dev = _device_of(query, cache, regions, block_table, positions, active, output, gate, workspace,
                     stream=stream)
    rows, heads = query.shape[0], query.shape[1]
    if splits is None:
        splits = lib.sparse_decode_splits(rows)
    need = lib.sparse_decode_workspace_bytes(rows, heads, splits)
    if workspace is None:
        workspace = default_workspace(dev, need, stream)
    ks, _keep_k = _scale_ptr(k_scale, dev)
    vs, _keep_v = _scale_ptr(v_scale, dev)
    descs = [describe(x) for x in (query, cache, regions, block_table, positions, active, output)]
    gd = describe(gate)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with _current(dev):
        rc = lib.sparse_decode_attention(*[_ref(d) for d in descs], float(scale), int(query_len),
                                         int(splits), ks, vs, _ref(gd), int(bool(clear_inactive)),
                                         int(region_tokens), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(), s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())


def sparse_decode_swa_splits(rows: int, window: int) -> int:
    return load().sparse_decode_swa_splits(int(rows), int(window))


def sparse_decode_swa_attention(query, cache, block_table, seq_lens, output, *, scale: float,
                                window: int, query_len: int = 1, splits: int | None = None,
                                k_scale=None, v_scale=None, gate=None,
                                workspace: torch.Tensor | None = None,
                                stream: torch.cuda.Stream | None = None) -> None:
    """Gated sliding-window decode into `output` (see include/sdattn.h).

    `splits=None` uses the library's window split policy."""
    lib = load()
    dev = _device_of(query, cache, block_table, seq_lens, output, gate, workspace, stream=stream)
    rows, heads = query.shape[0], query.shape[1]
    if splits is None:
        splits = lib.sparse_decode_swa_splits(rows, int(window))
    need = lib.sparse_decode_workspace_bytes(rows, heads, splits)
    if workspace is None:
        workspace = default_workspace(dev, need, stream)
    ks, _keep_k = _scale_ptr(k_scale, dev)
    vs, _keep_v = _scale_ptr(v_scale, dev)
    descs = [describe(x) for x in (query, cache, block_table, seq_lens, output)]
    gd = describe(gate)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with _current(dev):
        rc = lib.sparse_decode_swa_attention(*[_ref(d) for d in descs], float(scale), int(window),
                                             int(query_len), int(splits), ks, vs, _ref(gd), workspace.data_ptr(),
                                             workspace.numel() * workspace.element_size(), s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())


def sparse_decode_select_regions(scores, current, topk: int, regions=None, *, topk_lengths=None,
                                 stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Region selection into `regions` ([rows, topk] int32, allocated if None);
    see include/sdattn.h for the rule.  Returns `regions`."""
    lib = load()
    dev = _device_of(scores, current, topk_lengths, regions, stream=stream)
    if regions is None:
        regions = torch.empty((scores.shape[0], int(topk)), dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    d = [describe(x) for x in (scores, current, topk_lengths, regions)]
    with _current(dev):
        rc = lib.sparse_decode_select_regions(_ref(d[0]), _ref(d[1]), _ref(d[2]), int(topk), _ref(d[3]),
                                              s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())
    return regions


def sparse_decode_summary_scores(query, weights, summaries, block_table, seq_lens, *, block_size: int,
                                 n_cols: int | None = None, query_len: int = 1, scores=None,
                                 current=None, lengths=None, workspace=None,
                                 stream: torch.cuda.Stream | None = None):
    """Indexer decode scores into `scores` ([tokens * G, n_cols] fp32, allocated
    if None; n_cols defaults to block_table's width * block_size / 8), with the
    optional `current` / `lengths` outputs; see include/sdattn.h.  Returns
    `scores`."""
    lib = load()
    dev = _device_of(query, weights, summaries, block_table, seq_lens, scores, current, lengths, workspace,
                     stream=stream)
    rows = query.shape[0] * query.shape[1]
    if scores is None:
        if n_cols is None:
            n_cols = block_table.shape[1] * int(block_size) // 8
        scores = torch.empty((rows, int(n_cols)), dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    d = [describe(x) for x in (query, weights, summaries, block_table, seq_lens, scores, current, lengths)]
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _current(dev):
        rc = lib.sparse_decode_summary_scores(_ref(d[0]), _ref(d[1]), _ref(d[2]), _ref(d[3]), _ref(d[4]),
                                              int(block_size), int(query_len), _ref(d[5]), _ref(d[6]),
                                              _ref(d[7]), ws, wsb, s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())
    return scores


def read_errors(workspace: torch.Tensor, clear: bool = False,
                stream: torch.cuda.Stream | None = None) -> int:
    """Device error flags (FLAG_BOUNDS | FLAG_TIMEOUT) recorded in a workspace; synchronises."""
    lib = load()
    dev = _device_of(workspace, stream=stream)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    out = ctypes.c_uint32(0)
    with _current(dev):
        rc = lib.sparse_decode_read_errors(workspace.data_ptr(), ctypes.byref(out), int(clear), s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())
    return out.value


def set_wait_limit_ns(ns: int) -> None:
    load().sparse_decode_set_wait_limit_ns(int(ns))


def status_string(code: int) -> str:
    return load().sparse_decode_status_string(int(code)).decode()


def sparse_decode_attention_no_alloc(query, cache, regions, block_table, positions, active, output, *,
                                     scale: float, query_len: int = 1, splits: int | None = None,
                                     clear_inactive: bool = True, k_scale=None, v_scale=None, gate=None,
                                     region_tokens: int = 0, stream: torch.cuda.Stream | None = None) -> None:
    """The allocation-free C entry point: same contract as sparse_decode_attention
    but its scratch is the library's static 8 MiB device array (no workspace
    argument).  For callers that cannot allocate device memory; calls that
    overlap on the GPU race on the shared array.  Device flags collect in the
    array until read with `no_alloc_read_errors(clear=True)`.
    `k_scale`/`v_scale` must be device tensors here (uploading a python float
    would allocate)."""
    lib = load()
    fn = lib.sparse_decode_attention_no_alloc
    for x in (k_scale, v_scale):
        if x is not None and not isinstance(x, torch.Tensor):
            raise TypeError("k_scale / v_scale must be device tensors for the allocation-free call")
    dev = _device_of(query, cache, regions, block_table, positions, active, output, gate, stream=stream)
    rows = query.shape[0]
    if splits is None:
        splits = lib.sparse_decode_splits(rows)
    ks, _keep_k = _scale_ptr(k_scale, dev)
    vs, _keep_v = _scale_ptr(v_scale, dev)
    descs = [describe(x) for x in (query, cache, regions, block_table, positions, active, output)]
    gd = describe(gate)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with _current(dev):
        rc = fn(*[_ref(d) for d in descs], float(scale), int(query_len), int(splits), ks, vs, _ref(gd),
                int(bool(clear_inactive)), int(region_tokens), s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())


def no_alloc_read_errors(clear: bool = False, stream: torch.cuda.Stream | None = None,
                         device: torch.device | int | None = None) -> int:
    """Device error flags (FLAG_BOUNDS | FLAG_TIMEOUT) that the allocation-free
    entry point's calls on `device` (default: the current one) have collected
    in its static array; synchronises `stream`, optionally clears them."""
    lib = load()
    if device is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    elif isinstance(device, int):
        dev = torch.device("cuda", device)
    else:
        dev = torch.device(device)
        dev = torch.device("cuda", dev.index if dev.index is not None else torch.cuda.current_device())
    if stream is not None and stream.device != dev:
        raise ValueError(f"sparse_decode: stream of {stream.device} for {dev}")
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    out = ctypes.c_uint32(0)
    with _current(dev):
        rc = lib.sparse_decode_no_alloc_read_errors(ctypes.byref(out), int(clear), s.cuda_stream)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())
    return out.value


def timeline_buffer(buffer: torch.Tensor | None) -> None:
    """Registers a device buffer for the kernels' phase stamps (a library built
    with SDA_TIMELINE only; the regular one raises SdaError UNSUPPORTED)."""
    lib = load()
    ptr = buffer.data_ptr() if buffer is not None else None
    nbytes = buffer.numel() * buffer.element_size() if buffer is not None else 0
    rc = lib.sparse_decode_timeline_buffer(ptr, nbytes)
    if rc != SDA_OK:
        raise SdaError(rc, lib.sparse_decode_status_string(rc).decode())
