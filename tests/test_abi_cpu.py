"""Host-side tests of the C-ABI library (no GPU needed).

The library loads and exports every entry point include/sdattn.h declares;
the split policy and workspace sizing are exact; every contract violation is
rejected with its status code before any CUDA call is made."""
import ctypes
import os

import numpy as np
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from sparse_decode_attention_02_gb300 import _binding as B
from sparse_decode_attention_02_gb300 import build as lib_build

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return sda.load()


def test_exports_every_declared_symbol(lib):
    names = sda.declared_functions()
    assert {"sparse_decode_attention", "sparse_decode_splits", "sparse_decode_workspace_bytes",
            "sparse_decode_read_errors"} <= set(names)
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_splits_truth_table(lib):
    with open(os.path.join(GOLDEN, "sparse_decode_splits.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lo, hi, s = (int(x) for x in line.split())
            for rows in range(lo, hi + 1):
                assert sda.sparse_decode_splits(rows) == s, rows
    assert sda.sparse_decode_splits(10 ** 6) == 1


def test_workspace_bytes(lib):
    assert sda.workspace_bytes(100, 16, 1) == 256
    n = 128 * 2 * 16
    assert sda.workspace_bytes(128, 16, 2) == 256 + n * 192 * 4 + ((n * 4 + 255) // 256) * 256
    assert sda.workspace_bytes(4, 17, 1) == 0
    assert sda.workspace_bytes(4, 8, 65) == 0


class FakeDev:
    """Descriptors with fake device addresses: validation never dereferences them."""

    def __init__(self, rows=8, H=16, pages=64, G=2, Bk=64, R=8, reqs=4, W=16, fp8=False):
        self.rows, self.H = rows, H
        self.q = self.t(1, (rows, H, 192))
        self.cache = self.t(3 if fp8 else 1, (pages, G, Bk, 384))
        self.regions = self.t(4, (rows, R))
        self.table = self.t(4, (reqs, W))
        self.pos = self.t(4, (rows,))
        self.act = self.t(5, (rows,))
        self.out = self.t(1, (rows, H, 192))
        self.gate = None
        self.fp8 = fp8

    @staticmethod
    def t(dtype, shape, strides=None, addr=1 << 20):
        d = B.SdaTensor()
        d.data = addr
        d.dtype = dtype
        d.ndim = len(shape)
        if strides is None:
            strides, acc = [], 1
            for n in reversed(shape):
                strides.insert(0, acc)
                acc *= n
        for i, (n, s) in enumerate(zip(shape, strides)):
            d.shape[i] = n
            d.stride[i] = s
        return d

    def call(self, lib, splits=1, rt=0, ws_bytes=None, ws_addr=1 << 24, query_len=1, scale=0.07,
             kscale=True):
        ws_bytes = lib.sparse_decode_workspace_bytes(self.rows, self.H, splits) if ws_bytes is None else ws_bytes
        ks = ctypes.c_void_p(1 << 12) if (self.fp8 and kscale) else None
        r = ctypes.byref
        return lib.sparse_decode_attention(
            r(self.q), r(self.cache), r(self.regions), r(self.table), r(self.pos), r(self.act),
            r(self.out), scale, query_len, splits, ks, ks,
            r(self.gate) if self.gate is not None else None, 1, rt, ws_addr, ws_bytes, None)


def test_rejects_contract_violations(lib):
    INV, UNS, WS = B.SDA_ERR_INVALID, B.SDA_ERR_UNSUPPORTED, B.SDA_ERR_WORKSPACE
    f = FakeDev(H=17)
    f.q = f.t(1, (8, 17, 192)); f.out = f.t(1, (8, 17, 192))
    assert f.call(lib) == UNS                                   # heads > 16
    f = FakeDev(); f.q = f.t(1, (8, 16, 191)); assert f.call(lib) == INV     # dim != 192
    f = FakeDev(); f.cache = f.t(1, (64, 2, 64, 383)); assert f.call(lib) == INV
    f = FakeDev(); f.q = f.t(1, (8, 16, 192), (16 * 384, 384, 2)); assert f.call(lib) == INV  # inner stride
    f = FakeDev(); f.regions = f.t(4, (8, 8), (16, 2)); assert f.call(lib) == INV
    f = FakeDev(); f.regions = f.t(4, (7, 8)); assert f.call(lib) == INV      # rows mismatch
    f = FakeDev(); f.pos = f.t(1, (8,)); assert f.call(lib) == INV            # dtype
    f = FakeDev(fp8=True); assert f.call(lib, kscale=False) == INV            # FP8 without scales
    f = FakeDev(); assert f.call(lib, splits=0) == INV
    f = FakeDev(); assert f.call(lib, splits=65) == INV
    f = FakeDev(); assert f.call(lib, query_len=0) == INV
    f = FakeDev(); assert f.call(lib, scale=float("nan")) == INV
    f = FakeDev(rows=7); f.regions = f.t(4, (7, 8)); f.pos = f.t(4, (7,)); f.act = f.t(5, (7,))
    f.q = f.t(1, (7, 16, 192)); f.out = f.t(1, (7, 16, 192))
    assert f.call(lib) == INV                                   # rows not a multiple of G
    f = FakeDev(rows=12, reqs=2)
    for name in ("regions", "pos", "act"):
        pass
    f.regions = f.t(4, (12, 8)); f.pos = f.t(4, (12,)); f.act = f.t(5, (12,))
    f.q = f.t(1, (12, 16, 192)); f.out = f.t(1, (12, 16, 192))
    assert f.call(lib) == INV                                   # more requests than table rows
    f = FakeDev(); f.gate = f.t(1, (4, 31)); assert f.call(lib) == INV       # gate width != G*H
    f = FakeDev(); assert f.call(lib, rt=4) == UNS             # piece not a multiple of 8
    f = FakeDev(); assert f.call(lib, rt=24) == UNS            # RT not a multiple of the piece
    f = FakeDev(); f.cache = f.t(1, (64, 2, 64, 384), (2 * 64 * 384 + 3, 64 * 384, 384, 1))
    assert f.call(lib) == UNS                                   # page stride not 16-byte
    f = FakeDev(); assert f.call(lib, ws_bytes=100) == WS
    f = FakeDev(); assert f.call(lib, ws_addr=(1 << 24) + 16) == WS         # misaligned
    f = FakeDev(); assert f.call(lib, splits=2, ws_bytes=256) == WS
    f = FakeDev(rows=0); f.regions = f.t(4, (0, 8)); f.pos = f.t(4, (0,)); f.act = f.t(5, (0,))
    f.q = f.t(1, (0, 16, 192)); f.out = f.t(1, (0, 16, 192))
    assert f.call(lib) == B.SDA_OK                              # no rows: nothing to do


def test_status_strings(lib):
    for code in range(7):
        assert sda.status_string(code)
    assert "unknown" in sda.status_string(99)


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle, and a missing library raises."""
    import sys
    src_dir = os.path.dirname(sda.__file__)
    for name in os.listdir(src_dir):
        if name.endswith(".py"):
            text = open(os.path.join(src_dir, name)).read()
            assert "import oracle" not in text and "from oracle" not in text, name
    saved = B._lib, B.LIB_PATH
    try:
        B._lib, B.LIB_PATH = None, "/nonexistent/libsdattn.so"
        with pytest.raises(ImportError):
            B.load()
    finally:
        B._lib, B.LIB_PATH = saved


def test_swa_entry_validation(lib):
    INV, UNS = B.SDA_ERR_INVALID, B.SDA_ERR_UNSUPPORTED
    f = FakeDev()
    seq = f.t(4, (4,))
    r = ctypes.byref

    def call(window=256, seq_desc=seq, splits=1, cache=None, ql=1):
        ws = lib.sparse_decode_workspace_bytes(f.rows, f.H, splits)
        return lib.sparse_decode_swa_attention(r(f.q), r(cache or f.cache), r(f.table),
                                               r(seq_desc) if seq_desc is not None else None, r(f.out),
                                               0.07, window, ql, splits, None, None, None, 1 << 24, ws, None)
    assert call(window=0) == INV
    assert call(seq_desc=None) == INV
    assert call(seq_desc=f.t(4, (3,))) == INV                 # fewer lengths than requests
    assert call(seq_desc=f.t(1, (4,))) == INV                 # wrong dtype
    assert call(window=(1 << 30) + 1) == INV
    assert call(cache=f.t(1, (64, 2, 12, 384))) == UNS       # piece 12: not a multiple of 8
    assert sda.sparse_decode_swa_splits(2048, 4096) == 1
    assert sda.sparse_decode_swa_splits(4, 100) == 1
    assert sda.sparse_decode_swa_splits(64, 8192) == 4


def test_select_entry_validation(lib):
    INV = B.SDA_ERR_INVALID
    f = FakeDev()
    r = ctypes.byref
    sc, cur, ln, out = f.t(6, (8, 100)), f.t(4, (8,)), f.t(4, (8,)), f.t(4, (8, 16))

    def call(scores=sc, current=cur, lengths=ln, topk=16, regions=out):
        return lib.sparse_decode_select_regions(r(scores), r(current), r(lengths) if lengths else None,
                                                topk, r(regions), None)
    assert call(topk=0) == INV
    assert call(scores=f.t(1, (8, 100))) == INV                 # scores must be fp32
    assert call(scores=f.t(6, (8, 100), (200, 2))) == INV       # inner stride
    assert call(current=f.t(4, (7,))) == INV
    assert call(regions=f.t(4, (8, 15))) == INV                 # width != topk
    assert call(lengths=f.t(1, (8,))) == INV
    z = f.t(6, (0, 100))
    assert call(scores=z, current=f.t(4, (0,)), lengths=None, regions=f.t(4, (0, 16))) == B.SDA_OK


def test_summary_entry_validation(lib):
    INV, UNS, WS = B.SDA_ERR_INVALID, B.SDA_ERR_UNSUPPORTED, B.SDA_ERR_WORKSPACE
    f = FakeDev()
    r = ctypes.byref
    T, G = 8, 2
    q, w = f.t(2, (T, G, 8, 256)), f.t(6, (T, G, 8))
    m, bt, sl = f.t(3, (100, G, 256)), f.t(4, (4, 16)), f.t(4, (4,))
    sc, cur, ln = f.t(6, (T * G, 128)), f.t(4, (T * G,)), f.t(4, (T * G,))

    def call(query=q, weights=w, summ=m, table=bt, seq=sl, block=16, ql=2, scores=sc, current=cur,
             lengths=ln, ws=None, wsb=0):
        return lib.sparse_decode_summary_scores(r(query), r(weights), r(summ), r(table), r(seq), block, ql,
                                                r(scores), r(current) if current else None,
                                                r(lengths) if lengths else None, ws, wsb, None)
    assert call(block=12) == INV                                # block not a multiple of 8
    assert call(ql=0) == INV
    assert call(ql=3) == INV                                    # tokens not a multiple of query_len
    assert call(query=f.t(2, (T, G, 16, 256))) == INV           # 8 index heads
    assert call(query=f.t(2, (T, G, 8, 128))) == INV            # 256 dims
    assert call(query=f.t(1, (T, G, 8, 256))) == INV            # FP8 bytes only
    assert call(query=f.t(2, (T, G, 8, 256), (G * 4096, 4096, 512, 1))) == INV   # head stride
    assert call(weights=f.t(6, (T, G, 4))) == INV
    assert call(weights=f.t(1, (T, G, 8))) == INV
    assert call(summ=f.t(3, (100, G + 1, 256))) == INV          # groups mismatch
    assert call(summ=f.t(3, (100, G, 256), (G * 256 + 8, 256, 1))) == UNS       # slot stride
    assert call(table=f.t(4, (3, 16))) == INV                   # fewer table rows than requests
    assert call(seq=f.t(4, (3,))) == INV
    assert call(scores=f.t(6, (T * G - 1, 128))) == INV
    assert call(scores=f.t(6, (T * G, 128), (256, 2))) == INV   # inner stride
    assert call(current=f.t(4, (T * G - 1,))) == INV
    assert call(lengths=f.t(1, (T * G,))) == INV
    assert call(ws=(1 << 24) + 16, wsb=4096) == WS             # misaligned workspace
    assert call(ws=1 << 24, wsb=128) == WS                     # too small
    assert call(query=f.t(2, (T, 1, 8, 256)), weights=f.t(6, (T, 1, 8)), summ=f.t(3, (100, 1, 256)),
                scores=f.t(6, (T, 128)), current=None, lengths=None, ql=8, table=f.t(4, (1, 16)),
                seq=f.t(4, (1,))) == UNS                        # query_len > 4
    z = dict(query=f.t(2, (0, G, 8, 256)), weights=f.t(6, (0, G, 8)), scores=f.t(6, (0, 128)),
             current=f.t(4, (0,)), lengths=f.t(4, (0,)))
    assert call(**z) == B.SDA_OK                                # no tokens: nothing to do


def test_binding_rejects_host_tensors(lib):
    """Host (CPU) tensors never reach the kernels: every Python entry raises before it
    allocates a workspace or calls into the library."""
    bf, i32 = torch.bfloat16, torch.int32
    q, out = torch.zeros(4, 16, 192, dtype=bf), torch.zeros(4, 16, 192, dtype=bf)
    cache = torch.zeros(8, 1, 16, 384, dtype=bf)
    regions, table = torch.zeros(4, 2, dtype=i32), torch.zeros(4, 2, dtype=i32)
    pos, act, seq = torch.zeros(4, dtype=i32), torch.ones(4, dtype=torch.bool), torch.ones(4, dtype=i32)
    calls = [
        lambda: sda.sparse_decode_attention(q, cache, regions, table, pos, act, out, scale=0.1, splits=1),
        lambda: sda.sparse_decode_attention_no_alloc(q, cache, regions, table, pos, act, out, scale=0.1,
                                                     splits=1),
        lambda: sda.sparse_decode_swa_attention(q, cache, table, seq, out, scale=0.1, window=4, splits=1),
        lambda: sda.sparse_decode_select_regions(torch.zeros(4, 8), pos, 2),
        lambda: sda.sparse_decode_summary_scores(torch.zeros(4, 1, 8, 256, dtype=torch.uint8),
                                                 torch.zeros(4, 1, 8), torch.zeros(16, 1, 256, dtype=torch.uint8),
                                                 table, seq, block_size=16),
        lambda: sda.read_errors(torch.zeros(256, dtype=torch.uint8)),
    ]
    before = dict(B._workspaces)
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    assert B._workspaces == before


def test_binding_device_resolution():
    """One device for all tensor arguments and the stream; None entries are skipped."""
    from types import SimpleNamespace as NS
    c0, c1 = torch.device("cuda", 0), torch.device("cuda", 1)
    assert B._device_of(NS(device=c0), None, NS(device=c0)) == c0
    with pytest.raises(ValueError, match="one device"):
        B._device_of(NS(device=c0), NS(device=c1))
    with pytest.raises(ValueError, match="stream"):
        B._device_of(NS(device=c0), stream=NS(device=c1))
    with pytest.raises(ValueError, match="CUDA tensor"):
        B._device_of(NS(device=c0), NS(device=torch.device("meta")))
    with pytest.raises(ValueError, match="no tensor"):
        B._device_of(None)


def test_swa_splits_policy(lib):
    """The window split policy as include/sdattn.h states it: the sparse path's split count for
    the row count (its golden truth table), halved while a split would cover fewer than 256
    window tokens."""
    table = []
    with open(os.path.join(GOLDEN, "sparse_decode_splits.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                table.append(tuple(int(x) for x in line))
    for lo, hi, s in table:
        for rows in sorted({lo, hi, (lo + hi) // 2}):
            for window in (1, 100, 255, 256, 257, 511, 512, 1024, 2048, 4096, 8192, 1 << 20):
                want = s
                while want > 1 and window // want < 256:
                    want //= 2
                assert sda.sparse_decode_swa_splits(rows, window) == want, (rows, window)


def test_timeline_entry_point_is_a_stub_in_the_regular_library():
    """The phase stamps exist only in a diagnostic build (SDA_TIMELINE); the regular
    library refuses the buffer without touching the GPU."""
    import ctypes
    from sparse_decode_attention_02_gb300 import _binding as B
    lib = B.load()
    assert lib.sparse_decode_timeline_buffer(None, 0) == B.SDA_ERR_UNSUPPORTED
    assert lib.sparse_decode_timeline_buffer(ctypes.c_void_p(16), 1 << 30) == B.SDA_ERR_UNSUPPORTED
