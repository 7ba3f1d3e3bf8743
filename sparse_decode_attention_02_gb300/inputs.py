"""Seeded synthetic workloads for sparse decode attention (no attention arithmetic here).

Both the CUDA path and the CPU oracle are fed from this module; it only draws
random numbers and lays them out.  The five workloads follow the decode
shapes of the vLLM page "vllm.models.step5.nvidia.ops.sparse_decode_attention"
(`sparse_decode_attention` docstring: query/output [rows, heads, 192],
cache [pages, G, block, 384] with K then V, regions [rows, R] with -1 unused,
per-row positions and active flags, G * query_len rows per request sharing one
block_table row):

  tiny    4 tokens, G=1, 8 heads, bf16, block = region = 16, R=4, 32 pages
  gqa     64 requests, G=2, 16 heads, bf16, block = region = 64, R=32, ctx 8K-32K
  fp8     128 requests, G=2, 16 heads, FP8 E4M3, R=32, ctx 32K-64K, gate, 5% inactive
  spec    256 requests x 2 query tokens, G=4, bf16, R=64 with 0-16 -1 pads, gate, 8% inactive
  large   512 requests, G=4, FP8 E4M3, R=128 (half recent, half older), ctx 128K-256K
  swa     256 requests x 2 query tokens, G=4, bf16, sliding window 4096, ctx 16K-64K, gate
          (the non-DSA layers' fused gated sliding-window decode; no regions)

Integer metadata (positions, regions, block tables, active flags) comes from
numpy's PCG64 seeded with the workload index, so it is identical on every
device; values (q, K, V, gate) come from a seeded torch generator on the
device the workload is built on.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

DIM = 192
ROW = 384
FP8_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    requests: int
    query_len: int
    groups: int
    heads: int
    block: int
    region_tokens: int
    num_regions: int
    ctx: tuple[int, int] | None      # context length range (inclusive); None = tiny layout
    fp8: bool = False
    gate: bool = False
    inactive_frac: float = 0.0
    short_frac: float = 0.0          # rows with fewer live regions (tail -1)
    pad_max: int = 0                 # rows get U{0..pad_max} -1 entries at random slots
    selection: str = "uniform"       # "uniform" | "recent_half"
    splits: int | None = None        # None: the library's sparse_decode_splits(rows)
    seed: int = 0
    window: int = 0                  # > 0: sliding-window decode workload (no regions)

    @property
    def rows(self) -> int:
        return self.requests * self.query_len * self.groups

    @property
    def tokens(self) -> int:
        return self.requests * self.query_len


CONFIGS = {
    "tiny": Config("tiny", requests=4, query_len=1, groups=1, heads=8, block=16, region_tokens=16,
                   num_regions=4, ctx=None, splits=1, seed=0),
    "gqa": Config("gqa", requests=64, query_len=1, groups=2, heads=16, block=64, region_tokens=64,
                  num_regions=32, ctx=(8 * 1024, 32 * 1024), short_frac=0.10, seed=1),
    "fp8": Config("fp8", requests=128, query_len=1, groups=2, heads=16, block=64, region_tokens=64,
                  num_regions=32, ctx=(32 * 1024, 64 * 1024), fp8=True, gate=True,
                  inactive_frac=0.05, seed=2),
    "spec": Config("spec", requests=256, query_len=2, groups=4, heads=16, block=64, region_tokens=64,
                   num_regions=64, ctx=(64 * 1024, 128 * 1024), gate=True, inactive_frac=0.08,
                   pad_max=16, seed=3),
    "large": Config("large", requests=512, query_len=1, groups=4, heads=16, block=64,
                    region_tokens=64, num_regions=128, ctx=(128 * 1024, 256 * 1024), fp8=True,
                    selection="recent_half", seed=4),
    "swa": Config("swa", requests=256, query_len=2, groups=4, heads=16, block=64, region_tokens=64,
                  num_regions=0, ctx=(16 * 1024, 64 * 1024), gate=True, window=4096, seed=5),
}
ORDER = ["tiny", "gqa", "fp8", "spec", "large", "swa"]


@dataclasses.dataclass
class Workload:
    config: Config
    query: torch.Tensor          # [rows, H, 192] bf16
    cache: torch.Tensor          # [pages, G, B, 384] bf16 or uint8 (E4M3 bytes)
    regions: torch.Tensor        # [rows, R] int32
    block_table: torch.Tensor    # [requests, W] int32
    positions: torch.Tensor      # [rows] int32
    active: torch.Tensor         # [rows] uint8
    gate: torch.Tensor | None    # [tokens, G*H] bf16
    k_scale: float | None
    v_scale: float | None
    scale: float
    splits: int | None           # forced split count, or None for the library's policy
    filled_tiles: np.ndarray     # [n, 2] (page, group) tiles holding generated K|V
    seq_lens: torch.Tensor       # [requests] int32 context lengths (tokens incl. the decoded ones)

    @property
    def window(self) -> int:
        return self.config.window

    @property
    def rows(self) -> int:
        return self.query.shape[0]

    @property
    def fp8(self) -> bool:
        return self.cache.dtype == torch.uint8

    @property
    def heads(self) -> int:
        return self.query.shape[1]

    @property
    def groups(self) -> int:
        return self.cache.shape[1]

    @property
    def block(self) -> int:
        return self.cache.shape[2]

    @property
    def query_len(self) -> int:
        return self.config.query_len

    @property
    def region_tokens(self) -> int:
        return self.config.region_tokens


# ----------------------------------------------------------------------------
# Integer metadata (numpy, device independent)
# ----------------------------------------------------------------------------

def _positions(cfg: Config, rng: np.random.Generator):
    """Per-request context lengths L and per-row positions: token j of a request
    with query_len tokens sits at L - query_len + j (0-based)."""
    if cfg.ctx is None:                      # tiny: positions uniform in [40, 500]
        pos_tok = rng.integers(40, 501, size=cfg.tokens)
        lengths = pos_tok + 1
    else:
        lengths = rng.integers(cfg.ctx[0], cfg.ctx[1] + 1, size=cfg.requests)
        pos_tok = np.concatenate([L - cfg.query_len + np.arange(cfg.query_len) for L in lengths])
    pos_rows = np.repeat(pos_tok, cfg.groups).astype(np.int32)
    return lengths.astype(np.int64), pos_rows


def _select(cfg: Config, rng: np.random.Generator, pos: int, live: int) -> np.ndarray:
    """`live` distinct region ids visible at `pos`, the current one always included."""
    cur = pos // cfg.region_tokens
    if cfg.selection == "recent_half":
        half = live // 2
        lo = max(0, cur - 511)
        recent = rng.choice(np.arange(lo, cur), size=min(half - 1, cur - lo), replace=False)
        older = rng.choice(lo, size=min(live - half, lo), replace=False) if lo else np.zeros(0, np.int64)
        ids = np.concatenate([[cur], recent, older])
    else:
        k = min(live - 1, cur)
        ids = np.concatenate([[cur], rng.choice(cur, size=k, replace=False) if k else []])
    ids = ids.astype(np.int64)
    rng.shuffle(ids)                            # selection is unsorted
    return ids


def _regions(cfg: Config, rng: np.random.Generator, pos_rows: np.ndarray) -> np.ndarray:
    R = cfg.num_regions
    out = np.full((cfg.rows, R), -1, dtype=np.int32)
    short = np.zeros(cfg.rows, dtype=bool)
    if cfg.short_frac:
        short[rng.choice(cfg.rows, size=int(round(cfg.short_frac * cfg.rows)), replace=False)] = True
    for r in range(cfg.rows):
        if cfg.pad_max:
            live = R - int(rng.integers(0, cfg.pad_max + 1))
        elif short[r]:
            live = int(rng.integers(1, R))
        else:
            live = R
        ids = _select(cfg, rng, int(pos_rows[r]), live)
        if cfg.pad_max:                         # -1 entries at random slots
            slots = np.sort(rng.choice(R, size=len(ids), replace=False))
            out[r, slots] = ids
        else:                                    # -1 entries at the tail
            out[r, :len(ids)] = ids
    return out


def _block_table(cfg: Config, rng: np.random.Generator, lengths: np.ndarray):
    """[requests, W] int32 page ids (-1 past a request's blocks) and the pool size."""
    if cfg.ctx is None:                          # tiny: each request row an independent
        pages = 32                               # permutation of all 32 pages
        table = np.stack([rng.permutation(pages) for _ in range(cfg.requests)]).astype(np.int32)
        return table, pages
    nblocks = (lengths + cfg.block - 1) // cfg.block
    pages = int(nblocks.sum())
    pool = rng.permutation(pages).astype(np.int32)   # shuffled page pool
    width = int(nblocks.max())
    table = np.full((cfg.requests, width), -1, dtype=np.int32)
    off = 0
    for q, n in enumerate(nblocks):
        table[q, :n] = pool[off:off + n]
        off += n
    return table, pages


def _active(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    act = np.ones(cfg.rows, dtype=np.uint8)
    if cfg.inactive_frac:
        act[rng.choice(cfg.rows, size=int(round(cfg.inactive_frac * cfg.rows)), replace=False)] = 0
    return act


def referenced_tiles(cfg: Config, regions: np.ndarray, table: np.ndarray, pos_rows: np.ndarray) -> np.ndarray:
    """Distinct (page, group) tiles holding any token of any listed region.

    Row r reads group r % G of request r // (G * query_len); a region id covers
    blocks [id*RT // B, ((id+1)*RT - 1) // B]."""
    rows = np.arange(cfg.rows)
    req = rows // (cfg.groups * cfg.query_len)
    grp = rows % cfg.groups
    RT, B = cfg.region_tokens, cfg.block
    per_region = max(1, (RT + B - 1) // B)
    tiles = []
    ids = regions.astype(np.int64)
    live = ids >= 0
    for j in range(per_region):
        col = (ids * RT) // B + j
        ok = live & (col * B < (ids + 1) * RT) & (col < table.shape[1])
        rr, cc = np.nonzero(ok)
        page = table[req[rr], col[rr, cc]]
        good = page >= 0
        tiles.append(np.stack([page[good], grp[rr][good]], axis=1))
    t = np.concatenate(tiles).astype(np.int64)
    return np.unique(t, axis=0)


def window_columns(pos: int, window: int, block: int) -> range:
    """Block-table columns holding the tokens [max(0, pos - window + 1), pos]."""
    if pos < 0:
        return range(0)
    lo = max(0, pos - window + 1)
    return range(lo // block, pos // block + 1)


def window_tiles(cfg: Config, table: np.ndarray, pos_rows: np.ndarray) -> np.ndarray:
    """Distinct (page, group) tiles some row's window touches."""
    tiles = set()
    per_req = cfg.groups * cfg.query_len
    for r in range(cfg.rows):
        req, g = r // per_req, r % cfg.groups
        for col in window_columns(int(pos_rows[r]), cfg.window, cfg.block):
            page = int(table[req, col])
            if page >= 0:
                tiles.add((page, g))
    return np.array(sorted(tiles), dtype=np.int64).reshape(-1, 2)


# ----------------------------------------------------------------------------
# Values (torch, on the target device)
# ----------------------------------------------------------------------------

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _fill_tiles(cache: torch.Tensor, tiles: np.ndarray, cfg: Config, seed: int, fp8: bool,
                chunk: int = 4096):
    """Write N(0,1) K|V into the listed (page, group) tiles; FP8 caches get the
    per-tensor scales amax/448 (K and V separately) and saturated E4M3 bytes.
    Returns (k_scale, v_scale) or (None, None)."""
    dev = cache.device
    B = cfg.block
    n = len(tiles)
    if n == 0:
        return (1.0, 1.0) if fp8 else (None, None)
    t_page = torch.as_tensor(tiles[:, 0], device=dev)
    t_grp = torch.as_tensor(tiles[:, 1], device=dev)

    def values(i0, i1):
        g = _gen(dev, seed * 1_000_003 + i0)
        return torch.randn((i1 - i0, B, ROW), generator=g, device=dev, dtype=torch.float32)

    if not fp8:
        for i0 in range(0, n, chunk):
            i1 = min(n, i0 + chunk)
            cache[t_page[i0:i1], t_grp[i0:i1]] = values(i0, i1).to(torch.bfloat16)
        return None, None
    kmax = torch.zeros((), device=dev)
    vmax = torch.zeros((), device=dev)
    for i0 in range(0, n, chunk):               # pass 1: per-tensor amax
        v = values(i0, min(n, i0 + chunk))
        kmax = torch.maximum(kmax, v[..., :DIM].abs().amax())
        vmax = torch.maximum(vmax, v[..., DIM:].abs().amax())
    k_scale = float(kmax) / FP8_MAX
    v_scale = float(vmax) / FP8_MAX
    div = torch.tensor([k_scale] * DIM + [v_scale] * DIM, device=dev, dtype=torch.float32)
    for i0 in range(0, n, chunk):               # pass 2: regenerate and quantise
        i1 = min(n, i0 + chunk)
        q = (values(i0, i1) / div).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
        cache[t_page[i0:i1], t_grp[i0:i1]] = q.view(torch.uint8)
    return k_scale, v_scale


def make_workload(cfg: Config | str, device="cpu", *, splits: int | None = None,
                  fill: str = "referenced", page_stride_pad: int = 0) -> Workload:
    """Build one workload on `device`.

    fill="referenced" writes only the (page, group) tiles some row's regions
    touch (the rest of the pool stays uninitialised, as in a serving cache);
    fill="all" writes every tile.  page_stride_pad > 0 allocates each page with
    that many extra elements, giving a padded page stride as in a cache whose
    pages hold more than this layer's KV."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rng = np.random.default_rng(cfg.seed)
    lengths, pos_rows = _positions(cfg, rng)
    table, pages = _block_table(cfg, rng, lengths)
    if cfg.window:
        regions = np.zeros((cfg.rows, 0), dtype=np.int32)
    else:
        regions = _regions(cfg, rng, pos_rows)
    active = _active(cfg, rng)

    dev = torch.device(device)
    g = _gen(dev, cfg.seed)
    query = torch.randn((cfg.rows, cfg.heads, DIM), generator=g, device=dev).to(torch.bfloat16)
    gate = None
    if cfg.gate:
        gate = (2.0 * torch.randn((cfg.tokens, cfg.groups * cfg.heads), generator=g, device=dev)
                ).to(torch.bfloat16)

    dtype = torch.uint8 if cfg.fp8 else torch.bfloat16
    page_elems = cfg.groups * cfg.block * ROW
    if page_stride_pad:
        flat = torch.empty((pages, page_elems + page_stride_pad), dtype=dtype, device=dev)
        cache = flat[:, :page_elems].view(pages, cfg.groups, cfg.block, ROW)
    else:
        cache = torch.empty((pages, cfg.groups, cfg.block, ROW), dtype=dtype, device=dev)
    if fill == "all":
        pg, gr = np.meshgrid(np.arange(pages), np.arange(cfg.groups), indexing="ij")
        tiles = np.stack([pg.ravel(), gr.ravel()], axis=1)
    elif cfg.window:
        tiles = window_tiles(cfg, table, pos_rows)
    else:
        tiles = referenced_tiles(cfg, regions, table, pos_rows)
    k_scale, v_scale = _fill_tiles(cache, tiles, cfg, cfg.seed + 7919, cfg.fp8)

    return Workload(
        config=cfg, query=query, cache=cache,
        regions=torch.as_tensor(regions, device=dev),
        block_table=torch.as_tensor(table, device=dev),
        positions=torch.as_tensor(pos_rows, device=dev),
        active=torch.as_tensor(active, device=dev),
        gate=gate, k_scale=k_scale, v_scale=v_scale,
        scale=1.0 / math.sqrt(DIM),
        splits=splits or cfg.splits,
        filled_tiles=tiles,
        seq_lens=torch.as_tensor(lengths.astype(np.int32), device=dev),
    )


def scaled(cfg: Config | str, **changes) -> Config:
    """A copy of a workload configuration with some fields changed (smaller test sizes)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    return dataclasses.replace(cfg, **changes)


# ----------------------------------------------------------------------------
# Host copies for the oracle
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class HostProblem:
    """The arguments of an oracle call for a subset of a workload's rows.

    Row r of the workload becomes row i*G*query_len + r % (G*query_len) of the
    host problem (request i), so its group, token-in-request and gate column
    are unchanged; `row_ids` lists those rows.  The cache holds one tile per
    (page, group) the rows' regions touch; its group stride is 0 so every
    group index of a host page reads that tile."""
    query: torch.Tensor
    cache: torch.Tensor
    regions: torch.Tensor
    block_table: torch.Tensor
    positions: torch.Tensor
    active: torch.Tensor
    gate: torch.Tensor | None
    row_ids: np.ndarray
    kwargs: dict
    seq_lens: torch.Tensor       # [n] per host request (window workloads)


def host_subset(w: Workload, rows) -> HostProblem:
    """Host copies for the oracle of `rows` (regions for the sparse path; the
    window's blocks plus per-request seq_lens for a window workload)."""
    cfg = w.config
    rows = np.asarray(rows, dtype=np.int64)
    n = len(rows)
    G, ql = w.groups, w.query_len
    per_req = G * ql
    new_rows = np.arange(n) * per_req + rows % per_req

    regions = w.regions[torch.as_tensor(rows, device=w.regions.device)].cpu().numpy()
    positions = w.positions.cpu().numpy()[rows]
    table = w.block_table.cpu().numpy()
    req = rows // per_req
    grp = rows % G
    RT, B = w.region_tokens, w.block
    per_region = max(1, (RT + B - 1) // B)

    # host page k <- device tile (page, group); columns of each host request
    tiles = {}
    host_table = np.full((n, table.shape[1]), -1, dtype=np.int32)
    for i in range(n):
        if w.window:
            cols = list(window_columns(int(positions[i]), w.window, B))
        else:
            cols = []
            for rid in regions[i]:
                if rid < 0:
                    continue
                for j in range(per_region):
                    col = (int(rid) * RT) // B + j
                    if col < table.shape[1] and col * B < (int(rid) + 1) * RT:
                        cols.append(col)
        for col in cols:
            page = int(table[req[i], col])
            if page < 0:
                continue
            key = (page, int(grp[i]))
            k = tiles.setdefault(key, len(tiles))
            host_table[i, col] = k
    keys = np.array(list(tiles.keys()), dtype=np.int64).reshape(-1, 2)
    if len(keys):
        dev = w.cache.device
        data = w.cache[torch.as_tensor(keys[:, 0], device=dev), torch.as_tensor(keys[:, 1], device=dev)].cpu()
    else:
        data = torch.zeros((1, B, ROW), dtype=w.cache.dtype)
    cache = data.unsqueeze(1).expand(data.shape[0], G, B, ROW)   # group stride 0

    total = n * per_req
    query = torch.zeros((total, w.heads, DIM), dtype=torch.bfloat16)
    query[new_rows] = w.query[torch.as_tensor(rows, device=w.query.device)].cpu()
    reg = torch.full((total, regions.shape[1]), -1, dtype=torch.int32)
    reg[new_rows] = torch.as_tensor(regions)
    pos = torch.zeros(total, dtype=torch.int32)
    pos[new_rows] = torch.as_tensor(positions)
    act = torch.zeros(total, dtype=torch.uint8)
    act[new_rows] = w.active.cpu()[torch.as_tensor(rows)]
    gate = None
    if w.gate is not None:
        gate = torch.zeros((total // G, w.gate.shape[1]), dtype=torch.bfloat16)
        gate[torch.as_tensor(new_rows // G)] = w.gate.cpu()[torch.as_tensor(rows // G)]
    kwargs = dict(scale=w.scale, query_len=ql, region_tokens=RT,
                  k_scale=w.k_scale, v_scale=w.v_scale, cache_fp8=w.fp8)
    seq = w.seq_lens.cpu().numpy()[req].astype(np.int32)
    return HostProblem(query, cache, reg, torch.as_tensor(host_table), pos, act, gate,
                       new_rows.astype(np.int32), kwargs, torch.as_tensor(seq))


# ----------------------------------------------------------------------------
# Region-selection inputs
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class SelectWorkload:
    scores: torch.Tensor         # [rows, N] fp32 region scores
    current: torch.Tensor        # [rows] int32 region holding the row's token
    lengths: torch.Tensor        # [rows] int32 candidate count (regions up to the token)
    topk: int

    @property
    def rows(self) -> int:
        return self.scores.shape[0]


def make_select_workload(device="cpu", *, requests=512, groups=4, ctx=(128 * 1024, 256 * 1024),
                         region_tokens=8, topk=1024, seed=6) -> SelectWorkload:
    """Decode-row region scores shaped like the large workload's rows: one row per
    (token, KV group), ids of `region_tokens`-token regions up to the token's
    position, scores N(0,1)."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(ctx[0], ctx[1] + 1, size=requests)
    pos = np.repeat(lengths - 1, groups)
    cur = (pos // region_tokens).astype(np.int32)
    n_len = (cur + 1).astype(np.int32)
    dev = torch.device(device)
    g = _gen(dev, seed)
    scores = torch.randn((len(pos), int(n_len.max())), generator=g, device=dev)
    return SelectWorkload(scores, torch.as_tensor(cur, device=dev), torch.as_tensor(n_len, device=dev), topk)


# ----------------------------------------------------------------------------
# Indexer-score inputs
# ----------------------------------------------------------------------------

INDEX_HEADS = 8
INDEX_DIM = 256


@dataclasses.dataclass
class IndexWorkload:
    query: torch.Tensor          # [tokens, G, 8, 256] float8_e4m3fn index queries
    weights: torch.Tensor        # [tokens, G, 8] fp32 head weights
    summaries: torch.Tensor      # [pages * block / 8, G, 256] float8_e4m3fn region summaries
    block_table: torch.Tensor    # [requests, W] int32, -1 past the request's pages
    seq_lens: torch.Tensor       # [requests] int32
    block: int
    query_len: int
    n_cols: int                  # score columns per row

    @property
    def tokens(self) -> int:
        return self.query.shape[0]

    @property
    def groups(self) -> int:
        return self.query.shape[1]

    @property
    def rows(self) -> int:
        return self.tokens * self.groups


def _e4m3_normal(shape, gen, device, std=1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std
    return x.clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)


def make_index_workload(device="cpu", *, requests=512, groups=4, query_len=1,
                        ctx=(128 * 1024, 256 * 1024), block=64, n_cols=None, spare_pages=64,
                        seed=7, chunk_slots=1 << 20) -> IndexWorkload:
    """Indexer inputs for decode rows: request lengths U[ctx], each request's
    pages drawn from one shuffled pool (plus `spare_pages` unused ones), E4M3
    index queries and summaries from N(0,1), head weights N(0,1)/16.  The
    default matches the large workload's rows: 512 requests x 4 KV groups,
    contexts 128K-256K, 64-token pages, 8-token regions (32K score columns)."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(ctx[0], ctx[1] + 1, size=requests).astype(np.int64)
    n_pages = -(-lengths // block)
    width = int(n_pages.max()) if requests else 1
    pool = int(n_pages.sum()) + spare_pages
    order = rng.permutation(pool).astype(np.int32)
    table = np.full((requests, width), -1, dtype=np.int32)
    at = 0
    for r in range(requests):
        k = int(n_pages[r])
        table[r, :k] = order[at:at + k]
        at += k
    if n_cols is None:
        n_cols = width * block // 8
    dev = torch.device(device)
    gen = _gen(dev, seed)
    tokens = requests * query_len
    query = _e4m3_normal((tokens, groups, INDEX_HEADS, INDEX_DIM), gen, dev)
    weights = torch.randn((tokens, groups, INDEX_HEADS), generator=gen, device=dev) / 16
    slots = pool * (block // 8)
    summaries = torch.empty((slots, groups, INDEX_DIM), dtype=torch.float8_e4m3fn, device=dev)
    for s0 in range(0, slots, chunk_slots):
        s1 = min(slots, s0 + chunk_slots)
        summaries[s0:s1] = _e4m3_normal((s1 - s0, groups, INDEX_DIM), _gen(dev, seed * 7919 + s0), dev)
    return IndexWorkload(query, weights, summaries, torch.as_tensor(table, device=dev),
                         torch.as_tensor(lengths.astype(np.int32), device=dev), block, query_len,
                         int(n_cols))


def index_host_subset(w: IndexWorkload, requests) -> IndexWorkload:
    """Host copy of the listed requests (all their tokens and groups), their pages
    renumbered densely: the oracle's input for sampled rows of a large workload.
    Row k * G * query_len + i of the subset is row req_k * G * query_len + i."""
    requests = [int(r) for r in requests]
    table = w.block_table.cpu().numpy()
    per_page = w.block // 8
    used = sorted({int(p) for r in requests for p in table[r] if p >= 0})
    remap = {p: i for i, p in enumerate(used)}
    new_table = np.full((len(requests), table.shape[1]), -1, dtype=np.int32)
    for k, r in enumerate(requests):
        for c, p in enumerate(table[r]):
            if p >= 0:
                new_table[k, c] = remap[int(p)]
    page_ids = torch.as_tensor(used, dtype=torch.int64, device=w.summaries.device)
    pages = w.summaries.view(-1, per_page, w.groups, INDEX_DIM)[page_ids]
    toks = torch.as_tensor([r * w.query_len + i for r in requests for i in range(w.query_len)],
                           device=w.query.device)
    return IndexWorkload(w.query[toks].cpu(), w.weights[toks].cpu(),
                         pages.reshape(-1, w.groups, INDEX_DIM).cpu(), torch.as_tensor(new_table),
                         w.seq_lens.cpu()[torch.as_tensor(requests)], w.block, w.query_len, w.n_cols)


@dataclasses.dataclass
class DecodeChain:
    """The inputs of one DSA decode step: indexer operands, and the attention
    operands over the same pages (FP8 K|V cache, 16 query heads per group)."""
    index: IndexWorkload
    cache: torch.Tensor          # [pages, G, block, 384] float8_e4m3fn
    k_scale: float
    v_scale: float
    query: torch.Tensor          # [rows, 16, 192] bf16
    positions: torch.Tensor      # [rows] int32
    active: torch.Tensor         # [rows] bool
    topk: int
    scale: float = DIM ** -0.5


def make_decode_chain(device="cpu", *, requests=512, groups=4, query_len=1,
                      ctx=(128 * 1024, 256 * 1024), block=64, topk=1024, heads=16, seed=8,
                      chunk_pages=1 << 14, **index_kw) -> DecodeChain:
    """A decode step over the large workload's requests: every page of the pool
    holds N(0,1) K|V as E4M3 with scale 8/448 (saturating beyond 8 sigma) and
    its 8-token region summaries; the selection keeps `topk` 8-token regions
    (1024 x 8 = 8192 tokens, the large workload's selected tokens per row)."""
    idx = make_index_workload(device, requests=requests, groups=groups, query_len=query_len, ctx=ctx,
                              block=block, seed=seed, **index_kw)
    dev = torch.device(device)
    pages = idx.summaries.shape[0] // (block // 8)
    cache = torch.empty((pages, groups, block, ROW), dtype=torch.float8_e4m3fn, device=dev)
    s = 8.0 / FP8_MAX
    for p0 in range(0, pages, chunk_pages):
        p1 = min(pages, p0 + chunk_pages)
        x = torch.randn((p1 - p0, groups, block, ROW), generator=_gen(dev, seed * 104729 + p0), device=dev)
        cache[p0:p1] = (x / s).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
        del x
    g = _gen(dev, seed + 1)
    rows = idx.rows
    query = torch.randn((rows, heads, DIM), generator=g, device=dev).to(torch.bfloat16)
    seq = idx.seq_lens.to(torch.int64)
    tok = torch.arange(idx.tokens, device=dev)
    pos = (seq[tok // query_len] - query_len + tok % query_len).repeat_interleave(groups)
    return DecodeChain(idx, cache, s, s, query, pos.to(torch.int32),
                       torch.ones(rows, dtype=torch.bool, device=dev), topk)
