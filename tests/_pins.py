"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle library handle (the normal build or a
build with one planted mistake) and raises AssertionError when the oracle
disagrees with an independent fact:

  * torch's own E4M3 and bf16 decoders and its RNE bf16 cast;
  * torch's float64 scaled_dot_product_attention over a dense K/V sequence
    that this file scatters into pages itself (never through the oracle);
  * closed forms (one visible token returns V exactly; a zero query averages V);
  * invariants (region order, -1 placement, row permutation, split merging);
  * the split-count truth table derived by hand from the page's loop;
  * for the indexer scores, dense torch matrix products over summaries this
    file scatters into pages, one-hot closed forms and linearity in the weights.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# Dense problems scattered into a paged cache by this file alone
# ---------------------------------------------------------------------------

class Dense:
    """A small problem whose K/V exist as dense per-(request, group) sequences.

    Pages are assigned from a shuffled pool (plus unused decoy pages filled
    with NaN so a wrong page index cannot go unnoticed); every row selects all
    of its visible regions, in random order, padded with -1."""

    def __init__(self, seed, *, reqs=3, query_len=1, G=2, H=4, B=16, RT=16, lengths=None,
                 fp8=False, gate=False, extra_slots=3, page_pad=0):
        rng = np.random.default_rng(seed)
        self.reqs, self.ql, self.G, self.H, self.B, self.RT = reqs, query_len, G, H, B, RT
        self.fp8 = fp8
        if lengths is None:
            lengths = rng.integers(query_len + 1, 6 * B, size=reqs)
        self.lengths = np.asarray(lengths)
        nblk = (self.lengths + B - 1) // B
        used = int(nblk.sum())
        pages = used + 4                                   # 4 decoy pages
        pool = rng.permutation(pages)
        W = int(nblk.max()) + 1
        table = np.full((reqs, W), -1, np.int32)
        off = 0
        for q in range(reqs):
            table[q, :nblk[q]] = pool[off:off + nblk[q]]
            off += nblk[q]
        decoys = pool[off:]
        self.table = table

        # dense K|V: [req][g] -> [L, 384]
        self.kv_bytes = []
        self.kv = []
        if fp8:
            codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
            self.k_scale, self.v_scale = 0.013, 0.021
        else:
            self.k_scale = self.v_scale = None
        for q in range(reqs):
            row = []
            rowb = []
            for g in range(G):
                L = int(self.lengths[q])
                if fp8:
                    b = rng.choice(codes, size=(L, 384))
                    t = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64)
                    t[:, :192] *= self.k_scale
                    t[:, 192:] *= self.v_scale
                else:
                    b = torch.randn(L, 384, generator=torch.Generator().manual_seed(seed * 97 + q * 7 + g)
                                    ).to(torch.bfloat16)
                    t = b.to(torch.float64)
                rowb.append(b)
                row.append(t)
            self.kv.append(row)
            self.kv_bytes.append(rowb)

        dtype = torch.uint8 if fp8 else torch.bfloat16
        per_page = G * B * 384
        flat = torch.zeros((pages, per_page + page_pad), dtype=dtype)
        cache = flat[:, :per_page].view(pages, G, B, 384)
        if fp8:
            cache.fill_(0x7F)                  # NaN everywhere not written below
        else:
            cache.fill_(float("nan"))
        for q in range(reqs):
            for g in range(G):
                L = int(self.lengths[q])
                src = self.kv_bytes[q][g]
                for t in range(L):
                    p = table[q, t // B]
                    if fp8:
                        cache[p, g, t % B] = torch.from_numpy(np.ascontiguousarray(src[t]))
                    else:
                        cache[p, g, t % B] = src[t]
        self.cache = cache
        self.decoys = decoys

        rows = reqs * query_len * G
        self.rows = rows
        self.query = torch.randn(rows, H, 192, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
        pos = np.zeros(rows, np.int32)
        for r in range(rows):
            q = r // (G * query_len)
            j = (r // G) % query_len
            pos[r] = self.lengths[q] - query_len + j
        self.positions = pos
        nreg = [int(p) // RT + 1 for p in pos]
        R = max(nreg) + extra_slots
        regions = np.full((rows, R), -1, np.int32)
        for r in range(rows):
            ids = rng.permutation(nreg[r])
            slots = np.sort(rng.choice(R, size=nreg[r], replace=False))
            regions[r, slots] = ids
        self.regions = regions
        self.active = np.ones(rows, np.uint8)
        self.scale = 1.0 / math.sqrt(192)
        self.gate = None
        if gate:
            self.gate = (2 * torch.randn(rows // G, G * H, generator=torch.Generator().manual_seed(seed + 2))
                         ).to(torch.bfloat16)

    def oracle(self, lib=None, **kw):
        args = dict(scale=self.scale, query_len=self.ql, region_tokens=self.RT,
                    k_scale=self.k_scale, v_scale=self.v_scale, cache_fp8=self.fp8, lib=lib)
        args.update(kw)
        gate = args.pop("gate", self.gate)
        regions = args.pop("regions", self.regions)
        active = args.pop("active", self.active)
        positions = args.pop("positions", self.positions)
        return oracle.sparse_decode_attention(self.query, self.cache, regions, self.table,
                                              positions, active, gate=gate, **args)

    def textbook(self, r):
        """Causal decode attention of row r over tokens 0..pos, float64 SDPA on the dense sequence."""
        q = r // (self.G * self.ql)
        g = r % self.G
        pos = int(self.positions[r])
        kv = self.kv[q][g][:pos + 1]
        Q = self.query[r].to(torch.float64).unsqueeze(0)
        out = torch.nn.functional.scaled_dot_product_attention(
            Q, kv[:, :192].unsqueeze(0), kv[:, 192:].unsqueeze(0), scale=self.scale)
        return out[0].numpy()


def torch_gate(bits):
    """Reference gate factor(s): torch's fp32 sigmoid cast (RNE) to bf16."""
    b = np.atleast_1d(np.asarray(bits, dtype=np.uint16)).view(np.int16)
    g = torch.from_numpy(b.copy()).view(torch.bfloat16).float()
    out = torch.sigmoid(g).to(torch.bfloat16).double().numpy()
    return float(out[0]) if np.ndim(bits) == 0 else out


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------

def pin_e4m3_decode(lib):
    """All 256 codes against torch.float8_e4m3fn, plus the OCP format's landmark values."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_decode(c, lib) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)), "NaN codes differ"
    assert np.array_equal(ref[~nan], got[~nan]), "E4M3 decode differs from torch"
    with open(os.path.join(GOLDEN, "e4m3_landmarks.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, value = line.split()
            v = float.fromhex(value) if "p" in value else float(value)
            g = oracle.e4m3_decode(int(code, 16), lib)
            assert g == v or (math.isnan(v) and math.isnan(g)), (code, g, v)


def pin_bf16(lib):
    """bf16 decode against torch; fp32 -> bf16 rounding against torch's RNE cast."""
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]            # finite values
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_decode(int(b), lib) for b in bits])
    assert np.array_equal(ref, got)
    xs = np.concatenate([rng.standard_normal(3000).astype(np.float32),
                         (rng.standard_normal(1000) * 1e-30).astype(np.float32),
                         np.float32([0.5, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.0 - 2**-7])])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(x), lib) for x in xs], dtype=np.uint16)
    assert np.array_equal(ref, got)


def pin_gate(lib):
    """The gate factor: closed forms, then every finite bf16 input against torch."""
    def bits(x):
        return int(torch.tensor([x], dtype=torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    assert oracle.gate_factor(bits(0.0), lib) == 0.5
    assert oracle.gate_factor(bits(20.0), lib) == 1.0
    assert oracle.gate_factor(bits(-200.0), lib) == 0.0
    assert oracle.gate_factor(bits(1.0), lib) == float(torch.tensor(1 / (1 + math.exp(-1.0))).to(torch.bfloat16))
    allb = np.arange(1 << 16, dtype=np.uint32)
    finite = allb[(allb & 0x7F80) != 0x7F80][::3]
    refs = torch_gate(finite.astype(np.uint16))
    mism = 0
    for b, ref in zip(finite, refs):
        got = oracle.gate_factor(int(b), lib)
        if got != ref:
            mism += 1
            ulp = abs(ref) * 2**-7 if ref else 2**-133
            assert abs(got - ref) <= ulp, (hex(int(b)), got, ref)
    assert mism <= len(finite) // 1000, mism


def pin_splits(lib):
    """`sparse_decode_splits` against the hand-derived truth table."""
    with open(os.path.join(GOLDEN, "sparse_decode_splits.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lo, hi, s = (int(x) for x in line.split())
            for rows in range(lo, hi + 1):
                assert oracle.sparse_decode_splits(rows, lib) == s, (rows, s)
    for rows in range(5, 129):                 # ~256 programs: 128 < rows*splits <= 256
        s = oracle.sparse_decode_splits(rows, lib)
        assert 128 < rows * s <= 256, (rows, s)


def _dense_cases():
    return [
        dict(seed=11, reqs=3, G=2, H=4, B=16, RT=16),
        dict(seed=12, reqs=2, query_len=2, G=3, H=16, B=16, RT=8),     # regions smaller than blocks
        dict(seed=13, reqs=2, G=1, H=8, B=8, RT=32),                   # regions spanning pages
        dict(seed=14, reqs=3, G=2, H=5, B=16, RT=16, fp8=True),
        dict(seed=15, reqs=2, query_len=2, G=2, H=3, B=8, RT=8, fp8=True, page_pad=64),
    ]


def pin_dense_bruteforce(lib):
    """Selecting every visible region equals causal decode attention over tokens 0..pos."""
    for case in _dense_cases():
        d = Dense(**case)
        got = d.oracle(lib)
        for r in range(d.rows):
            ref = d.textbook(r)
            err = np.abs(got[r] - ref).max()
            assert err < 1e-12, (case, r, err)


def pin_gate_applied(lib):
    """With a gate, each head is the ungated result times torch's bf16 sigmoid of gate[token, g*H+h]."""
    d = Dense(21, reqs=2, query_len=2, G=2, H=3, B=16, RT=16, gate=True)
    base = d.oracle(lib, gate=None)
    gated = d.oracle(lib)
    gbits = d.gate.view(torch.int16).numpy().astype(np.int64) & 0xFFFF
    for r in range(d.rows):
        tok, g = r // d.G, r % d.G
        for h in range(d.H):
            f = torch_gate(int(gbits[tok, g * d.H + h]))
            assert np.array_equal(gated[r, h], base[r, h] * f), (r, h)


def pin_single_token(lib):
    """One visible token (the first of the current region) returns its V row exactly."""
    for fp8 in (False, True):
        d = Dense(31, reqs=3, G=2, H=6, B=16, RT=16, fp8=fp8)
        pos = d.positions.copy()
        regions = np.full_like(d.regions, -1)
        for r in range(d.rows):
            cur = int(pos[r]) // d.RT
            pos[r] = cur * d.RT
            regions[r, r % regions.shape[1]] = cur
        got = d.oracle(lib, positions=pos, regions=regions)
        for r in range(d.rows):
            q, g = r // (d.G * d.ql), r % d.G
            v = d.kv[q][g][int(pos[r]), 192:].numpy()
            for h in range(d.H):
                assert np.array_equal(got[r, h], v), (fp8, r, h)


def pin_zero_query_mean(lib):
    """q = 0 gives equal weights: the mean of the visible V rows."""
    d = Dense(41, reqs=2, G=2, H=2, B=16, RT=16)
    d.query.zero_()
    got = d.oracle(lib)
    for r in range(d.rows):
        q, g = r // (d.G * d.ql), r % d.G
        mean = d.kv[q][g][: int(d.positions[r]) + 1, 192:].mean(0).numpy()
        assert np.abs(got[r] - mean).max() < 1e-13


def pin_invariants(lib):
    """Region order and -1 placement do not matter; rows permute with their requests."""
    d = Dense(51, reqs=4, query_len=2, G=2, H=4, B=16, RT=16, gate=True)
    base = d.oracle(lib)
    rng = np.random.default_rng(0)
    shuffled = np.array([rng.permutation(row) for row in d.regions])
    padded = np.concatenate([np.full((d.rows, 3), -1, np.int32), shuffled], axis=1)
    for reg in (shuffled, padded):
        got = d.oracle(lib, regions=np.ascontiguousarray(reg))
        assert np.abs(got - base).max() < 1e-12
    # permute requests together with their rows, table rows and gate rows
    perm = rng.permutation(d.reqs)
    per = d.G * d.ql
    rows = np.concatenate([np.arange(p * per, (p + 1) * per) for p in perm])
    toks = np.concatenate([np.arange(p * d.ql, (p + 1) * d.ql) for p in perm])
    got = oracle.sparse_decode_attention(
        d.query[torch.from_numpy(rows)], d.cache, d.regions[rows], d.table[perm], d.positions[rows],
        d.active[rows], gate=d.gate[torch.from_numpy(toks)], scale=d.scale, query_len=d.ql,
        region_tokens=d.RT, lib=lib)
    assert np.array_equal(got, base[rows])


def pin_inactive(lib):
    """Inactive rows are +0.0 (sign bit clear); other rows are untouched by them."""
    d = Dense(61, reqs=3, G=2, H=4, B=16, RT=16, gate=True)
    base = d.oracle(lib)
    act = d.active.copy()
    act[[1, 4]] = 0
    got = d.oracle(lib, active=act)
    for r in range(d.rows):
        if act[r]:
            assert np.array_equal(got[r], base[r])
        else:
            assert (got[r] == 0).all() and not np.signbit(got[r]).any()


def pin_empty_rows(lib):
    """An active row with no live region, or whose regions all start past its position, is 0."""
    d = Dense(71, reqs=2, G=2, H=4, B=16, RT=16)
    regions = d.regions.copy()
    regions[0] = -1
    regions[1] = -1
    regions[1, 0] = int(d.positions[1]) // d.RT + 1       # starts past the position
    got = d.oracle(lib, regions=regions)
    assert (got[0] == 0).all() and (got[1] == 0).all()
    pos = d.positions.copy()
    pos[2] = -1
    got = d.oracle(lib, positions=pos)
    assert (got[2] == 0).all()


def pin_split_partials(lib):
    """Partials merged by their LSEs give the full result; S=1 is the full result; the
    partition is contiguous over the live list with floor boundaries."""
    d = Dense(81, reqs=3, query_len=1, G=2, H=4, B=8, RT=8)
    base = d.oracle(lib)
    kw = dict(scale=d.scale, query_len=d.ql, region_tokens=d.RT, lib=lib)
    for S in (1, 2, 3, 5, 32):
        part, lse = oracle.split_partials(d.query, d.cache, d.regions, d.table, d.positions,
                                          d.active, splits=S, **kw)
        m = lse.max(axis=1, keepdims=True)
        w = np.exp(lse - m)
        merged = (w[..., None] * part).sum(1) / w.sum(1)[..., None]
        assert np.abs(merged - base).max() < 1e-12, S
        if S == 1:
            assert np.abs(part[:, 0] - base).max() < 1e-15
    # each split alone equals the oracle run on exactly that chunk's regions
    S = 3
    part, lse = oracle.split_partials(d.query, d.cache, d.regions, d.table, d.positions,
                                      d.active, splits=S, **kw)
    for r in range(d.rows):
        live = [x for x in d.regions[r] if x >= 0 and x * d.RT <= d.positions[r]]
        n = len(live)
        for s in range(S):
            chunk = live[s * n // S:(s + 1) * n // S]
            reg = np.full_like(d.regions, -1)
            reg[r, :len(chunk)] = chunk
            one = d.oracle(lib, regions=reg, row_ids=[r])[0]
            assert np.abs(one - part[r, s]).max() < 1e-12, (r, s)
            if chunk:
                q, g = r // (d.G * d.ql), r % d.G
                toks = [t for c in chunk for t in range(c * d.RT, c * d.RT + d.RT) if t <= d.positions[r]]
                kv = d.kv[q][g][toks]
                logits = d.query[r].double() @ kv[:, :192].T * d.scale
                ref = torch.logsumexp(logits, dim=1).numpy()
                assert np.abs(lse[r, s] - ref).max() < 1e-12
            else:
                assert np.isneginf(lse[r, s]).all()


def _swa(d, lib, window, **kw):
    return oracle.swa_decode(d.query, d.cache, d.table, d.lengths.astype(np.int32), scale=d.scale,
                             window=window, query_len=d.ql, k_scale=d.k_scale, v_scale=d.v_scale,
                             cache_fp8=d.fp8, gate=kw.pop("gate", d.gate), lib=lib, **kw)


def pin_swa_dense(lib):
    """Sliding window: torch float64 SDPA over the dense slice [max(0, p-w+1), p]."""
    for case in (dict(seed=101, reqs=3, query_len=2, G=2, H=4, B=16, RT=16),
                 dict(seed=102, reqs=2, query_len=3, G=1, H=16, B=8, RT=8, fp8=True)):
        d = Dense(**case)
        for window in (1, 5, 17, 40, 10_000):
            got = _swa(d, lib, window)
            for r in range(d.rows):
                q, g = r // (d.G * d.ql), r % d.G
                pos = int(d.positions[r])
                lo = max(0, pos - window + 1)
                kv = d.kv[q][g][lo:pos + 1]
                Q = d.query[r].to(torch.float64).unsqueeze(0)
                ref = torch.nn.functional.scaled_dot_product_attention(
                    Q, kv[:, :192].unsqueeze(0), kv[:, 192:].unsqueeze(0), scale=d.scale)[0].numpy()
                assert np.abs(got[r] - ref).max() < 1e-12, (case, window, r)
                if window == 1:
                    assert np.array_equal(got[r], np.broadcast_to(d.kv[q][g][pos, 192:].numpy(), got[r].shape))


def pin_swa_matches_sparse_path(lib):
    """A window equals the sparse path with one-token regions listing exactly the window's tokens."""
    d = Dense(111, reqs=3, query_len=2, G=2, H=3, B=16, RT=16, gate=True)
    window = 23
    got = _swa(d, lib, window)
    R = window + 2
    regions = np.full((d.rows, R), -1, np.int32)
    for r in range(d.rows):
        pos = int(d.positions[r])
        ids = np.arange(max(0, pos - window + 1), pos + 1)
        regions[r, :len(ids)] = ids[::-1]
    ref = d.oracle(lib, regions=regions, region_tokens=1)
    assert np.abs(got - ref).max() < 1e-12


def _select_numpy(scores, cur, topk, length):
    """Brute force with numpy's sort: rank (score desc, id asc), NaN last."""
    forced = 0 <= cur < length
    ids = np.array([i for i in range(length) if not (forced and i == cur)], dtype=np.int64)
    sc = scores[ids].astype(np.float64)
    key = np.where(np.isnan(sc), np.inf, -sc)
    order = np.lexsort((ids, key))
    keep = ids[order[:max(0, topk - int(forced))]]
    return ([cur] if forced else []) + sorted(keep.tolist())


def pin_select_regions(lib):
    """Region selection against numpy brute force, with its invariants."""
    rng = np.random.default_rng(7)
    for rows, n, topk in ((40, 300, 16), (20, 64, 80), (10, 5000, 1024)):
        scores = rng.standard_normal((rows, n)).astype(np.float32)
        scores[0, :7] = np.nan
        scores[1, 10:40] = 0.25                     # ties
        lengths = rng.integers(0, n + 1, size=rows).astype(np.int32)
        lengths[2] = n
        current = np.array([rng.integers(-1, max(1, l)) for l in lengths], dtype=np.int32)
        current[3] = -1                              # no current region
        got = oracle.select_regions(scores, current, topk, lengths, lib=lib)
        for r in range(rows):
            L, cur = int(lengths[r]), int(current[r])
            row = [int(x) for x in got[r] if x >= 0]
            assert all(x == -1 for x in got[r][len(row):]), r
            forced = 0 <= cur < L
            assert len(row) == min(topk, L), (r, len(row))
            if forced:
                assert row[0] == cur
            others = row[1:] if forced else row
            assert others == sorted(others) and len(set(others)) == len(others)
            chosen = set(others)
            rest = [i for i in range(L) if i not in chosen and not (forced and i == cur)]
            if chosen and rest:                       # every kept score >= every dropped one
                kept = scores[r, sorted(chosen)]
                drop = scores[r, rest]
                lo = np.min(np.where(np.isnan(kept), -np.inf, kept))
                hi = np.max(np.where(np.isnan(drop), -np.inf, drop))
                assert lo >= hi, r
            if r != 1:                                # unique answer without ties
                assert row == _select_numpy(scores[r], cur, topk, L), r
    # closed forms
    sc = np.array([[5.0, 4.0, 3.0, 2.0, 1.0]], np.float32)
    assert oracle.select_regions(sc, np.array([4], np.int32), 2, lib=lib).tolist() == [[4, 0]]
    assert oracle.select_regions(sc, np.array([0], np.int32), 9, lib=lib).tolist() == [[0, 1, 2, 3, 4, -1, -1, -1, -1]]
    sc = np.array([[-np.inf, np.nan, 1.0]], np.float32)
    assert oracle.select_regions(sc, np.array([-1], np.int32), 2, lib=lib).tolist() == [[0, 2]]


# ---------------------------------------------------------------------------
# Indexer decode scores
# ---------------------------------------------------------------------------

def _finite_e4m3(rng, shape):
    b = rng.integers(0, 256, size=shape, dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0                        # no NaN codes
    return b


def _e4m3_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64)


class DenseSummaries:
    """Per-(request, group) dense region summaries, scattered by this file into
    the pages of a shuffled pool (decoy pages hold NaN codes), with FP8 index
    queries and fp32 head weights for every (token, group)."""

    def __init__(self, seed, *, seq_lens, G=2, B=16, query_len=1, n_cols=None, decoys=3):
        rng = np.random.default_rng(seed)
        self.G, self.B, self.query_len = G, B, query_len
        self.seq_lens = np.asarray(seq_lens, np.int32)
        reqs = len(seq_lens)
        W = max(1, -(-int(max(seq_lens)) // B))
        per = B // 8
        self.n_cols = W * per if n_cols is None else n_cols
        self.dense = _finite_e4m3(rng, (reqs, G, W * per, 256))
        pages = reqs * W + decoys
        order = rng.permutation(pages)
        self.table = order[:reqs * W].reshape(reqs, W).astype(np.int32)
        self.summaries = np.full((pages * per, G, 256), 0x7F, np.uint8)
        for r in range(reqs):
            for c in range(W):
                p = self.table[r, c]
                self.summaries[p * per:(p + 1) * per] = self.dense[r, :, c * per:(c + 1) * per].transpose(1, 0, 2)
        tokens = reqs * query_len
        self.query = _finite_e4m3(rng, (tokens, G, 8, 256))
        self.weights = rng.standard_normal((tokens, G, 8)).astype(np.float32)

    def run(self, lib, **kw):
        return oracle.summary_scores(self.query, self.weights, self.summaries, self.table, self.seq_lens,
                                     block=self.B, n_cols=self.n_cols, query_len=self.query_len,
                                     lib=lib, **kw)

    def expected(self, row):
        """Dense torch float64: relu(M q^T) w over the row's scored regions, -inf after."""
        tok, g = divmod(row, self.G)
        req = tok // self.query_len
        pos = int(self.seq_lens[req]) - self.query_len + tok % self.query_len
        n = min(pos // 8 + 1, self.n_cols) if pos >= 0 else 0
        out = torch.full((self.n_cols,), -math.inf, dtype=torch.float64)
        if n:
            m = _e4m3_f64(self.dense[req, g, :n])
            q = _e4m3_f64(self.query[tok, g])
            w = torch.from_numpy(self.weights[tok, g]).to(torch.float64)
            out[:n] = torch.relu(m @ q.T) @ w
        return out.numpy(), (pos // 8 if pos >= 0 else -1), n


def pin_summary_dense(lib):
    """Indexer scores against a dense torch computation over summaries this file
    scattered into shuffled pages (decoys full of NaN codes)."""
    cases = (dict(seq_lens=[37, 130, 9], G=2, B=16),
             dict(seq_lens=[200, 64, 1], G=4, B=64, query_len=2),
             dict(seq_lens=[95, 260], G=1, B=32, query_len=3, n_cols=20))
    for i, kw in enumerate(cases):
        d = DenseSummaries(100 + i, **kw)
        scores, cur, lens = d.run(lib)
        for row in range(len(d.query) * d.G):
            exp, ecur, en = d.expected(row)
            assert cur[row] == ecur and lens[row] == en, (i, row, cur[row], ecur, lens[row], en)
            fin = np.isfinite(exp)
            assert np.array_equal(np.isfinite(scores[row]), fin), (i, row)
            assert np.allclose(scores[row][fin], exp[fin], rtol=1e-12, atol=1e-9), (i, row)
        sub = [3, 0, 5]
        s2, c2, l2 = d.run(lib, row_ids=sub)
        assert np.array_equal(s2, scores[sub]) and np.array_equal(l2, lens[sub])


def pin_summary_closed_forms(lib):
    """One-hot queries read single summary values back: with q_h = +/-e_d on one
    head, the score is w_h * max(0, +/-m_j[d]); weights enter linearly."""
    d = DenseSummaries(7, seq_lens=[41, 17], G=2, B=16)
    one = 0x38                                        # E4M3 code of 1.0
    for sign, code in ((1.0, one), (-1.0, one | 0x80)):
        for g in range(2):
            q = np.zeros_like(d.query)
            q[:, g, 5, 77] = code
            d2 = DenseSummaries(7, seq_lens=[41, 17], G=2, B=16)
            d2.query = q
            d2.weights[:, :, 5] = 2.5
            scores, _, lens = d2.run(lib)
            for tok in range(2):
                row = tok * 2 + g
                n = int(lens[row])
                m = _e4m3_f64(d.dense[tok, g, :n, 77]).numpy()
                assert np.array_equal(scores[row, :n], 2.5 * np.maximum(0.0, sign * m)), (sign, g, tok)
                other = tok * 2 + (1 - g)                    # the other group's query is zero
                assert np.all(scores[other, :int(lens[other])] == 0.0)
    rng = np.random.default_rng(3)                    # multiples of 1/8: sums are exact in fp32
    w1 = (rng.integers(-16, 17, d.weights.shape) / 8).astype(np.float32)
    w2 = (rng.integers(-16, 17, d.weights.shape) / 8).astype(np.float32)
    d.weights = w1
    a, _, _ = d.run(lib)
    d.weights = w2
    b, _, _ = d.run(lib)
    d.weights = w1 + w2
    c, _, _ = d.run(lib)
    fin = np.isfinite(a)
    assert np.allclose(c[fin], (a + b)[fin], rtol=1e-12, atol=1e-6)
    assert np.all(c[~fin] == -np.inf)


ALL_PINS = [pin_e4m3_decode, pin_bf16, pin_gate, pin_splits, pin_dense_bruteforce,
            pin_gate_applied, pin_single_token, pin_zero_query_mean, pin_invariants,
            pin_inactive, pin_empty_rows, pin_split_partials, pin_swa_dense,
            pin_swa_matches_sparse_path, pin_select_regions, pin_summary_dense,
            pin_summary_closed_forms]
