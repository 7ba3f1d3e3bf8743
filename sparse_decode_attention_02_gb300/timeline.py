"""Per-CTA phase timeline of the split and combine kernels (a measurement aid).

Builds a diagnostic copy of the library with SDA_TIMELINE (its kernels stamp
%globaltimer at their phase boundaries; the regular library carries no stamps),
runs one workload with L2 flushed between calls, and prints when the split
kernel's CTAs pass each phase and when the combine kernel's CTAs start and pass
their wait on the split kernel (programmatic dependent launch), relative to the
first split CTA's start, as median and last CTA over the calls.

    python -m sparse_decode_attention_02_gb300.timeline --config gqa
    python -m sparse_decode_attention_02_gb300.timeline --config fp8 --empty
"""
from __future__ import annotations

import argparse
import os
import statistics

import numpy as np
import torch

from . import _binding as B
from . import build as lib_build
from . import inputs

PHASES = ["start", "consumers released", "first K|V stage landed", "stage loop done",
          "output writes start", "done"]
UNITS = 1 << 20                        # split stamps: [UNITS][8]; combine stamps after them: [UNITS][2]


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="gqa", choices=[c for c in inputs.ORDER])
    ap.add_argument("--splits", type=int, default=None)
    ap.add_argument("--calls", type=int, default=12)
    ap.add_argument("--empty", action="store_true", help="every region id -1: the call moves no K|V")
    args = ap.parse_args()

    path = os.path.join(lib_build.OUT_DIR, "libsdattn_timeline.so")
    lib_build.build(extra=["-DSDA_TIMELINE"], out=path)
    B.use_library(path)
    dev = torch.device("cuda", 0)
    w = inputs.make_workload(args.config, dev)
    if args.empty:
        w.regions.fill_(-1)
    if w.window:
        raise SystemExit("window workloads are not covered")
    splits = args.splits or B.sparse_decode_splits(w.rows)
    units = w.rows * splits
    if units > UNITS:
        raise SystemExit(f"{units} split CTAs: more than the {UNITS} the stamp buffer holds")
    stamps = torch.zeros(10 * UNITS, dtype=torch.int64, device=dev)
    B.timeline_buffer(stamps)
    ws = torch.zeros(B.workspace_bytes(w.rows, w.heads, splits), dtype=torch.uint8, device=dev)
    ks = torch.tensor([w.k_scale], dtype=torch.float32, device=dev) if w.fp8 else None
    vs = torch.tensor([w.v_scale], dtype=torch.float32, device=dev) if w.fp8 else None
    out = torch.empty_like(w.query)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    split_t, comb_t, event_us = [], [], []
    for call in range(args.calls + 2):
        stamps.zero_()
        flush.zero_()
        torch.cuda._sleep(2_000_000)            # the host queues the call before the GPU reaches it
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        B.sparse_decode_attention(w.query, w.cache, w.regions, w.block_table, w.positions, w.active, out,
                                  scale=w.scale, query_len=w.query_len, splits=splits, k_scale=ks,
                                  v_scale=vs, gate=w.gate, region_tokens=w.region_tokens, workspace=ws)
        b.record()
        torch.cuda.synchronize()
        if call < 2:                            # warm-up calls
            continue
        st = stamps[:UNITS * 8].view(UNITS, 8)[:units, :6].cpu().numpy().astype(np.float64)
        cb = stamps[UNITS * 8:].view(UNITS, 2)[:w.rows].cpu().numpy().astype(np.float64)
        t0 = st[:, 0].min()
        st = np.where(st > 0, (st - t0) / 1e3, np.nan)
        cb = np.where(cb > 0, (cb - t0) / 1e3, np.nan)
        split_t.append(st)
        comb_t.append(cb)
        event_us.append(a.elapsed_time(b) * 1e3)
    B.timeline_buffer(None)
    st = np.stack(split_t)
    print(f"# {args.config}: {w.rows} rows, splits {splits}, {units} split CTAs"
          f"{', every region id -1' if args.empty else ''}; {args.calls} calls, L2 flushed between them")
    print(f"# CUDA events around the call: median {statistics.median(event_us):.1f} us")
    print("| phase (us from the first split CTA's start) | median CTA | last CTA |")
    print("|---|---|---|")
    for k, name in enumerate(PHASES):
        col = st[:, :, k]
        if np.isnan(col).all():
            continue
        med = np.nanmedian(np.nanmedian(col, axis=1))
        last = np.nanmedian(np.nanmax(col, axis=1))
        print(f"| split: {name} | {med:.2f} | {last:.2f} |")
    if splits > 1:
        cb = np.stack(comb_t)
        for k, name in enumerate(["start (before the wait)", "past the wait on the split kernel"]):
            first = np.nanmedian(np.nanmin(cb[:, :, k], axis=1))
            last = np.nanmedian(np.nanmax(cb[:, :, k], axis=1))
            print(f"| combine: {name}, first / last CTA | {first:.2f} | {last:.2f} |")


if __name__ == "__main__":
    main()
