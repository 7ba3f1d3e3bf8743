"""The committed ncu records and summaries describe the kernels as they are now.

bench.py scales each traffic record's DRAM bytes to the timed launch and
reports null once the kernel source no longer matches the recorded hash; these
tests make a kernel change without fresh captures fail loudly instead, for the
traffic records and for every summary under profiles/."""
import hashlib
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fields(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].split()
            if len(line) == 2:
                out[line[0]] = line[1]
    return out


@pytest.mark.parametrize("record,source", [("ncu_traffic.txt", "sdattn.cu"),
                                           ("ncu_traffic_index.txt", "sda_index.cu")])
def test_traffic_record_matches_kernel_source(record, source):
    f = _fields(os.path.join(ROOT, "profiles", record))
    src = os.path.join(ROOT, "sparse_decode_attention_02_gb300", "csrc", source)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    assert f["kernel_source_sha256_16"] == sha, f"re-capture {record}: {source} changed"
    dram, alg = int(f["dram_bytes"]), int(f["algorithmic_bytes"])
    assert 0.95 < dram / alg < 1.2          # no large re-reads in the captured launch


def test_index_traffic_accounting():
    import numpy as np
    import torch
    import bench
    from sparse_decode_attention_02_gb300 import inputs
    w = inputs.IndexWorkload(torch.zeros(3, 2, 8, 256, dtype=torch.uint8), torch.zeros(3, 2, 8),
                             torch.zeros(40, 2, 256, dtype=torch.uint8), torch.zeros(3, 5, dtype=torch.int32),
                             torch.tensor([17, 0, 64], dtype=torch.int32), 16, 1, 10)
    # scored regions 3, 0, 8 -> 11 x 2 groups x 256 B; scores 6 x 10 x 4 B; queries and weights
    # 3 x 2 x 8 x (256 + 4) B; table entries 2 + 0 + 4 (16-token pages), 3 seq_lens
    expect = 11 * 2 * 256 + 6 * 10 * 4 + 3 * 2 * 8 * 260 + 6 * 4 + 3 * 4
    assert bench.index_traffic(w) == expect
    assert bench.index_traffic(w, with_outputs=True) == expect + 6 * 8


def test_profile_summaries_name_current_sources():
    """Every ncu summary states the kernel-source hash(es) it was taken on, and each is the
    hash of a current source: a kernel change without fresh captures fails here."""
    import glob
    import re
    csrc = os.path.join(ROOT, "sparse_decode_attention_02_gb300", "csrc")
    current = {hashlib.sha256(open(os.path.join(csrc, n), "rb").read()).hexdigest()[:16]: n
               for n in ("sdattn.cu", "sda_index.cu", "sda_select.cu")}
    summaries = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert summaries
    for path in summaries:
        hashes = set(re.findall(r"\b[0-9a-f]{16}\b", open(path).read()))
        assert hashes, f"{os.path.basename(path)} names no kernel-source hash"
        stale = sorted(h for h in hashes if h not in current)
        assert not stale, f"{os.path.basename(path)}: stale source hash(es) {stale}; re-capture"
