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


def test_split_traffic_accounting():
    """Algorithmic bytes of the sparse and window paths on a hand-counted workload: one request,
    2 tokens at positions 40 and 41, 2 groups, 16-token blocks = regions, 4 heads, bf16."""
    import numpy as np
    import torch
    import bench
    from sparse_decode_attention_02_gb300 import inputs
    cfg = inputs.Config("hand", requests=1, query_len=2, groups=2, heads=4, block=16, region_tokens=16,
                        num_regions=3, ctx=(42, 42))
    i32 = lambda a: torch.tensor(a, dtype=torch.int32)
    w = inputs.Workload(cfg, torch.zeros(4, 4, 192, dtype=torch.bfloat16),
                        torch.zeros(4, 2, 16, 384, dtype=torch.bfloat16),
                        i32([[0, 2, -1], [1, 2, 5], [2, -1, -1], [0, 1, 2]]), i32([[0, 1, 2, 3]]),
                        i32([40, 40, 41, 41]), torch.tensor([1, 1, 1, 0], dtype=torch.uint8), None,
                        None, None, 192 ** -0.5, None, np.zeros((0, 2), np.int64), i32([42]))
    # row 0: region 0 (16) + region 2 (tokens 32..40: 9); row 1: 16 + 9, region 5 is in the future;
    # row 2: region 2 up to 41 (10); row 3 is inactive
    assert bench.visible_tokens(w).tolist() == [25, 25, 10, 0]
    # distinct tokens per (request, group): group 0 rows 0 and 2 -> regions {0, 2} up to 41: 16 + 10;
    # group 1 row 1 only -> regions {1, 2} up to 40: 16 + 9
    assert bench.unique_kv_bytes(w) == 51 * 384 * 2
    per_row = 4 * 192 * 2 * 2 + 3 * 4 + 8                       # Q + out, region ids, position+flag
    table = (2 + 2 + 1) * 4                                     # ceil(visible / 16) entries per row
    assert bench.traffic(w, 1) == (60 * 384 * 2, 60 * 384 * 2 + 3 * per_row + table)
    partials = 3 * 2 * 4 * 193 * 4 * 2                          # active rows x S x H x (O + LSE), w + r
    assert bench.traffic(w, 2)[1] == 60 * 384 * 2 + 3 * per_row + table + partials
    # window mode, window 8 (window rows have no active flag: every row runs): each row sees
    # 8 tokens; the union per (request, group) is 33..41, 9 tokens, for both groups
    import dataclasses
    ww = dataclasses.replace(w, config=dataclasses.replace(cfg, window=8, num_regions=0),
                             regions=torch.zeros(4, 0, dtype=torch.int32),
                             active=torch.ones(4, dtype=torch.uint8))
    assert bench.visible_tokens(ww).tolist() == [8, 8, 8, 8]
    assert bench.unique_kv_bytes(ww) == 18 * 384 * 2
    assert bench.traffic(ww, 1) == (32 * 384 * 2, 18 * 384 * 2 + 4 * (4 * 192 * 4 + 8) + 4 * 4)
