"""The committed ncu traffic records describe the kernels as they are now.

bench.py scales each record's DRAM bytes to the timed launch and reports
null once the kernel source no longer matches the recorded hash; this test
makes a kernel change without a fresh capture fail loudly instead."""
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
