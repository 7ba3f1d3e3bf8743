"""Failure detection on the GPU without a fault: bounded waits report, never hang.

The pipeline waits inside the split kernel give up after a limit (1 s by
default).  Setting the limit to 0 makes them run out while copies are still in
flight; the kernel must then flag SDA_FLAG_TIMEOUT in the workspace, let its
copies land, and return, leaving the context usable: the next call with the
normal limit is correct.  Bad indices are covered by the parity tests
(test_bad_indices_are_flagged_not_faulted)."""
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import check, oracle_rows, run
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("fp8,splits", [(True, 1), (False, 2)])
def test_wait_timeout_is_flagged_and_recoverable(fp8, splits):
    cfg = inputs.scaled("large", requests=16, ctx=(36864, 40000), fp8=fp8)
    w = inputs.make_workload(cfg, DEV)
    sda.set_wait_limit_ns(0)
    try:
        _, flags = run(w, splits=splits)
    finally:
        sda.set_wait_limit_ns(10 ** 9)
    assert flags & sda.FLAG_TIMEOUT
    out, flags = run(w, splits=splits)
    assert flags == 0
    rows = list(range(0, w.rows, 7))
    check(w, out, oracle_rows(w, rows), rows)
