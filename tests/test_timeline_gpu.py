"""The diagnostic timeline build (SDA_TIMELINE): its phase stamps are ordered within
every split CTA, and the combine kernel passes its wait only after every split CTA
is done (programmatic dependent launch keeps the data dependency).  The regular
library is restored afterwards."""
import os

import numpy as np
import pytest
import torch

import sparse_decode_attention_02_gb300 as sda
from gpu_util import check, oracle_all, scales
from sparse_decode_attention_02_gb300 import _binding as B
from sparse_decode_attention_02_gb300 import build as lib_build
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
UNITS = 1 << 20


def test_timeline_stamps_are_ordered_and_the_combine_waits():
    path = os.path.join(lib_build.OUT_DIR, "libsdattn_timeline.so")
    lib_build.build(extra=["-DSDA_TIMELINE"], out=path)
    B.use_library(path)
    try:
        w = inputs.make_workload(inputs.scaled("gqa", requests=8, ctx=(2000, 6000), gate=True), DEV, fill="all")
        S = 2
        stamps = torch.zeros(10 * UNITS, dtype=torch.int64, device=DEV)
        sda.timeline_buffer(stamps)
        ws = torch.zeros(sda.workspace_bytes(w.rows, w.heads, S), dtype=torch.uint8, device=DEV)
        out = torch.full_like(w.query, float("nan"))
        sda.sparse_decode_attention(w.query, w.cache, w.regions, w.block_table, w.positions, w.active, out,
                                    scale=w.scale, splits=S, gate=w.gate, workspace=ws)
        torch.cuda.synchronize()
        sda.timeline_buffer(None)
        check(w, out, oracle_all(w))                      # the stamps change nothing
        st = stamps[:UNITS * 8].view(UNITS, 8)[:w.rows * S, :6].cpu().numpy()
        cb = stamps[UNITS * 8:].view(UNITS, 2)[:w.rows].cpu().numpy()
        assert (st[:, 0] > 0).all() and (st[:, 5] > 0).all() and (cb > 0).all()
        for k in range(1, 6):
            have = st[:, k] > 0                            # phase 2 is absent for a split with no pieces
            assert (st[have, k] >= st[have, 0]).all()
        assert (st[:, 5] >= st[:, 4]).all() and (st[:, 4] >= st[:, 3]).all()
        assert (cb[:, 1] >= st[:, 5].max()).all()          # past griddepcontrol.wait only after the split grid
        assert (cb[:, 1] >= cb[:, 0]).all()
    finally:
        B.use_library(B.LIB_PATH)
    with pytest.raises(sda.SdaError) as e:                 # the regular library has no stamps
        sda.timeline_buffer(torch.zeros(1, device=DEV))
    assert e.value.status == B.SDA_ERR_UNSUPPORTED
