"""The C ABI from C alone: tests/c_abi_caller.c (C99, no Python, no torch) is
built with gcc against the in-tree library, reads a seeded problem, calls
sparse_decode_splits, sparse_decode_workspace_bytes, sparse_decode_attention
(bf16, or FP8 with device-scalar scales, with or without the gate) and
sparse_decode_read_errors on the GPU, and writes its output, which must match
the oracle within the tolerance of its cache type."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from sparse_decode_attention_02_gb300 import build as lib_build
from sparse_decode_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def caller(tmp_path_factory):
    lib = lib_build.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    out = str(tmp_path_factory.mktemp("c_caller") / "c_abi_caller")
    libdir = os.path.dirname(lib)
    r = subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", os.path.join(HERE, "c_abi_caller.c"),
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                        "-L", libdir, "-lsdattn", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                        f"-Wl,-rpath,{libdir}", "-o", out], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def bits(t: torch.Tensor) -> bytes:
    return t.contiguous().view(torch.int16).numpy().tobytes() if t.dtype == torch.bfloat16 \
        else t.contiguous().numpy().tobytes()


@pytest.mark.parametrize("cfg", ["tiny", inputs.scaled("gqa", requests=4), inputs.scaled("fp8", requests=4)],
                         ids=["tiny", "gqa4", "fp8_gate4"])
def test_c_program_matches_oracle(caller, cfg, tmp_path):
    w = inputs.make_workload(cfg, "cpu", fill="all")
    w.active[1] = 0                                                   # at least one cleared row
    q, cache, reg, table = w.query, w.cache, w.regions, w.block_table
    head = np.array([w.rows, w.heads, cache.shape[0], w.groups, w.block, reg.shape[1], table.shape[0],
                     table.shape[1], w.query_len, w.region_tokens, int(w.fp8), int(w.gate is not None)],
                    dtype=np.int64).tobytes()
    scales = np.array([w.scale, w.k_scale or 1.0, w.v_scale or 1.0], dtype=np.float32).tobytes()
    src, dst = tmp_path / "problem.bin", tmp_path / "output.bin"
    src.write_bytes(head + scales + bits(q) + bits(cache) + bits(reg) + bits(table) + bits(w.positions)
                    + bits(w.active.to(torch.uint8)) + (bits(w.gate) if w.gate is not None else b""))
    r = subprocess.run([caller, str(src), str(dst)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    raw = dst.read_bytes()
    n = w.rows * w.heads * 192
    got = torch.frombuffer(bytearray(raw[:2 * n]), dtype=torch.bfloat16).float().view(w.rows, w.heads, 192)
    flags = int(np.frombuffer(raw[2 * n:], dtype=np.uint32)[0])
    assert flags == 0
    ref = oracle.sparse_decode_attention(q, cache, reg, table, w.positions, w.active, gate=w.gate,
                                         scale=w.scale, query_len=w.query_len, region_tokens=w.region_tokens,
                                         k_scale=w.k_scale, v_scale=w.v_scale, cache_fp8=w.fp8)
    assert np.isfinite(got.numpy()).all()
    assert float(np.abs(got.numpy() - ref).max()) <= (5e-2 if w.fp8 else 2e-2)
    inactive = ~w.active.numpy().astype(bool)                         # cleared rows are +0.0 exactly
    assert (got.view(torch.int16).numpy()[inactive] == 0).all()
