"""Builds libsdattn.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", name) for name in ("sdattn.cu", "sda_select.cu", "sda_index.cu")]
HEADER = os.path.join(ROOT, "include", "sdattn.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsdattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          out: str = LIB) -> str:
    """Compile the library unless it is newer than its sources; returns its path."""
    if (not force and not extra and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(x) for x in [*SOURCES, HEADER])):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include"), *(extra or [])]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    objs = [f"{tmp}.{i}.o" for i in range(len(SOURCES))]
    procs = [subprocess.Popen([*common, "-c", src, "-o", obj], stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True)
             for src, obj in zip(SOURCES, objs)]            # translation units in parallel
    logs = [p.communicate() for p in procs]
    failed = [p.returncode for p in procs if p.returncode]
    if not failed:
        r = subprocess.run([nvcc(), *ARCH, "-shared", *objs, "-o", tmp], capture_output=True, text=True)
        logs.append((r.stdout, r.stderr))
        failed = [r.returncode] if r.returncode else []
    for obj in objs:
        if os.path.exists(obj):
            os.remove(obj)
    if failed or verbose:
        sys.stderr.write("".join(a + b for a, b in logs))
    if failed:
        raise RuntimeError("nvcc failed building libsdattn.so")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
