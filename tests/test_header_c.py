"""include/sdattn.h is a plain C header: a C99 translation unit that includes
it and takes the address of every declared entry point (with the header's own
prototypes) compiles with -Werror, and every declared name is exported by the
built library under the same C symbol."""
import os
import subprocess
import tempfile

import pytest

import sparse_decode_attention_02_gb300 as sda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c99():
    names = sda.declared_functions()
    assert "sparse_decode_summary_scores" in names and "sparse_decode_attention" in names
    body = "\n".join(f"    (sdattn_fn)&{n}," for n in names)
    src = ('#include "sdattn.h"\n'
           "typedef void (*sdattn_fn)(void);\n"
           f"sdattn_fn sdattn_entry_points[] = {{\n{body}\n}};\n"
           "int sdattn_status_count = (int)SDA_ERR_BOUNDS + 1;\n")
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "abi.c")
        with open(path, "w") as f:
            f.write(src)
        r = subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-c", path,
                            "-I", os.path.join(ROOT, "include"), "-o", os.path.join(d, "abi.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_library_symbols_are_unmangled():
    from sparse_decode_attention_02_gb300 import build
    lib = build.build()
    r = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm unavailable")
    exported = {line.split()[-1] for line in r.stdout.splitlines() if line.strip()}
    for n in sda.declared_functions():
        assert n in exported, n
