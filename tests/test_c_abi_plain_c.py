"""The boundary is a C ABI: the public headers compile as strict C99 (and as
C++), and a plain C program links against libmla_decode.so and calls its
host-side entry points (no GPU needed for these)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "mla_latent_kv_fp8_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mla_decode.h"
#include "mla_decode_testing.h"

int main(void) {
    const int32_t lens[4] = {8192, 100, 0, 5000};
    mla_tensor_t t;
    memset(&t, 0, sizeof t);
    printf("%d %d %d %d %zu %s\n",
           (int)mla_auto_splits(8, 1, 12, 512, 152),
           (int)mla_auto_splits(32, 1, 96, 278, 152),
           (int)mla_plan_splits(4, 4, 12, lens, 128, 152),
           (int)mla_split_chunk_pages(512, 19),
           mla_decode_workspace_bytes(8, 1, 12, 19),
           mla_status_string(MLA_ERR_INVALID_ARG));
    return 0;
}
"""


@pytest.fixture(scope="module")
def built(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    so = os.path.join(PKG, "libmla_decode.so")
    if not os.path.exists(so):
        from mla_latent_kv_fp8_gb300 import build
        build.build()
    d = tmp_path_factory.mktemp("cabi")
    src = d / "main.c"
    src.write_text(PROGRAM)
    exe = d / "main"
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INC, str(src),
           "-L", PKG, "-lmla_decode", "-Wl,-rpath," + PKG, "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_headers_compile_as_cxx(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "main.cc"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-I", INC, "-c", str(src), "-o",
                    str(tmp_path / "main.o")], check=True, capture_output=True, text=True)


def test_plain_c_program_calls_the_library(built):
    r = subprocess.run([str(built)], check=True, capture_output=True, text=True, timeout=60)
    auto8, auto32, plan, chunk, ws, msg = r.stdout.split(maxsplit=5)
    from mla_latent_kv_fp8_gb300 import _lib
    assert int(auto8) == _lib.mla_auto_splits(8, 1, 12, 512, 152) == 19
    assert int(auto32) == 3
    assert int(plan) == _lib.mla_plan_splits(4, 4, 12, [8192, 100, 0, 5000], 128, 152)
    assert int(chunk) == 27
    assert int(ws) == _lib.mla_decode_workspace_bytes(8, 1, 12, 19)
    assert msg.strip() == _lib.mla_status_string(1)


def test_library_exports_only_the_declared_entry_points():
    """Built with hidden visibility: the defined functions the library exports are
    exactly the MLA_API declarations of include/*.h (the C++ internals stay
    private; weak C++ standard-library instantiations are not functions of ours)."""
    import re
    if shutil.which("nm") is None:
        pytest.skip("no nm")
    so = os.path.join(PKG, "libmla_decode.so")
    if not os.path.exists(so):
        from mla_latent_kv_fp8_gb300 import build
        build.build()
    declared = set()
    for h in os.listdir(INC):
        if h.endswith(".h"):
            declared |= set(re.findall(r"^MLA_API [^(]*?\b(mla_\w+)\(", open(os.path.join(INC, h)).read(), re.M))
    out = subprocess.run(["nm", "-D", "--defined-only", so], check=True, capture_output=True, text=True).stdout
    exported = {parts[2] for parts in (ln.split() for ln in out.splitlines()) if len(parts) == 3 and parts[1] == "T"}
    assert declared and exported == declared, (sorted(exported - declared), sorted(declared - exported))
