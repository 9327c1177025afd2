"""The C ABI from C, without a GPU: include/kvb.h compiles as strict C99 and
C11 (pedantic, warnings as errors), and a C program links against libkvb.so
and runs the host-only entry points (ABI version, page bytes, op validation
with its error codes)."""
import os
import shutil
import subprocess

import pytest

from hierarchical_kv_cache_backup_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include "kvb.h"
#include <stdio.h>

int main(void) {
    kv_layout lay = {32, 2, 4096, 16, 8, 256, KV_LAYER_FIRST, KV_NHD, 2, 0};
    kv_layout bad = lay;
    uint64_t pb = 0;
    int32_t src[3] = {5, 17, 4095}, slots[3] = {0, 1, 2}, dup[3] = {0, 1, 1};
    int32_t oob[1] = {4096}, zero[1] = {0};
    int fails = 0;
    fails += kv_abi_version() != KVB_ABI_VERSION;
    fails += kv_layout_page_bytes(&lay, &pb) != KV_OK || pb != 2097152ull;
    fails += kv_op_validate(&lay, 16, 0, src, slots, 3, -1) != KV_OK;          /* backup */
    fails += kv_op_validate(&lay, 16, 1, slots, src, 3, 31) != KV_OK;          /* restore, layer */
    fails += kv_op_validate(&lay, 16, 0, src, dup, 3, -1) != KV_ERR_DUPLICATE;
    fails += kv_op_validate(&lay, 16, 0, oob, zero, 1, -1) != KV_ERR_OUT_OF_RANGE;
    fails += kv_op_validate(&lay, 16, 1, zero, zero, 1, 32) != KV_ERR_OUT_OF_RANGE;
    bad.head_bytes = 100;                                                    /* not 16-B */
    fails += kv_layout_page_bytes(&bad, &pb) == KV_OK;
    fails += kv_last_error() == NULL || kv_last_error()[0] == '\0';
    printf("c-abi fails=%d\n", fails);
    return fails;
}
"""


@pytest.fixture(scope="module")
def gcc():
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("gcc not found")
    return cc


@pytest.mark.parametrize("std", ["c99", "c11"])
def test_header_compiles_as_strict_c(gcc, tmp_path, std):
    src = tmp_path / "t.c"
    src.write_text(PROGRAM)
    subprocess.run([gcc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE,
                    "-fsyntax-only", str(src)], check=True)


def test_c_program_links_and_runs(gcc, tmp_path):
    lib = kbuild.build_library()
    libdir = os.path.dirname(lib)
    src = tmp_path / "t.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-L", libdir,
                    "-lkvb", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "fails=0" in out.stdout
