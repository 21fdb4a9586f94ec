"""The public header is plain C: a C99 program that includes it, links
against libgemm_gb300.so and calls the host-only entry points builds and
runs on a machine without a GPU."""
import os
import subprocess
import sys

import pytest

from dense_tensor_core_02_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gemm_gb300.h"

int main(void) {
    int64_t plan[10];
    int m = -1, n = -1;
    if (strcmp(gemm_status_string(GEMM_ERR_MISALIGNED), "GEMM_ERR_MISALIGNED") != 0) return 1;
    if (strcmp(gemm_status_string(GEMM_ERR_UNSUPPORTED_LAYOUT), "GEMM_ERR_UNSUPPORTED_LAYOUT") != 0) return 2;
    if (gemm_plan(8192, 8192, 8192, 152, plan) != GEMM_OK || plan[0] != 1 || plan[1] != 256 || plan[2] != 256)
        return 3;
    if (gemm_tile_coords(9, 32, 32, 8, &m, &n) != GEMM_OK || m != 1 || n != 1) return 4;
    /* argument errors are reported before any device work */
    if (gemm(NULL, NULL, NULL, NULL, 64, 64, 64, 64, 64, 64, 64, 0, 0, 1.0f, 0.0f, GEMM_F16, GEMM_F32, NULL) !=
        GEMM_ERR_INVALID_ARG)
        return 5;
    if (gemm_host(NULL, NULL, NULL, NULL, 1, 1, 1, 1, 1, 1, 1, 0, 0, 1.0f, 0.0f, 7, GEMM_F32, NULL) !=
        GEMM_ERR_UNSUPPORTED_DTYPE)
        return 6;
    printf("ok\n");
    return 0;
}
"""


def test_c_program_builds_links_and_runs(tmp_path):
    lib = build_mod.build()
    src = tmp_path / "use_gemm.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_gemm"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           lib, "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
