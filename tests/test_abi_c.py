"""The C ABI from plain C: include/gemm.h compiles as C99 with warnings as
errors, and a C program links against the library and calls it.  Without a
GPU the plan cannot be created; the program checks that this is reported as
an error code (not a crash) and that argument checks work without a plan."""
import os
import subprocess
import sys

import pytest

import dense_fp16_gemm_04_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "gemm.h"

int main(void) {
    gemm_plan_t plan = 0;
    gemm_status_t s = gemm_plan_create(&plan, 0);
    printf("create %d %s\n", (int)s, gemm_status_string(s));
    if (s != GEMM_OK) {
        if (plan != 0) return 2;                       /* *out must stay NULL */
        if (gemm_run(0, 0, 0, 0, 8, 8, 8, GEMM_ACC_F32, 0) != GEMM_ERR_INVALID_ARG) return 3;
        if (gemm_run_ex(0, 0, GEMM_K_CONTIGUOUS, 0, GEMM_MN_CONTIGUOUS, 0, 8, 8, 8,
                        GEMM_ACC_F16, 0) != GEMM_ERR_INVALID_ARG) return 4;
        if (gemm_plan_destroy(0) != GEMM_OK) return 5;
        printf("variants %d first %s\n", (int)gemm_variant_count(), gemm_variant_name(0));
        return 0;
    }
    gemm_plan_destroy(plan);
    return 0;
}
"""


@pytest.fixture(scope="module")
def libpath():
    return g.build()


def test_header_compiles_as_c99(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "gemm.h"\nint main(void) { return (int)GEMM_OK; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o",
                    str(tmp_path / "h.o")], check=True)


def test_c_program_links_and_runs(tmp_path, libpath):
    src = tmp_path / "prog.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    libdir = os.path.dirname(libpath)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lgb300gemm",
                    f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("create ")
