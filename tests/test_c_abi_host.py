"""The boundary as a C program sees it (no GPU): the header compiles as C99
and C++11 with -pedantic, and a C program linked against the library makes
host-only calls (planning, validation, status strings) through it."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mt_rowreduce.h"

int main(void) {
    mt_plan_t p;
    char text[256];
    /* planning and introspection: host only */
    if (mt_plan_query(MT_OP_RMSNORM, 1024, 4096, &p) != MT_OK) return 1;
    if (mt_plan_check(MT_OP_RMSNORM, 4096, &p) != MT_OK) return 2;
    mt_describe_plan(&p, text, sizeof text);
    if (strncmp(text, "path=", 5) != 0) return 3;
    if (mt_private_slot_bound(10, 4, 2) != 4) return 4;
    /* argument checks happen before any CUDA call */
    if (mt_rmsnorm_f32(NULL, NULL, NULL, 4, 8, 1e-6f, NULL) !=
        MT_ERR_INVALID_ARGUMENT) return 5;
    if (mt_softmax_bf16(NULL, NULL, 0, 8, NULL) != MT_OK) return 6;
    if (strcmp(mt_status_string(MT_ERR_OUT_OF_RESOURCES),
               "MT_ERR_OUT_OF_RESOURCES") != 0) return 7;
    printf("%s\n", text);
    return 0;
}
"""


@pytest.mark.parametrize("std,lang", [("c99", "c"), ("c++11", "c++")])
def test_header_is_plain_c_and_cxx(tmp_path, std, lang):
    src = tmp_path / "inc.c"
    src.write_text('#include "mt_rowreduce.h"\nint main(void) { return 0; }\n')
    cc = "gcc" if lang == "c" else "g++"
    subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic",
                    "-Werror", "-fsyntax-only", "-x", lang, "-I", INCLUDE,
                    str(src)], check=True)


def test_c_program_through_the_library(tmp_path):
    sys.path.insert(0, ROOT)
    from row_reduction_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(str(lib))
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", INCLUDE,
                    str(src), "-o", str(exe), "-L", libdir, "-lmt_rowreduce",
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.startswith("path=registers W=")
