"""The boundary from C: include/rownorm.h compiles as C99 and the library
links into a plain C program (no GPU: only host-side calls run).

gcc builds a small C program that includes the header with -Wall -Werror
-pedantic, takes the address of every entry point (so each must be declared
with a C-compatible signature and exported), and calls the host-only ones:
status strings, plans, and argument validation that rejects bad calls
before anything is launched.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rownorm.h")
LIBDIR = os.path.join(ROOT, "row_wise_normalization_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "rownorm.h"

typedef void (*fnptr)(void);

int main(void) {
    volatile fnptr all[] = { %s };
    rn_plan plan;
    float *A = (float *)(size_t)0x10000000;
    int bad = 0;
    (void)all;
    if (strcmp(rn_status_str(RN_OK), "ok") != 0) bad |= 1;
    if (rn_plan_for(RN_OP_LN, RN_VARIANT_AUTO, 768, A, A + (1 << 24), A, A, &plan) != RN_OK)
        bad |= 2;
    if (plan.variant != RN_VARIANT_WARP || plan.vec != 4) bad |= 4;
    /* validation happens before any launch */
    if (ln_fwd(A, A + 4096, A + 8192, A + 16384, NULL, NULL, -1, 768, 1e-5f, NULL) != RN_ERR_SIZE)
        bad |= 8;
    if (rms_fwd(A, A + 4096, A + 8, 4, 16, 1e-5f, NULL) != RN_ERR_ALIAS) bad |= 16;
    if (ln_fwd_strided(RN_DTYPE_F32, RN_VARIANT_AUTO, A, 10, A, A, A + 4096, 12, NULL, NULL,
                       4, 12, 1e-5f, NULL) != RN_ERR_SIZE)
        bad |= 32;
    if (rn_selftest_bounded_wait(0, NULL) != RN_ERR_SIZE) bad |= 64;
    printf("%%d\n", bad);
    return bad;
}
"""


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\w[\w\s\*]*?\b(\w+)\s*\(", text, re.M)) - {"typedef"})


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_library_links_from_c(tmp_path):
    lib = os.path.join(LIBDIR, "librownorm.so")
    if not os.path.exists(lib):
        pytest.skip("library not built")
    names = _declared()
    assert {"ln_fwd", "rms_fwd", "ln_bwd", "ln_fwd_batched"} <= set(names)
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM % ", ".join(f"(fnptr){n}" for n in names))
    exe = tmp_path / "abi"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), "-L", LIBDIR, "-lrownorm",
                           f"-Wl,-rpath,{LIBDIR}"])
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, f"C program reported {out.stdout!r} {out.stderr!r}"
