"""include/smx.h is a C ABI: a plain C99 program (and a C++17 one) compiles
against it with every warning an error, links against the library and runs.
Without a device the program sees the host-side checks answer and the calls
that need a GPU report SMX_ERR_UNSUPPORTED; with one, the host-buffer call
returns a normalised row with +0 in its masked lanes.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <string.h>
#include "smx.h"

int main(void) {
    float x[2][8], y[2][8];
    int32_t vl[2] = {8, 3};
    smx_status st;
    int i, j;
    for (i = 0; i < 2; ++i)
        for (j = 0; j < 8; ++j) x[i][j] = (float)(j - 3 * i);
    if (smx_version() < 100) return 10;
    if (smx_status_string(SMX_ERR_ALIAS) == NULL) return 11;
    /* host-side checks answer before any CUDA call */
    if (smx_softmax_rows(x, y, -1, 8, NULL, SMX_F32, SMX_F32, NULL) != SMX_ERR_INVALID_ARG) return 12;
    if (smx_softmax_rows_host(x, (char *)x + 4, 2, 8, NULL, SMX_F32, SMX_F32, NULL) != SMX_ERR_ALIAS)
        return 13;
    if (smx_softmax_rows_host(NULL, NULL, 0, 8, NULL, SMX_F32, SMX_F32, NULL) != SMX_OK) return 14;
    if (smx_softmax_merge_stats(NULL, NULL, NULL, NULL, NULL, NULL, -1, NULL) != SMX_ERR_INVALID_ARG)
        return 15;
    memset(y, 0xff, sizeof y);
    st = smx_softmax_rows_host(x, y, 2, 8, vl, SMX_F32, SMX_F32, NULL);
    if (st == SMX_ERR_UNSUPPORTED) {
        printf("no device\n");
        return 0;
    }
    if (st != SMX_OK) return 20;
    if (smx_last_device_status(NULL) != SMX_OK) return 21;
    for (i = 0; i < 2; ++i) {
        double s = 0.0;
        for (j = 0; j < 8; ++j) s += y[i][j];
        if (fabs(s - 1.0) > 1e-5) return 22;
    }
    for (j = 3; j < 8; ++j)
        if (y[1][j] != 0.0f || signbit(y[1][j])) return 23;
    printf("device ok\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from numerically_stable_online_gb300 import build

    build.build()
    return os.path.join(ROOT, "numerically_stable_online_gb300", "_build")


@pytest.mark.parametrize("compiler,flags,suffix", [
    ("gcc", ["-std=c99", "-pedantic"], ".c"),
    ("g++", ["-std=c++17", "-pedantic"], ".cpp"),
])
def test_header_compiles_links_and_runs(libdir, tmp_path, compiler, flags, suffix):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    src = tmp_path / f"prog{suffix}"
    src.write_text(PROGRAM)
    exe = tmp_path / "prog"
    cmd = [compiler, *flags, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-L", libdir, "-lsmx", f"-Wl,-rpath,{libdir}", "-lm", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() in ("no device", "device ok")
