"""The boundary from plain C: a C99 program that includes only
include/shardstep.h and links libshardstep.so calls the host-only entry
points (layout of the FlatParameter worked example, the memory ledger, an
argument error) and prints what it got.  No GPU is needed."""
import os
import shutil
import subprocess

import pytest

import sharded_optimizer_step_gb300 as ss
from sharded_optimizer_step_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "shardstep.h"

int main(void) {
    /* "Infra: Data Parallel", FSDP1 figure: three (4,2) weights, two ranks */
    const int64_t numels[3] = {8, 8, 8};
    shardstep_layout_info_t info;
    int64_t off[3], lo[6], hi[6];
    int rc = fsdp_layout(numels, 3, 2, &info, off, lo, hi);
    printf("layout %d %lld %lld %lld\n", rc, (long long)info.total, (long long)info.padded,
           (long long)info.shard);
    printf("offsets %lld %lld %lld\n", (long long)off[0], (long long)off[1], (long long)off[2]);
    /* the ZeRO-3 state per GPU at psi = 7e9, N_d = 8, k = 12 */
    printf("zero3 %.3f\n", shardstep_state_bytes(7e9, 8, 3, 12.0) / 1e9);
    rc = fsdp_layout(numels, 3, 0, &info, off, lo, hi);
    printf("bad %d %s\n", rc, shardstep_last_error());
    printf("sizes %u %u\n", (unsigned)sizeof(shardstep_adamw_t),
           (unsigned)sizeof(shardstep_adamw_state_t));
    return 0;
}
"""


@pytest.fixture(scope="module")
def built():
    ss.build()


def test_c99_program_calls_the_library(built, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_shardstep.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_shardstep"
    lib = _capi.lib_path()
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0] == "layout 0 24 24 12"
    assert out[1] == "offsets 0 8 16"
    assert out[2] == "zero3 14.000"
    assert out[3].startswith("bad -1 ") and "nd" in out[3]
    assert out[4] == "sizes 48 56"
