"""The boundary from plain C: C99 programs that include only
include/shardstep.h and link libshardstep.so call the host-only entry
points (layout of the FlatParameter worked example, the memory ledger, an
argument error; a checkpoint saved by 2 ranks, its header read back,
verified and loaded into rank 1 of 3 through the reshard plan) and print
what they got.  No GPU is needed."""
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


CKPT_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "shardstep.h"

/* a unit of 10 fp32 values saved by 2 ranks (shards of 5), then rank 1 of
 * 3 (shard of 4: elements 4..7) loaded through the reshard plan */
int main(int argc, char** argv) {
    char path[2][512];
    float flat[10];
    for (int i = 0; i < 10; ++i) flat[i] = 0.5f * (float)i;
    const int64_t total = 10;
    for (int r = 0; r < 2; ++r) {
        snprintf(path[r], sizeof path[r], "%s/rank%d.shst", argc > 1 ? argv[1] : ".", r);
        shardstep_ckpt_section_t sec = {0, 0, 5 * (int64_t)sizeof(float), flat + 5 * r};
        int rc = shardstep_ckpt_save_rank(path[r], 2, r, 7, &total, 1, &sec, 1);
        if (rc != 0) { printf("save %d %s\n", rc, shardstep_last_error()); return 1; }
    }
    shardstep_ckpt_info_t info;
    int64_t totals[1];
    int rc = shardstep_ckpt_info(path[1], &info, totals, 1);
    printf("info %d %d %d %d %lld %lld\n", rc, info.nd, info.rank, info.n_sections,
           (long long)info.step, (long long)totals[0]);
    printf("verify %d %d\n", shardstep_ckpt_verify(path[0]), shardstep_ckpt_verify(path[1]));
    shardstep_ckpt_piece_t pieces[4];
    int32_t n = 0;
    rc = fsdp_reshard_plan(total, 2, 3, 1, pieces, 4, &n);
    float got[4] = {0, 0, 0, 0};
    for (int k = 0; k < n && rc == 0; ++k)
        rc = shardstep_ckpt_read(path[pieces[k].old_rank], 0, 0,
                                 pieces[k].old_offset * (int64_t)sizeof(float),
                                 pieces[k].count * (int64_t)sizeof(float),
                                 got + pieces[k].new_offset);
    printf("load %d %d %.1f %.1f %.1f %.1f\n", rc, n, got[0], got[1], got[2], got[3]);
    return 0;
}
"""


def test_c99_program_saves_and_reshards_a_checkpoint(built, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "ckpt.c"
    src.write_text(CKPT_PROGRAM)
    exe = tmp_path / "ckpt"
    lib = _capi.lib_path()
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True,
                         check=True).stdout.split("\n")
    assert out[0] == "info 0 2 1 1 7 10"
    assert out[1] == "verify 0 0"
    # rank 1 of 3 holds elements 4..7: the last of old shard 0, the first three of shard 1
    assert out[2] == "load 0 2 2.0 2.5 3.0 3.5"
