"""The whole step from a plain C client, with no Python or PyTorch in it.

A C99 program that includes only include/shardstep.h and the CUDA runtime's
C header, and links libshardstep.so and libcudart, reads a unit's tensors
from a file, allocates device memory with cudaMalloc, and runs one
optimizer step of every rank through the C ABI on a stream of its own: pack
the fp32 master and each rank's bf16 gradients into FlatParameters
("Infra: Data Parallel", FSDP1 section), every rank's fused reduce-scatter
average + AdamW + bf16 cast, the all-gather of the ranks' shards and the
views of the gathered unit.  The test compares what it writes back with the
oracle, bit for bit."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from sharded_optimizer_step_gb300 import _capi
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "shardstep.h"

#define MAXT 16
#define CK(x) do { int rc_ = (x); if (rc_ != SHARDSTEP_OK) { \
    fprintf(stderr, "%s: %d %s\n", #x, rc_, shardstep_last_error()); return 2; } } while (0)
#define CU(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 3; } } while (0)

static int rd(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }

int main(int argc, char** argv) {
    if (argc != 3) return 1;
    FILE* in = fopen(argv[1], "rb");
    if (!in) return 1;
    int32_t nd, n, step;
    double h[5];
    int64_t numels[MAXT];
    if (rd(in, &nd, 4) || rd(in, &n, 4) || rd(in, &step, 4) || rd(in, h, sizeof h)) return 1;
    if (n < 1 || n > MAXT || nd < 1 || nd > 64) return 1;
    if (rd(in, numels, 8 * (size_t)n)) return 1;

    shardstep_layout_info_t info;
    int64_t off[MAXT];
    int64_t* lo = malloc(sizeof(int64_t) * (size_t)n * (size_t)nd);
    int64_t* hi = malloc(sizeof(int64_t) * (size_t)n * (size_t)nd);
    CK(fsdp_layout(numels, n, nd, &info, off, lo, hi));
    const int64_t T = info.total, P = info.padded, S = info.shard;

    cudaStream_t st;
    CU(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
    /* the unit's fp32 master tensors and every rank's bf16 gradient tensors */
    void* mt[MAXT];
    void** gt = malloc(sizeof(void*) * (size_t)n * (size_t)nd);
    for (int t = 0; t < n; ++t) {
        size_t b = 4 * (size_t)numels[t];
        void* hbuf = malloc(b + 1);
        if (rd(in, hbuf, b)) return 1;
        CU(cudaMalloc(&mt[t], b + 16));
        CU(cudaMemcpy(mt[t], hbuf, b, cudaMemcpyHostToDevice));
        free(hbuf);
    }
    for (int q = 0; q < nd; ++q)
        for (int t = 0; t < n; ++t) {
            size_t b = 2 * (size_t)numels[t];
            void* hbuf = malloc(b + 1);
            if (rd(in, hbuf, b)) return 1;
            CU(cudaMalloc(&gt[q * n + t], b + 16));
            CU(cudaMemcpy(gt[q * n + t], hbuf, b, cudaMemcpyHostToDevice));
            free(hbuf);
        }
    fclose(in);

    float *master, *m, *v;
    uint16_t *full, *shards;
    uint16_t** gflat = malloc(sizeof(uint16_t*) * (size_t)nd);
    CU(cudaMalloc((void**)&master, 4 * (size_t)P));
    CU(cudaMalloc((void**)&m, 4 * (size_t)P));
    CU(cudaMalloc((void**)&v, 4 * (size_t)P));
    CU(cudaMalloc((void**)&full, 2 * (size_t)P));
    CU(cudaMalloc((void**)&shards, 2 * (size_t)P));
    CU(cudaMemsetAsync(m, 0, 4 * (size_t)P, st));
    CU(cudaMemsetAsync(v, 0, 4 * (size_t)P, st));
    for (int q = 0; q < nd; ++q) CU(cudaMalloc((void**)&gflat[q], 2 * (size_t)P));

    /* pack: the master once, each rank's gradient */
    CK(fsdp_flat_pack((const void* const*)mt, numels, n, nd, SHARDSTEP_DTYPE_F32, master, st));
    for (int q = 0; q < nd; ++q)
        CK(fsdp_flat_pack((const void* const*)&gt[q * n], numels, n, nd, SHARDSTEP_DTYPE_BF16,
                          gflat[q], st));

    /* every rank's fused step on its shard: slice r of each rank's gradient */
    shardstep_adamw_t hp = {h[0], h[1], h[2], h[3], h[4], step};
    const void** slices = malloc(sizeof(void*) * (size_t)nd);
    const uint16_t** outs = malloc(sizeof(uint16_t*) * (size_t)nd);
    for (int r = 0; r < nd; ++r) {
        for (int q = 0; q < nd; ++q) slices[q] = gflat[q] + (size_t)r * (size_t)S;
        CK(fsdp_rs_avg_adamw_cast(slices, SHARDSTEP_DTYPE_BF16, nd, S, master + r * S,
                                  m + r * S, v + r * S, shards + r * S, &hp, st));
        outs[r] = shards + r * S;
    }
    /* all-gather the bf16 shards into the unit's full flat buffer */
    CK(fsdp_ag_unpack(outs, nd, S, full, st));
    CU(cudaStreamSynchronize(st));

    /* views of the gathered unit: offsets and counts */
    void* vp[MAXT];
    int64_t cnt[MAXT];
    CK(fsdp_views(numels, n, nd, -1, full, 2, vp, cnt));
    FILE* out = fopen(argv[2], "wb");
    if (!out) return 1;
    int64_t hdr[3] = {T, P, S};
    fwrite(hdr, 8, 3, out);
    for (int t = 0; t < n; ++t) {
        int64_t o = (int64_t)((uint16_t*)vp[t] - full);
        fwrite(&o, 8, 1, out);
        fwrite(&cnt[t], 8, 1, out);
    }
    void* hb = malloc(4 * (size_t)P + 1);
    float* devs[3] = {master, m, v};
    for (int k = 0; k < 3; ++k) {
        CU(cudaMemcpy(hb, devs[k], 4 * (size_t)P, cudaMemcpyDeviceToHost));
        fwrite(hb, 4, (size_t)P, out);
    }
    CU(cudaMemcpy(hb, full, 2 * (size_t)P, cudaMemcpyDeviceToHost));
    fwrite(hb, 2, (size_t)P, out);
    fclose(out);
    printf("ok %lld %lld %lld\n", (long long)T, (long long)P, (long long)S);
    return 0;
}
"""


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    ss.build()
    d = tmp_path_factory.mktemp("c_client")
    src = d / "step_client.c"
    src.write_text(PROGRAM)
    path = d / "step_client"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib = _capi.lib_path()
    libdirs = [p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib"))
               if os.path.isdir(p)]
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           str(src), lib, *[f"-L{p}" for p in libdirs], "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib),
           *[f"-Wl,-rpath,{p}" for p in libdirs], "-o", str(path)]
    subprocess.run(cmd, check=True)
    return path


CASES = [([(4, 2), (4, 2), (4, 2)], 2),                # the FSDP1 figure's unit
         ([(1024, 96), (96,), (0,), (4099,), (37, 3)], 8),
         ([(70001,), (5, 5)], 3),
         ([(2048 * 152 + 13,)], 4)]


@pytest.mark.parametrize("shapes,nd", CASES, ids=["figure", "nd8_ragged", "nd3", "nd4_large"])
def test_c_client_runs_the_step(exe, tmp_path, shapes, nd):
    numels = [int(np.prod(s)) for s in shapes]
    hp = AdamWConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    step = 3
    seed = 17 + nd + sum(numels)
    mh = [synth.host_fill(synth.normal_stream(seed, (1, t), 0.02), 0, n, "f32")
          for t, n in enumerate(numels)]
    gh = [[synth.host_fill(synth.normal_stream(seed, (2, q, t), 1e-3), 0, n, "bf16")
           for t, n in enumerate(numels)] for q in range(nd)]
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(struct.pack("<iii", nd, len(numels), step))
        f.write(struct.pack("<5d", hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay))
        f.write(np.array(numels, dtype="<i8").tobytes())
        for x in mh:
            f.write(x.astype("<f4").tobytes())
        for q in range(nd):
            for x in gh[q]:
                f.write(x.astype("<u2").tobytes())
    outp = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(inp), str(outp)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr

    # the oracle: pack, every rank's shard step at step 3 from zero moments, gather
    want_p, lay = oracle.flat_pack(mh, nd)
    want_g = [oracle.flat_pack(g, nd)[0] for g in gh]
    S, P = lay.shard, lay.padded
    z = np.zeros(S, np.float32)
    res = [oracle.fsdp_shard_step(want_g, rr, S, want_p[rr * S:(rr + 1) * S], z, z, hp, step)
           for rr in range(nd)]
    want_full, _ = oracle.ag_unpack([x[3] for x in res], lay)

    raw = outp.read_bytes()
    T_, P_, S_ = struct.unpack_from("<3q", raw, 0)
    assert (T_, P_, S_) == (lay.total, P, S)
    pos = 24
    for t, nt in enumerate(numels):
        o, c = struct.unpack_from("<2q", raw, pos)
        pos += 16
        assert (o, c) == (lay.offsets[t], nt), t
    arrs = []
    for dt in ("<f4", "<f4", "<f4"):
        arrs.append(np.frombuffer(raw, dtype=dt, count=P, offset=pos))
        pos += 4 * P
    got_full = np.frombuffer(raw, dtype="<u2", count=P, offset=pos)
    assert pos + 2 * P == len(raw)
    for name, got, k in (("master", arrs[0], 0), ("m", arrs[1], 1), ("v", arrs[2], 2)):
        assert_bits(got, np.concatenate([x[k] for x in res]), name)
    assert_bits(got_full, want_full, "gathered unit")
