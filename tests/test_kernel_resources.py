"""No kernel of the library spills registers or uses local memory.

Every kernel is a streaming pass whose speed rests on keeping each thread's
loads in registers; a spill turns part of them into local-memory traffic
(the fused step with 16 fp32 slices, compiled for a fixed N_d, spilled 136
bytes per thread and ran 9% slower than the loop over any N_d).  ptxas
reports spills and local-memory use per kernel; this compiles every CUDA
translation unit with the library's own flags (cross-compiling: no GPU is
needed) and fails on any such report."""
import importlib
import os
import shutil
import subprocess
import tempfile

import pytest

B = importlib.import_module("sharded_optimizer_step_gb300.build")

CUDA_SOURCES = [s for s in B.SOURCES if s.endswith(".cu")]


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not on PATH")
def test_no_kernel_spills_or_local_memory():
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        for src in CUDA_SOURCES:
            cmd = ["nvcc", *B.nvcc_flags(), "-Xptxas", "-warn-spills,-warn-lmem-usage", "-c",
                   os.path.join(B.CSRC, src), "-o", os.path.join(tmp, src + ".o")]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
        reports = []
        for src, p in procs:
            out, _ = p.communicate()
            assert p.returncode == 0, f"nvcc failed on {src}:\n{out}"
            reports += [f"{src}: {line}" for line in out.splitlines()
                        if "spill" in line.lower() or "local memory" in line.lower()]
    assert not reports, "\n".join(reports)
