"""The emulated traffic counter against the pages' communication formulas.

The collectives are emulated in one GPU's memory, so no byte crosses a
link; ``comm_counter`` adds up what each accepted call's ranks would send if
its collective ran as a ring (the model of "Infra: Data Parallel", ZeRO
section, and "4.1 数据并行详解" sections 5 and 8, with the (N_d - 1) / N_d
factor kept).  These tests run the steps the pages count and compare the
counter with the ledger's exact volumes (``comm_bytes(..., exact=True)``,
itself pinned by the printed 4 Psi / 6 Psi figures and a simulated ring):
  ZeRO-1/2: one rank's fused step over its shard of every unit and the
            all-gather of every unit, 2 Psi + 2 Psi;
  ZeRO-3:   the same with the two all-gathers of every unit (forward and
            backward), 2 Psi + 2 Psi + 2 Psi;
  DDP:      the bucketed all-reduce of the whole gradient, 4 Psi;
  hybrid:   the reduce inside the group of F and across the groups plus the
            all-gather inside the group;
  FSDP2:    the reduce-scatter of the chunk-cat buffer and the all-gather
            copied out;
with Psi the padded element count, in bytes of the 16-bit (or, for fp32
contributions, 32-bit) elements moved."""
import numpy as np
import pytest
import torch

import sharded_optimizer_step_gb300 as ss
from sharded_optimizer_step_gb300.engine import RankShardOptimizer
from synth import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    yield
    torch.cuda.empty_cache()


def _rank_step(units, nd, F=None, gathers=1):
    """One rank's step: the fused update of its shard of every unit, then
    `gathers` all-gathers of every unit; returns (counter delta, padded Psi)."""
    opt = RankShardOptimizer(units, nd, 0, ss.AdamW(), device=DEV, shard_group=F or 0)
    fulls = [torch.empty(lay.padded, dtype=torch.bfloat16, device=DEV) for lay in opt.layouts]
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    opt.step()
    for _ in range(gathers):
        for u in range(len(units)):
            own = opt.unit_slice(opt.params, u)
            opt.gather_unit(u, [own] * opt.F, fulls[u])
    got = ss.comm_counter(reset=True)
    torch.cuda.synchronize()
    return got, sum(lay.padded for lay in opt.layouts)


@pytest.mark.parametrize("nd", [8, 7, 2])
def test_zero12_step_counts_2psi_plus_2psi(nd):
    units = W.gpt2_small().units
    got, psi = _rank_step(units, nd)
    assert psi % nd == 0 and (nd != 7 or psi > W.gpt2_small().psi)     # padded at N_d = 7
    for kind in ("zero1", "zero2"):
        assert got == pytest.approx(ss.comm_bytes(psi, nd, kind, exact=True), rel=1e-12)
    assert got == pytest.approx(4 * psi * (nd - 1) / nd, rel=1e-12)


def test_zero3_step_counts_6psi():
    units = W.gpt2_small().units
    got, psi = _rank_step(units, 8, gathers=2)
    assert got == pytest.approx(ss.comm_bytes(psi, 8, "zero3", exact=True), rel=1e-12)


@pytest.mark.parametrize("nd,F", [(16, 8), (8, 2), (8, 1)])
def test_hybrid_step_counts_intra_plus_inter(nd, F):
    units = W.gpt2_small().units[:4]
    got, psi = _rank_step(units, nd, F=F)
    want = (ss.hybrid_comm_bytes(psi, nd, F, "intra", exact=True) +
            ss.hybrid_comm_bytes(psi, nd, F, "inter", exact=True))
    assert got == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("nd", [8, 3])
@pytest.mark.parametrize("fused", [False, True])
def test_ddp_step_counts_4psi(nd, fused):
    unit = [768, 768, 768 * 3072, 768 * 3072, 1024 * 1024]
    numels = unit * 4 + [768 * 3072]
    _, _, boff = ss.ddp_bucket_plan(numels, 2, 4 << 20)
    psi = boff[-1]
    grads = [torch.zeros(psi, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    if fused:
        st = [torch.zeros(psi, device=DEV) for _ in range(3)]
        params = torch.empty(psi, dtype=torch.bfloat16, device=DEV)
        ss.ddp_bucket_allreduce_avg_adamw_cast(grads, boff, *st, params, ss.AdamW(), 1)
    else:
        out = torch.empty(psi, dtype=torch.bfloat16, device=DEV)
        for b in range(len(boff) - 1):      # bucket by bucket, as they become ready
            ss.ddp_bucket_allreduce_avg(grads, boff, out, first=b, count=1)
    got = ss.comm_counter(reset=True)
    assert got == pytest.approx(ss.comm_bytes(psi, nd, "ddp", exact=True), rel=1e-12)


def test_fsdp2_step_counts_rs_plus_ag():
    nd = 8
    shapes = [(4096, 4096), (11008, 4096), (4096,), (4099, 7)]
    lay = ss.fsdp2_layout(shapes, nd)
    L = lay.local
    grads = [torch.zeros(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    cc = [ss.fsdp2_chunk_cat(grads, nd) for _ in range(nd)]         # local: counts 0
    assert ss.comm_counter() == 0.0
    st = [torch.zeros(L, device=DEV) for _ in range(3)]
    out = torch.empty(L, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([c[:L] for c in cc], *st, out, ss.AdamW(), 1)
    params = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    ss.fsdp2_all_gather_copy_out([out] * nd, params)
    got = ss.comm_counter(reset=True)
    assert got == pytest.approx(ss.comm_bytes(nd * L, nd, "zero1", exact=True), rel=1e-12)
    # the same step read straight from the gradients counts the same bytes,
    # padding rows included
    shapes2 = [(4099, 7), (13,), (1030, 3)]
    L2 = ss.fsdp2_layout(shapes2, nd).local
    g2 = [[torch.zeros(s, dtype=torch.bfloat16, device=DEV) for s in shapes2] for _ in range(nd)]
    st2 = [torch.zeros(L2, device=DEV) for _ in range(3)]
    out2 = torch.empty(L2, dtype=torch.bfloat16, device=DEV)
    params2 = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes2]
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    ss.fsdp2_rs_avg_adamw_cast(g2, 0, *st2, out2, ss.AdamW(), 1)
    ss.fsdp2_all_gather_copy_out([out2] * nd, params2)
    got = ss.comm_counter(reset=True)
    assert got == pytest.approx(ss.comm_bytes(nd * L2, nd, "zero1", exact=True), rel=1e-12)


def test_fp32_contributions_and_the_scaler_flag():
    """The fused last micro-batch reduces fp32 sums: 4-byte elements; the
    gradient scaler's check adds only the all-reduce of its flag."""
    nd, S = 4, 70001
    acc = [torch.zeros(S, device=DEV) for _ in range(nd)]
    last = [torch.zeros(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    st = [torch.zeros(S, device=DEV) for _ in range(3)]
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    ss.fsdp_accumulate_rs_avg_adamw_cast(acc, last, 0.25, *st, out, ss.AdamW(), 1)
    assert ss.comm_counter(reset=True) == (nd - 1) * S * 4
    sc = ss.GradScaler(device=DEV)
    sc.check([x.to(torch.float16) for x in last])
    assert ss.comm_counter(reset=True) == pytest.approx(2 * (nd - 1) / nd * 4, rel=1e-15)
    torch.cuda.synchronize()
    assert np.isfinite(float(sc.scale.item()))
