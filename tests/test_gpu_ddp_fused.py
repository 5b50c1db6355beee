"""DDP's replicated step fused: bucket all-reduce average + AdamW + bf16 cast
in one pass (``ddp_bucket_allreduce_avg_adamw_cast``).

"Infra: Data Parallel", section "Naïve Data Parallelism", and "4.1 数据并行详解"
section 4.2: the gradients are all-reduce-averaged bucket by bucket (bf16,
the dtype the all-reduce keeps) and every rank runs the same update.  The
fused call must give the oracle's ``ddp_step`` bit for bit -- the update
consumes the bf16-rounded mean -- and the same bits as the two calls it
replaces, whether buckets are updated one by one as they become ready or all
at once, with or without the averaged gradient kept."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = AdamWConfig(1e-3, 0.9, 0.999, 1e-8, 0.01)
HPC = ss.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    yield
    assert ss.device_status() == 0


def _dev16(h, shift=0):
    buf = torch.empty(h.size + shift + 8, dtype=torch.int16, device=DEV)
    t = buf[shift:shift + h.size]
    t.copy_(torch.from_numpy(np.ascontiguousarray(h).view(np.int16)))
    return t.view(torch.bfloat16)


def _devf(x, shift=0):
    buf = torch.empty(x.size + shift + 8, dtype=torch.float32, device=DEV)
    t = buf[shift:shift + x.size]
    t.copy_(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)))
    return t


def _h16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


NUMELS = [768, 3, 768 * 30, 5, 4096 * 3, 768, 1, 2000, 70_001]


@pytest.mark.parametrize("nd", [1, 2, 3, 5, 8, 9, 11, 13, 16, 64])
@pytest.mark.parametrize("cap", [64, 5000, 1 << 22])
@pytest.mark.parametrize("keep_mean", [True, False])
@pytest.mark.parametrize("shift", [0, 1])
def test_fused_ddp_step_matches_oracle(nd, cap, keep_mean, shift):
    off, of, boff = ss.ddp_bucket_plan(NUMELS, 2, cap)
    total = boff[-1]
    steps = 2
    ph = synth.host_fill(synth.normal_stream(nd, (86, 100), 0.02), 0, total, "f32")
    master, m, v = _devf(ph, shift), _devf(np.zeros(total), shift), _devf(np.zeros(total), shift)
    params = _dev16(np.zeros(total, np.uint16), shift)
    mean = _dev16(np.zeros(total, np.uint16), shift) if keep_mean else None
    p, mm, vv = ph, np.zeros(total, np.float32), np.zeros(total, np.float32)
    for t in range(1, steps + 1):
        gh = [synth.host_fill(synth.normal_stream(nd, (86, t, q), 1e-3), 0, total, "bf16")
              for q in range(nd)]
        grads = [_dev16(h, (q + shift) % 2) for q, h in enumerate(gh)]
        for b in range(len(boff) - 1):        # bucket by bucket, as each is ready
            ss.ddp_bucket_allreduce_avg_adamw_cast(grads, boff, master, m, v, params, HPC, t,
                                                   mean_out=mean, first=b, count=1)
        avg, p, mm, vv, pb = oracle.ddp_step(gh, boff, p, mm, vv, HP, t)
        torch.cuda.synchronize()
        if keep_mean:
            assert_bits(_h16(mean), avg, f"mean, step {t}")
    assert_bits(master.cpu().numpy(), p, "master")
    assert_bits(m.cpu().numpy(), mm, "m")
    assert_bits(v.cpu().numpy(), vv, "v")
    assert_bits(_h16(params), pb, "params")


def test_fused_ddp_step_equals_the_two_calls_on_the_ddp_sweep_shape():
    """Psi = 351M (the DDP bucketing sweep's parameter list), N_d = 8, caps of
    1 and 256 MiB: one fused call over all buckets and the bucket all-reduce
    followed by the fused step at N_d = 1 agree on every element over two
    steps."""
    unit = [768, 768, 768 * 3072, 768 * 3072, 4096 * 4096]
    numels = unit * 16 + [768 * 3072] * 3
    total = sum(numels)
    assert total == 351_035_392
    nd = 8
    grads = [torch.empty(total, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    for cap in (1 << 20, 256 << 20):
        off, of, boff = ss.ddp_bucket_plan(numels, 2, cap)
        a = {k: torch.empty(total, device=DEV) for k in ("p", "m", "v")}
        synth.dev_fill(synth.normal_stream(5, (87, 0), 0.02), a["p"])
        a["m"].zero_()
        a["v"].zero_()
        b = {k: x.clone() for k, x in a.items()}
        pa = torch.empty(total, dtype=torch.bfloat16, device=DEV)
        pb = torch.empty_like(pa)
        mean_a = torch.empty_like(pa)
        mean_b = torch.empty_like(pa)
        for t in (1, 2):
            for q in range(nd):
                synth.dev_fill(synth.normal_stream(5, (87, t, q), 1e-3), grads[q])
            before = ss.launch_count()
            ss.ddp_bucket_allreduce_avg_adamw_cast(grads, boff, a["p"], a["m"], a["v"], pa, HPC,
                                                   t, mean_out=mean_a)
            assert ss.launch_count() - before == 1
            assert ss.last_kernel() == "ddp_allreduce_adamw_cast_vec4<8> (register-staged)"
            ss.ddp_bucket_allreduce_avg(grads, boff, mean_b)
            ss.fsdp_rs_avg_adamw_cast([mean_b], b["p"], b["m"], b["v"], pb, HPC, t)
        torch.cuda.synchronize()
        assert torch.equal(mean_a.view(torch.int16), mean_b.view(torch.int16)), cap
        for k in ("p", "m", "v"):
            assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), (cap, k)
        assert torch.equal(pa.view(torch.int16), pb.view(torch.int16)), cap
    # and sampled elements against the oracle (the last cap's final step)
    rng = np.random.default_rng(5)
    loc = np.unique(rng.integers(0, total, 20_000))
    it = torch.from_numpy(loc).to(DEV)
    ph = synth.host_gather(synth.normal_stream(5, (87, 0), 0.02), loc, "f32")
    g1, g2 = ([synth.host_gather(synth.normal_stream(5, (87, t, q), 1e-3), loc, "bf16")
               for q in range(nd)] for t in (1, 2))
    z = np.zeros(loc.size, np.float32)
    _, p1, m1, v1, _ = oracle.ddp_step(g1, [0, loc.size], ph, z, z, HP, 1)
    avg, p2, m2, v2, pb2 = oracle.ddp_step(g2, [0, loc.size], p1, m1, v1, HP, 2)
    assert_bits(_h16(mean_a[it]), avg, "mean")
    assert_bits(a["p"][it].cpu().numpy(), p2, "master")
    assert_bits(a["m"][it].cpu().numpy(), m2, "m")
    assert_bits(a["v"][it].cpu().numpy(), v2, "v")
    assert_bits(_h16(pa[it]), pb2, "params")


def test_fused_ddp_rejects_overlaps_and_bad_ranges():
    total = 4096
    g = [torch.zeros(total, dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    p, m, v = (torch.zeros(total, device=DEV) for _ in range(3))
    pb = torch.zeros(total, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ss.ShardstepError):           # params is a gradient
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, total], p, m, v, g[1], HPC, 1)
    with pytest.raises(ss.ShardstepError):           # mean_out is the parameters
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, total], p, m, v, pb, HPC, 1,
                                               mean_out=pb)
    with pytest.raises(ss.ShardstepError):           # m is v
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, total], p, v, v, pb, HPC, 1)
    with pytest.raises(ss.ShardstepError):           # step 0
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, total], p, m, v, pb, HPC, 0)
    with pytest.raises(ValueError):
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, total], p, m, v, pb, HPC, 1, first=1,
                                               count=1)
