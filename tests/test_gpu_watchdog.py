"""The TMA-staged kernels' bounded waits, made to run out on purpose.

"4.1 数据并行详解" section 4.2 names the failure this guards against: a wait
that never ends (there a bucket that never fills).  Every wait of a TMA-staged
kernel -- a consumer warp's for a staged tile, the producer's for a free
stage -- has a limit, after which the kernel sets a bit of the device status
word and returns.  Here the limit is set to 1 ns, so the waits run out even
though every copy lands; each kernel must still return, set the status and
leave the context usable, the block's own bulk copies drained before it
exits (status bit 2 stays clear), and the next call with the default limit
must match the oracle bit for bit.  Nothing here can fault or hang the GPU:
the copies read valid device memory and the drain has its own fixed limit."""
import numpy as np
import pytest
import torch

import oracle
import oracle.scaler as osc
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = AdamWConfig(1e-3, 0.9, 0.999, 1e-8, 0.01)
HPC = ss.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
S = 2048 * 152 * 6 + 2048 * 3 + 8 * 5 + 3      # several tiles per block, a ragged tail
DRAIN_BIT = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    ss.device_status(clear=True)
    yield
    ss.set_tma_wait_ns(0)
    assert ss.device_status() == 0


@pytest.fixture
def tma_path():
    prev = ss.set_fused_path("tma")
    yield
    ss.set_fused_path(prev)


def _dev16(h):
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(DEV)


def _short_limit_then_default(run, tries=3):
    """Runs `run` under a 1 ns wait limit (up to `tries` launches, until one
    of them reports a wait that ran out) and returns the status bits."""
    prev = ss.set_tma_wait_ns(1)
    assert prev == 2_000_000_000
    st = 0
    try:
        for _ in range(tries):
            run()
            torch.cuda.synchronize()          # the launch ends: no wait lasts
            st |= ss.device_status(clear=True)
            if st & 3:
                break
    finally:
        assert ss.set_tma_wait_ns(0) == 1
    return st


def _grads(nd, dtype="bf16", seed=0):
    return [synth.host_fill(synth.normal_stream(seed, (85, q), 1e-3), 0, S, dtype)
            for q in range(nd)]


@pytest.mark.parametrize("nd", [8, 9])
def test_fused_step_wait_runs_out_then_recovers(nd, tma_path):
    gh = _grads(nd)
    grads = [_dev16(h).view(torch.bfloat16) for h in gh]
    p = synth.host_fill(synth.normal_stream(1, (85, 99), 0.02), 0, S, "f32")
    master = torch.from_numpy(p.copy()).to(DEV)
    m = torch.zeros(S, device=DEV)
    v = torch.zeros(S, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)

    st = _short_limit_then_default(
        lambda: ss.fsdp_rs_avg_adamw_cast(grads, master, m, v, out, HPC, 1))
    assert ss.last_kernel() == "staged_stream<AdamOp<bf16>> (TMA-staged)"
    assert st & 3, "no wait ran out under a 1 ns limit"
    assert not st & DRAIN_BIT, "a block exited before its own copies had landed"

    # the results of the cut-short launch are incomplete; start again
    master.copy_(torch.from_numpy(p))
    m.zero_()
    v.zero_()
    ss.fsdp_rs_avg_adamw_cast(grads, master, m, v, out, HPC, 1)
    z = np.zeros(S, np.float32)
    p1, m1, v1, o1 = oracle.fsdp_shard_step(gh, 0, S, p, z, z, HP, 1)
    torch.cuda.synchronize()
    assert ss.device_status() == 0
    assert_bits(master.cpu().numpy(), p1, "master")
    assert_bits(m.cpu().numpy(), m1, "m")
    assert_bits(v.cpu().numpy(), v1, "v")
    assert_bits(out.view(torch.int16).cpu().numpy().view(np.uint16), o1, "bf16")


def test_bucket_allreduce_wait_runs_out_then_recovers(tma_path):
    nd = 8
    gh = _grads(nd, seed=2)
    grads = [_dev16(h).view(torch.bfloat16) for h in gh]
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    boff = [0, S // 2 & ~7, S]                # two buckets: a dependent launch too
    st = _short_limit_then_default(lambda: ss.ddp_bucket_allreduce_avg(grads, boff, out))
    assert st & 3 and not st & DRAIN_BIT
    ss.ddp_bucket_allreduce_avg(grads, boff, out)
    torch.cuda.synchronize()
    assert ss.device_status() == 0
    assert_bits(out.view(torch.int16).cpu().numpy().view(np.uint16),
                oracle.bucket_allreduce_avg(gh, boff), "avg")


def test_accumulate_wait_runs_out_then_recovers(tma_path):
    gh = _grads(2, seed=3)
    acc = torch.empty(S, device=DEV)
    g = [_dev16(h).view(torch.bfloat16) for h in gh]
    st = _short_limit_then_default(lambda: ss.fsdp_grad_accumulate(g[0], acc, 0.5, True))
    assert st & 3 and not st & DRAIN_BIT
    ss.fsdp_grad_accumulate(g[0], acc, 0.5, True)
    ss.fsdp_grad_accumulate(g[1], acc, 0.5, False)
    torch.cuda.synchronize()
    assert ss.device_status() == 0
    assert_bits(acc.cpu().numpy(), oracle.grad_accumulate(gh, np.float32(0.5)), "acc")


def test_check_wait_runs_out_then_recovers(tma_path):
    nd = 5
    hs = [synth.host_fill(synth.normal_stream(4, (85, q), 0.3), 0, S, "f16") for q in range(nd)]
    hs[2][S - 9] = 0x7C00
    grads = [_dev16(h).view(torch.float16) for h in hs]
    sc = ss.GradScaler(init_scale=128.0, device=DEV)
    st = _short_limit_then_default(lambda: sc.check(grads))
    assert st & 3 and not st & DRAIN_BIT
    sc.found_inf.zero_()
    sc.check(grads)
    want = osc.found_inf([(h, "f16") for h in hs], nd, 0, S, np.float32(1.0 / 128.0))
    torch.cuda.synchronize()
    assert ss.device_status() == 0
    assert bool(int(sc.found_inf.item())) == want is True


def test_wait_limit_setting_is_validated():
    with pytest.raises(ss.ShardstepError):
        ss.set_tma_wait_ns(-1)
    assert ss.set_tma_wait_ns(0) == 2_000_000_000
