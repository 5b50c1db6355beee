"""The division by N_d that ends every reduce, and the light reduce kernels at
the world sizes that are not powers of two.

"4.1 数据并行详解" section 2: the data-parallel gradient is the mean of the
N_d local-mean gradients, so each reduce divides its rank-order fp32 sum by
N_d.  The kernels divide without a divide instruction (an exact reciprocal
for a power of two, else RN(1/N_d) and one fma correction); the first test
runs that division and IEEE fp32 division on all 2^32 fp32 bit patterns for
every N_d the library accepts and requires the same bits everywhere.  The
others compare the bucket all-reduce and the gradient scaler's check at N_d =
3, 5, 6 and 7 (and at 9..64, past the compiled counts) with the oracle,
under every kernel choice, on buckets with ragged tails, unaligned starts
and one planted non-finite value."""
import numpy as np
import pytest
import torch

import oracle
import oracle.scaler as osc
import sharded_optimizer_step_gb300 as ss
import synth
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    yield
    assert ss.device_status() == 0


@pytest.fixture(params=["auto", "register", "tma"])
def path(request):
    prev = ss.set_fused_path(request.param)
    yield request.param
    ss.set_fused_path(prev)


def _dev16(h, shift=0):
    buf = torch.empty(h.size + shift + 8, dtype=torch.int16, device=DEV)
    t = buf[shift:shift + h.size]
    t.copy_(torch.from_numpy(np.ascontiguousarray(h).view(np.int16)))
    return t


def test_division_by_every_nd_is_ieee_on_all_fp32_inputs():
    bad = {}
    for nd in range(1, ss.MAX_ND + 1):
        n, first = ss.check_mean_division(nd, device=DEV)
        if n:
            bad[nd] = (n, hex(first))
    assert not bad, f"patterns whose quotient differs from IEEE division: {bad}"


def test_division_check_reports_a_mismatch_count_of_the_right_form():
    # the count is added to the caller's word: two calls on one word double it
    # (zero stays zero), and the smallest bad pattern stays the sentinel
    count = torch.zeros(1, dtype=torch.int64, device=DEV)
    first = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    import ctypes
    from sharded_optimizer_step_gb300 import _capi
    for _ in range(2):
        _capi.check("shardstep_check_mean_division", _capi.lib().shardstep_check_mean_division(
            3, ctypes.c_void_p(count.data_ptr()), ctypes.c_void_p(first.data_ptr()), None))
    torch.cuda.synchronize()
    assert int(count.item()) == 0 and int(first.item()) == -1
    for nd in (0, ss.MAX_ND + 1):
        with pytest.raises(ss.ShardstepError):
            ss.check_mean_division(nd, device=DEV)


@pytest.mark.parametrize("nd", [3, 5, 6, 7])
def test_bucket_allreduce_light_nd_matches_oracle(nd, path):
    # buckets: large ones with ragged tails (several vectors per thread, the
    # last group of a thread partly past the end), a 16-byte aligned one, a
    # tiny one, one whose start is not 8-byte aligned
    boff = [0, 300_001, 300_001 + 4099, 300_001 + 4099 + 65_536, 300_001 + 4099 + 65_536 + 7,
            300_001 + 4099 + 65_536 + 7 + 1_048_579]
    total = boff[-1]
    gh = [synth.host_fill(synth.normal_stream(nd, (81, q), 1e-3), 0, total, "bf16")
          for q in range(nd)]
    # large sums in one rank push some means to the edge of bf16's range
    gh[0][:: 997] = 0x7F00
    grads = [_dev16(h) for h in gh]
    out = torch.empty(total, dtype=torch.int16, device=DEV)
    for b in range(len(boff) - 1):
        ss.ddp_bucket_allreduce_avg([g.view(torch.bfloat16) for g in grads], boff,
                                    out.view(torch.bfloat16), first=b, count=1)
    torch.cuda.synchronize()
    assert_bits(out.cpu().numpy().view(np.uint16), oracle.bucket_allreduce_avg(gh, boff), "avg")


@pytest.mark.parametrize("nd", [3, 5, 6, 7])
@pytest.mark.parametrize("where", [None, 0, 1, 2, 3, "last"])
def test_check_light_nd_finds_one_planted_value(nd, where, path):
    """One +inf in one rank's fp16 slice is found in whichever of a thread's
    vectors it sits (the kernel loads several vectors per thread before
    summing); a clean gradient sets nothing."""
    S = 128 * 8 * 4 * 40 + 4 * 5 + 3
    hs = [synth.host_fill(synth.normal_stream(nd, (82, q), 0.3), 0, S, "f16") for q in range(nd)]
    if where is not None:
        pos = S - 1 if where == "last" else (128 * 8 * 4 * 17 + where * 128 * 4 + 4 * 33 + 2)
        hs[nd - 1][pos] = 0x7C00
    sc = ss.GradScaler(init_scale=256.0, device=DEV)
    sc.check([_dev16(h).view(torch.float16) for h in hs])
    want = osc.found_inf([(h, "f16") for h in hs], nd, 0, S, np.float32(1.0 / 256.0))
    torch.cuda.synchronize()
    assert bool(int(sc.found_inf.item())) == want == (where is not None)


@pytest.mark.parametrize("nd", [3, 5, 6, 7])
def test_fused_step_non_power_of_two_nd_matches_oracle(nd, path):
    """The fused step divides by N_d with the same correction; sums that take
    the IEEE fallback (zeros, subnormals) sit among the ordinary ones."""
    from oracle.numerics import AdamWConfig
    hp = AdamWConfig(1e-3, 0.9, 0.999, 1e-8, 0.01)
    hpc = ss.AdamW(1e-3, 0.9, 0.999, 1e-8, 0.01)
    S = 2048 * 152 + 4099
    gh = [synth.host_fill(synth.normal_stream(nd, (83, q), 1e-3), 0, S, "bf16")
          for q in range(nd)]
    for q in range(nd):
        gh[q][5::101] = 0                 # zero sums
        gh[q][7::211] = 0x0001 if q == 0 else 0   # a subnormal sum
    p = synth.host_fill(synth.normal_stream(nd, (83, 99), 0.02), 0, S, "f32")
    master = torch.from_numpy(p.copy()).to(DEV)
    m = torch.zeros(S, device=DEV)
    v = torch.zeros(S, device=DEV)
    out = torch.empty(S, dtype=torch.int16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([_dev16(h).view(torch.bfloat16) for h in gh], master, m, v,
                              out.view(torch.bfloat16), hpc, 1)
    z = np.zeros(S, np.float32)
    p1, m1, v1, o1 = oracle.fsdp_shard_step(gh, 0, S, p, z, z, hp, 1)
    torch.cuda.synchronize()
    assert_bits(master.cpu().numpy(), p1, "master")
    assert_bits(m.cpu().numpy(), m1, "m")
    assert_bits(v.cpu().numpy(), v1, "v")
    assert_bits(out.cpu().numpy().view(np.uint16), o1, "bf16")


@pytest.mark.parametrize("nd", [9, 16, 23, 33, 64])
def test_light_kernels_at_large_nd_match_oracle(nd, path):
    """Past N_d = 8 the all-reduce and the check take the TMA-staged kernel
    where two stages fit (N_d <= 22 for 16-bit slices) and the register
    kernel's loop over batches of 8 slices beyond: both against the oracle,
    buckets with a ragged tail and an unaligned start, one planted inf."""
    boff = [0, 2048 * 152 + 4099, 2048 * 152 + 4099 + 13, 2048 * 152 + 4099 + 13 + 70_001]
    total = boff[-1]
    gh = [synth.host_fill(synth.normal_stream(nd, (84, q), 1e-3), 0, total, "bf16")
          for q in range(nd)]
    out = torch.empty(total, dtype=torch.int16, device=DEV)
    ss.ddp_bucket_allreduce_avg([_dev16(h).view(torch.bfloat16) for h in gh], boff,
                                out.view(torch.bfloat16))
    torch.cuda.synchronize()
    assert_bits(out.cpu().numpy().view(np.uint16), oracle.bucket_allreduce_avg(gh, boff), "avg")
    S = boff[1]
    hs = [synth.host_fill(synth.normal_stream(nd, (85, q), 0.3), 0, S, "f16") for q in range(nd)]
    for plant in (False, True):
        if plant:
            hs[nd // 2][S - 77] = 0x7C00
        sc = ss.GradScaler(init_scale=64.0, device=DEV)
        sc.check([_dev16(h).view(torch.float16) for h in hs])
        want = osc.found_inf([(h, "f16") for h in hs], nd, 0, S, np.float32(1.0 / 64.0))
        torch.cuda.synchronize()
        assert bool(int(sc.found_inf.item())) == want == plant
