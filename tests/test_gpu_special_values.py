"""Special values through the GPU path against the oracle: signed zeros,
bf16 subnormals (fp32 arithmetic keeps subnormals on both sides: no
flush-to-zero), the largest finite bf16 on every rank (the fp32 sum
overflows to inf), +inf and -inf at the same element on two ranks (their sum
is NaN), NaN gradients, and huge or subnormal master weights.  Every result
is compared bit for bit, except the payload of NaN results: IEEE leaves the
NaN an invalid operation produces to the platform (the GPU, x86 and Arm each
produce a different default NaN), so where the oracle has a NaN the GPU
must have a NaN, and everywhere else the bits must match."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = AdamWConfig()
HPC = ss.AdamW()


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    assert ss.device_status() == 0


@pytest.fixture(params=["auto", "register", "tma"])
def path(request):
    prev = ss.set_fused_path(request.param)
    yield request.param
    ss.set_fused_path(prev)


def _nan32(bits):
    b = np.asarray(bits).view(np.uint32)
    return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x007FFFFF) != 0)


def _nan16(bits):
    b = np.asarray(bits).view(np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def assert_same_up_to_nan_payload(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape
    isnan = _nan16 if got.dtype == np.uint16 else _nan32
    gn, wn = isnan(got), isnan(want)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    keep = ~wn
    assert got[keep].tobytes() == want[keep].tobytes(), f"{what}: not bit-exact"


BF16_SPECIALS = {"pzero": 0x0000, "nzero": 0x8000, "sub_min": 0x0001, "sub_max": 0x007F,
                 "nsub": 0x8005, "max": 0x7F7F, "nmax": 0xFF7F, "pinf": 0x7F80,
                 "ninf": 0xFF80, "nan": 0x7FC0, "nan_payload": 0x7F81, "min_normal": 0x0080}


def _special_grads(nd, S, seed):
    """Normal gradients with special values planted at fixed positions."""
    g = [synth.host_fill(synth.normal_stream(seed, (66, q), 1e-3), 0, S, "bf16")
         for q in range(nd)]
    pos = {}
    k = 7
    for name, bits in BF16_SPECIALS.items():
        pos[name] = k
        for q in range(nd):
            g[q][k] = bits                          # every rank: the same special
        k += 977
    # mixed cases: one rank only, and opposite infinities on two ranks
    pos["one_inf"] = k
    g[nd // 2][k] = 0x7F80
    k += 977
    pos["inf_minus_inf"] = k
    g[0][k] = 0x7F80
    g[nd - 1][k] = 0xFF80
    k += 977
    pos["one_nan"] = k
    g[nd - 1][k] = 0x7FC0
    k += 977
    pos["max_plus_tiny"] = k                        # overflow by accumulation only
    for q in range(nd):
        g[q][k] = 0x7F7F if q % 2 == 0 else 0x0001
    assert k < S
    return g, pos


def _special_master(S, seed):
    p = synth.host_fill(synth.normal_stream(seed, (67,), 0.02), 0, S, "f32")
    bits = p.view(np.uint32)
    for k, b in ((3, 0x00000000), (5, 0x80000000), (11, 0x00000001), (13, 0x807FFFFF),
                 (17, 0x7F7FFFFF), (19, 0xFF7FFFFF), (23, 0x7F800000), (29, 0x00800000)):
        bits[k] = b
    return p


def _dev16(h):
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(DEV).view(torch.bfloat16)


@pytest.mark.parametrize("nd,S", [(8, 70001), (8, 2048 * 152 + 13), (3, 40000), (1, 20000),
                                  (16, 30000)])
def test_fused_step_with_special_values(nd, S, path):
    g, _ = _special_grads(nd, S, nd)
    p0 = _special_master(S, nd)
    m0 = np.zeros(S, np.float32)
    v0 = np.zeros(S, np.float32)
    dp = torch.from_numpy(p0.copy()).to(DEV)
    dm = torch.zeros(S, device=DEV)
    dv = torch.zeros(S, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    p, m, v = p0, m0, v0
    for t in (1, 2):
        ss.fsdp_rs_avg_adamw_cast([_dev16(x) for x in g], dp, dm, dv, out, HPC, t)
        with np.errstate(all="ignore"):
            p, m, v, ob = oracle.fsdp_shard_step(g, 0, S, p, m, v, HP, t)
    torch.cuda.synchronize()
    assert_same_up_to_nan_payload(dp.cpu().numpy().view(np.uint32), p.view(np.uint32), "master")
    assert_same_up_to_nan_payload(dm.cpu().numpy().view(np.uint32), m.view(np.uint32), "m")
    assert_same_up_to_nan_payload(dv.cpu().numpy().view(np.uint32), v.view(np.uint32), "v")
    assert_same_up_to_nan_payload(out.view(torch.int16).cpu().numpy().view(np.uint16), ob,
                                  "bf16")


def test_special_values_take_the_expected_ieee_paths():
    """The planted cases behave as IEEE fp32 says, on the GPU: the sum of the
    largest bf16 over 8 ranks overflows to inf, +inf + -inf is NaN, a single
    inf or NaN makes the mean inf or NaN, subnormal gradients survive."""
    nd, S = 8, 70001
    g, pos = _special_grads(nd, S, 1)
    dp = torch.zeros(S, device=DEV)
    dm = torch.zeros(S, device=DEV)
    dv = torch.zeros(S, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([_dev16(x) for x in g], dp, dm, dv, out, HPC, 1)
    torch.cuda.synchronize()
    m = dm.cpu().numpy()
    # m = (1 - beta1) * mean after one step from zero
    assert np.isinf(m[pos["max"]]) and m[pos["max"]] > 0
    assert np.isinf(m[pos["one_inf"]])
    assert np.isnan(m[pos["inf_minus_inf"]]) and np.isnan(m[pos["nan"]])
    assert np.isnan(m[pos["one_nan"]])
    assert m[pos["sub_min"]] != 0 and abs(m[pos["sub_min"]]) < 1e-37     # no flush to zero
    assert m[pos["pzero"]] == 0 and m[pos["nzero"]] == 0
    assert np.isfinite(m[pos["min_normal"]])


@pytest.mark.parametrize("n", [70001, 13])
def test_accumulate_with_special_values(n, path):
    M = 3
    micro = []
    for j in range(M):
        h = synth.host_fill(synth.normal_stream(n, (68, j), 1e-3), 0, n, "bf16")
        for k, b in enumerate(BF16_SPECIALS.values()):
            if 2 * k + j < n:
                h[2 * k + j] = b
        micro.append(h)
    acc = torch.full((n,), 3.0, device=DEV)
    for j in range(M):
        ss.fsdp_grad_accumulate(_dev16(micro[j]), acc, float(np.float32(1 / 3)), j == 0)
    with np.errstate(all="ignore"):
        want = oracle.grad_accumulate(micro, np.float32(1 / 3))
    torch.cuda.synchronize()
    assert_same_up_to_nan_payload(acc.cpu().numpy().view(np.uint32), want.view(np.uint32),
                                  "acc")


@pytest.mark.parametrize("nd", [2, 8, 5])
def test_bucket_allreduce_with_special_values(nd, path):
    S = 70001
    g, _ = _special_grads(nd, S, 20 + nd)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    ss.ddp_bucket_allreduce_avg([_dev16(x) for x in g], [0, 4096, S], out)
    with np.errstate(all="ignore"):
        want = oracle.bucket_allreduce_avg(g, [0, 4096, S])
    torch.cuda.synchronize()
    assert_same_up_to_nan_payload(out.view(torch.int16).cpu().numpy().view(np.uint16), want,
                                  "avg")
