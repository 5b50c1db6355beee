"""Pins for the oracle's bf16 cast, reduce-scatter average, accumulation and
AdamW, each against something other than the oracle itself: IEEE facts and
torch's own bf16 conversion, the gradient-mean identity of "4.1 数据并行详解"
section 2 on a least-squares model, exact rational sums, torch.optim.AdamW in
float64, and closed forms of the update."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle.numerics import AdamWConfig

# ------------------------------------------------------------------ bf16


def _f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("bits,want", [
    (0x3F800000, 0x3F80),   # 1.0
    (0x3F808000, 0x3F80),   # 1 + 2^-8: halfway, ties to even (down)
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: halfway, ties to even (up)
    (0x3F808001, 0x3F81),   # just above halfway
    (0x3F807FFF, 0x3F80),   # just below halfway
    (0xBF808001, 0xBF81),   # sign is kept
    (0x7F7F7FFF, 0x7F7F),   # largest finite bf16, below the overflow point
    (0x7F7F8000, 0x7F80),   # max + ulp/2 overflows to +inf (ties to even)
    (0x7F800000, 0x7F80),   # +inf
    (0xFF800000, 0xFF80),   # -inf
    (0x00000000, 0x0000),
    (0x80000000, 0x8000),   # -0 stays -0
    (0x00008000, 0x0000),   # subnormal halfway to 0x0001, ties to even
    (0x00018000, 0x0002),   # subnormal halfway, ties up to even
    (0x007FFFFF, 0x0080),   # largest subnormal rounds up to the smallest normal
])
def test_f32_to_bf16_ieee_cases(bits, want):
    got = oracle.f32_to_bf16(_f32([bits]))[0]
    assert int(got) == want


def test_f32_to_bf16_nan_stays_nan():
    got = oracle.f32_to_bf16(_f32([0x7FC00000, 0xFF800001]))
    for g in got:
        assert (int(g) & 0x7F80) == 0x7F80 and (int(g) & 0x7F) != 0


def _torch_bf16_bits(x):
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_f32_to_bf16_matches_torch_on_all_exponents_and_rounding_bits():
    # every upper half (sign, exponent, 7 mantissa bits) with the lower halves
    # that decide the rounding, plus random lower halves
    upper = np.arange(1 << 16, dtype=np.uint32)
    lowers = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF],
                      dtype=np.uint32)
    rng = np.random.default_rng(0)
    lowers = np.concatenate([lowers, rng.integers(0, 1 << 16, 24).astype(np.uint32)])
    bits = ((upper[:, None] << 16) | lowers[None, :]).reshape(-1)
    x = bits.view(np.float32)
    finite = np.isfinite(x)
    ours = oracle.f32_to_bf16(x[finite])
    ref = _torch_bf16_bits(np.ascontiguousarray(x[finite]))
    assert np.array_equal(ours, ref)


def test_bf16_round_trip_is_exact():
    u = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = oracle.bf16_to_f32(u)
    keep = np.isfinite(x)
    assert np.array_equal(oracle.f32_to_bf16(x[keep]), u[keep])
    # the upcast is the exact value: matches torch's widening
    ref = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(x[keep], ref[keep])


def test_f32_to_bf16_is_nearest():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32)
    b = oracle.f32_to_bf16(x)
    y = oracle.bf16_to_f32(b).astype(np.float64)
    # neighbours one bf16 step up and down are never closer
    up = oracle.bf16_to_f32((b.astype(np.int32) + 1).astype(np.uint16)).astype(np.float64)
    dn = oracle.bf16_to_f32((b.astype(np.int32) - 1).astype(np.uint16)).astype(np.float64)
    err = np.abs(y - x)
    ok = np.isfinite(up) & np.isfinite(dn) & (b & 0x7FFF != 0)
    assert np.all(err[ok] <= np.abs(up - x)[ok])
    assert np.all(err[ok] <= np.abs(dn - x)[ok])


# -------------------------------------------------- gradient-mean identity

def _lsq_problem(B, d, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, d))
    y = rng.standard_normal(B)
    theta = rng.standard_normal(d)
    return X, y, theta


def _mean_grad(X, y, theta):
    # loss (1/b) sum_i 1/2 (x_i . theta - y_i)^2  ->  grad (1/b) X^T (X theta - y)
    return X.T @ (X @ theta - y) / X.shape[0]


@pytest.mark.parametrize("nd", [2, 4, 8])
def test_rs_avg_gives_global_batch_gradient(nd):
    X, y, theta = _lsq_problem(64, 24, nd)
    g = _mean_grad(X, y, theta)
    parts = np.split(np.arange(64), nd)
    local = [_mean_grad(X[p], y[p], theta) for p in parts]     # each rank's local-mean grad
    S = 24 // nd
    got = np.concatenate([oracle.rs_avg(local, r, S) for r in range(nd)])
    assert np.allclose(got, g, rtol=0, atol=1e-12)
    # negative control 1: summing instead of averaging is N times the gradient
    summed = np.sum(local, axis=0)
    assert np.allclose(summed, nd * g, atol=1e-12) and not np.allclose(summed, g, atol=1e-6)


def test_rs_avg_identity_breaks_with_unequal_local_batches():
    X, y, theta = _lsq_problem(64, 8, 5)
    g = _mean_grad(X, y, theta)
    parts = [np.arange(0, 8), np.arange(8, 64)]   # 8 and 56 samples
    local = [_mean_grad(X[p], y[p], theta) for p in parts]
    got = oracle.rs_avg(local, 0, 8)
    assert not np.allclose(got, g, atol=1e-6)


def test_accumulation_with_loss_over_m_gives_local_gradient():
    # a rank's local batch of 32 split into M = 4 micro-batches of 8, each
    # micro-batch loss divided by M
    X, y, theta = _lsq_problem(32, 6, 9)
    g_local = _mean_grad(X, y, theta)
    micro = [_mean_grad(X[j * 8:(j + 1) * 8], y[j * 8:(j + 1) * 8], theta) for j in range(4)]
    acc = oracle.grad_accumulate(micro, 1.0 / 4)
    assert np.allclose(acc, g_local, rtol=0, atol=1e-12)


def _nearest_f32(q: Fraction):
    """Correctly rounded fp32 of a rational (test helper, brute neighbour search)."""
    c = np.float32(float(q))
    best = c
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        if abs(Fraction(float(cand)) - q) < abs(Fraction(float(best)) - q):
            best = cand
        elif abs(Fraction(float(cand)) - q) == abs(Fraction(float(best)) - q):
            if int(np.array(cand, np.float32).view(np.uint32)) % 2 == 0:
                best = cand
    return best


@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 7, 8])
def test_rs_avg_exact_rational_mean(nd):
    # bf16 inputs with small integer mantissas: the fp32 sum is exact, so the
    # result must be the correctly rounded exact mean
    rng = np.random.default_rng(nd)
    S = 50
    ints = rng.integers(-255, 256, size=(nd, S * nd))
    scale = rng.integers(-12, 4, size=(nd, S * nd))
    vals = (ints * np.exp2(scale)).astype(np.float32)
    contribs = [oracle.f32_to_bf16(v) for v in vals]
    for r in range(nd):
        got = oracle.rs_avg(contribs, r, S)
        for i in range(S):
            q = sum(Fraction(float(vals[k, r * S + i])) for k in range(nd)) / nd
            assert got[i] == _nearest_f32(q), (r, i)


def test_rs_avg_sums_in_rank_order():
    # 1 + 2^24 rounds back to 2^24 in fp32, so the rank order decides the
    # result; the reading fixes order 0..N_d-1
    c = [np.array([1.0], np.float32), np.array([2.0 ** 24], np.float32),
         np.array([-(2.0 ** 24)], np.float32)]
    assert oracle.rs_avg(c, 0, 1)[0] == np.float32(0.0)
    assert oracle.rs_avg(c[::-1], 0, 1)[0] == np.float32(1.0) / np.float32(3.0)


def test_accumulate_bf16_inputs_upcast_exactly():
    g = [np.array([0x3F80, 0xC000], np.uint16), np.array([0x3F00, 0x4040], np.uint16)]
    acc = oracle.grad_accumulate(g, np.float32(0.5))
    # (1.0 + 0.5) / 2, (-2 + 3) / 2
    assert acc.dtype == np.float32
    assert np.array_equal(acc, np.array([0.75, 0.5], np.float32))


# ----------------------------------------------------------------- AdamW

HP = AdamWConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _torch_adamw(p0, grads, hp):
    p = torch.nn.Parameter(torch.from_numpy(p0.astype(np.float64).copy()))
    opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                            weight_decay=hp.weight_decay, foreach=False)
    for g in grads:
        p.grad = torch.from_numpy(g.astype(np.float64).copy())
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


@pytest.mark.parametrize("hp", [HP, AdamWConfig(lr=3e-2, beta1=0.8, beta2=0.95, eps=1e-6,
                                                weight_decay=0.1)])
def test_adamw_matches_torch_adamw_in_float64(hp):
    rng = np.random.default_rng(3)
    n = 4096
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(10)]
    ref_p, ref_m, ref_v = _torch_adamw(p0, grads, hp)
    # the oracle in float64 follows the same math: agreement to rounding
    p, m, v = p0.astype(np.float64), np.zeros(n), np.zeros(n)
    for t, g in enumerate(grads, 1):
        p, m, v = oracle.adamw(p, m, v, g.astype(np.float64), hp, t)
    # (torch orders the same operations differently: lerp for m, a multiplied
    # decay; elements near zero see cancellation, hence the scale-based bound)
    for ours, ref in ((p, ref_p), (m, ref_m), (v, ref_v)):
        assert np.max(np.abs(ours - ref)) <= 1e-11 * np.max(np.abs(ref))
    # the fp32 oracle stays within fp32 rounding of the float64 result
    p, m, v = p0, np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t, g in enumerate(grads, 1):
        p, m, v = oracle.adamw(p, m, v, g, hp, t)
    assert p.dtype == np.float32
    for ours, ref in ((p, ref_p), (m, ref_m), (v, ref_v)):
        assert np.max(np.abs(ours - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_adamw_first_step_closed_form():
    # from m = v = 0, step 1: m_hat = g, v_hat = g^2, so
    # p1 = p0 (1 - lr wd) - lr g / (|g| + eps)
    rng = np.random.default_rng(4)
    hp = AdamWConfig(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-3, weight_decay=0.1)
    p0 = rng.standard_normal(1000)
    g = rng.standard_normal(1000) * 1e-2
    p, m, v = oracle.adamw(p0, np.zeros(1000), np.zeros(1000), g, hp, 1)
    want = p0 * (1 - hp.lr * hp.weight_decay) - hp.lr * g / (np.abs(g) + hp.eps)
    assert np.allclose(p, want, rtol=1e-13, atol=1e-15)
    assert np.allclose(m, (1 - hp.beta1) * g, rtol=1e-14, atol=0)
    assert np.allclose(v, (1 - hp.beta2) * g * g, rtol=1e-14, atol=0)


def test_adamw_constant_gradient_closed_form():
    # a constant gradient keeps m_hat = g and v_hat = g^2 at every step, so
    # p_T = p0 d^T - lr g/(|g|+eps) * sum_{k<T} d^k  with d = 1 - lr wd
    hp = AdamWConfig(lr=5e-3, beta1=0.85, beta2=0.99, eps=1e-2, weight_decay=0.05)
    g = np.array([3e-2, -1e-1, 2.0, -5e-4])
    p = np.array([0.5, -0.25, 1.0, 0.0])
    p0 = p.copy()
    m, v = np.zeros(4), np.zeros(4)
    T = 12
    for t in range(1, T + 1):
        p, m, v = oracle.adamw(p, m, v, g, hp, t)
    d = 1 - hp.lr * hp.weight_decay
    want = p0 * d ** T - hp.lr * g / (np.abs(g) + hp.eps) * sum(d ** k for k in range(T))
    assert np.allclose(p, want, rtol=1e-12, atol=1e-15)
    assert np.allclose(m, (1 - hp.beta1 ** T) * g, rtol=1e-12)
    assert np.allclose(v, (1 - hp.beta2 ** T) * g * g, rtol=1e-12)


def test_adamw_zero_gradient_is_pure_decay():
    p0 = np.array([0.02, -1.5, 3.0e-3, 0.0], np.float32)
    z = np.zeros(4, np.float32)
    p, m, v = oracle.adamw(p0, z, z, z, HP, 1)
    want = p0.astype(np.float64) * (1 - HP.lr * HP.weight_decay)
    assert np.all(np.abs(p - want) <= np.abs(want) * 2 ** -23)
    assert not m.any() and not v.any()


def test_adamw_without_moments_is_normalised_sign_step():
    # beta1 = beta2 = 0, wd = 0: p <- p - lr g / (|g| + eps)
    hp = AdamWConfig(lr=0.1, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.0)
    p0 = np.array([1.0, 2.0, -3.0])
    g = np.array([4.0, -0.5, 1e-3])
    for t in (1, 2, 7):
        p, _, _ = oracle.adamw(p0, np.zeros(3), np.zeros(3), g, hp, t)
        assert np.allclose(p, p0 - 0.1 * g / (np.abs(g) + 1e-8), rtol=1e-15)


def test_adamw_is_elementwise_so_shards_update_independently():
    # "Infra: Data Parallel", ZeRO-1: updating N_d shards separately equals
    # updating the whole vector
    rng = np.random.default_rng(6)
    n, nd = 96, 4
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = (rng.random(n) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    whole = oracle.adamw(p, m, v, g, HP, 3)
    S = n // nd
    parts = [oracle.adamw(p[r * S:(r + 1) * S], m[r * S:(r + 1) * S], v[r * S:(r + 1) * S],
                          g[r * S:(r + 1) * S], HP, 3) for r in range(nd)]
    for k in range(3):
        assert np.array_equal(np.concatenate([x[k] for x in parts]), whole[k])


def test_adamw_rejects_step_zero():
    with pytest.raises(ValueError):
        oracle.adamw_scalars(HP, 0)


def test_fsdp_shard_step_composes_reduce_update_cast():
    rng = np.random.default_rng(7)
    nd, S = 4, 64
    contribs = [oracle.f32_to_bf16((rng.standard_normal(nd * S) * 1e-3).astype(np.float32))
                for _ in range(nd)]
    for r in range(nd):
        p = (rng.standard_normal(S) * 0.02).astype(np.float32)
        z = np.zeros(S, np.float32)
        p1, m1, v1, out = oracle.fsdp_shard_step(contribs, r, S, p, z, z, HP, 1)
        g = oracle.rs_avg(contribs, r, S)
        p2, m2, v2 = oracle.adamw(p, z, z, g, HP, 1)
        assert np.array_equal(p1, p2) and np.array_equal(m1, m2) and np.array_equal(v1, v2)
        assert np.array_equal(out, oracle.f32_to_bf16(p2))
