"""Pins for the oracle's sharded gradient scaler: torch's own amp routines
(torch._amp_update_scale_ for the scale schedule,
torch._amp_foreach_non_finite_check_and_unscale_ for the check and the
unscale), torch's fp16 widening, and the equivalence the page claims: with a
power-of-two scale and no overflow, the scaled step is the unscaled step."""
import numpy as np
import pytest
import torch

import oracle
from oracle import scaler
from oracle.numerics import AdamWConfig

HP = AdamWConfig()


def test_f16_widening_matches_torch_on_every_pattern():
    u = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = scaler.f16_to_f32(u)
    ref = torch.from_numpy(u.view(np.int16)).view(torch.float16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("growth,backoff,interval", [(2.0, 0.5, 3), (2.0, 0.5, 1), (1.5, 0.25, 5)])
def test_scaler_update_matches_torch(growth, backoff, interval):
    rng = np.random.default_rng(interval)
    for start in (65536.0, 1.0, 3.0e38, 1e-30):
        s_ref = torch.tensor([start], dtype=torch.float32)
        g_ref = torch.tensor([0], dtype=torch.int32)
        s, tr = np.float32(start), 0
        for _ in range(60):
            found = bool(rng.random() < 0.2)
            torch._amp_update_scale_(s_ref, g_ref, torch.tensor([1.0 if found else 0.0]),
                                     growth, backoff, interval)
            s, tr = scaler.scaler_update(s, tr, found, growth, backoff, interval)
            assert np.float32(s).view(np.uint32) == s_ref.numpy().view(np.uint32)[0]
            assert tr == int(g_ref.item())


def _f16(x):
    return np.asarray(x, np.float16).view(np.uint16)


@pytest.mark.parametrize("nd,F", [(4, 4), (8, 8), (8, 2)])
def test_check_and_unscale_match_torch(nd, F):
    rng = np.random.default_rng(nd + F)
    S = 64
    vals = [(rng.standard_normal(F * S) * 1000).astype(np.float16) for _ in range(nd)]
    vals[1][5] = np.float16(np.inf)          # one rank overflowed, in shard 0
    contribs = [(_f16(v), "f16") for v in vals]
    inv = np.float32(1.0 / 1024)
    for f in range(F):
        ours = scaler.unscaled_mean(contribs, F, f, S, inv)
        mean = torch.from_numpy(oracle.hybrid_rs_avg([scaler.f16_to_f32(c[0]) for c in contribs],
                                                     F, f, S).copy())
        found = torch.tensor([0.0])
        torch._amp_foreach_non_finite_check_and_unscale_([mean], found, torch.tensor([inv]))
        assert np.array_equal(ours, mean.numpy(), equal_nan=True)
        assert scaler.found_inf(contribs, F, f, S, inv) == bool(found.item())
    assert scaler.found_inf(contribs, F, 0, S, inv)
    if F > 1:
        assert not scaler.found_inf(contribs, F, 1, S, inv)


@pytest.mark.parametrize("nd,F", [(4, 4), (8, 4)])
def test_power_of_two_scaling_is_exact(nd, F):
    # gradients whose scaled values stay normal fp16 numbers: the scaled step
    # with 1/s equals the unscaled step bit for bit
    rng = np.random.default_rng(3)
    S = 256
    s = np.float32(2.0 ** 7)
    g = [rng.integers(-2000, 2000, size=F * S).astype(np.float16) * np.float16(2.0 ** -12)
         for _ in range(nd)]
    scaled = [(_f16(x.astype(np.float32) * s), "f16") for x in g]
    plain = [(_f16(x), "f16") for x in g]
    for f in range(F):
        p0 = (rng.standard_normal(S) * 0.02).astype(np.float32)
        z = np.zeros(S, np.float32)
        a = scaler.scaled_shard_step(scaled, F, f, S, p0, z, z, None, HP, 1, 1 / s, False)
        b = scaler.scaled_shard_step(plain, F, f, S, p0, z, z, None, HP, 1, 1.0, False)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_skip_leaves_the_state_untouched():
    p = np.array([1.0, 2.0], np.float32)
    m = np.array([0.5, 0.25], np.float32)
    v = np.array([0.1, 0.2], np.float32)
    prev = np.array([7, 9], np.uint16)
    contribs = [(_f16([np.inf, 1.0]), "f16"), (_f16([1.0, 1.0]), "f16")]
    assert scaler.found_inf(contribs, 2, 0, 2, 1.0)
    out = scaler.scaled_shard_step(contribs, 2, 0, 2, p, m, v, prev, HP, 3, 1.0, True)
    for x, y in zip(out, (p, m, v, prev)):
        assert x is y


def test_nan_gradient_is_found():
    contribs = [(_f16([np.nan, 1.0]), "f16"), (_f16([1.0, 1.0]), "f16")]
    assert scaler.found_inf(contribs, 2, 0, 2, 0.5)
    contribs = [(_f16([-np.inf, 1.0]), "f16"), (_f16([np.inf, 1.0]), "f16")]
    assert scaler.found_inf(contribs, 2, 0, 2, 0.5)   # inf - inf = NaN
