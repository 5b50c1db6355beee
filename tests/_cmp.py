"""Comparison helpers for the parity tests (the acceptance bar of the path):
  * indexing, padding, copies: bit-exact;
  * fp32 master weights and moments: max relative error <= 1e-6, relative to
    max(|oracle|, 1e-30), pairs that are exactly equal skipped;
  * bf16 outputs: within 1 ulp (adjacent bit patterns of the same sign)."""
import numpy as np

F32_RTOL = 1e-6
BF16_ULP = 1


def f32_max_rel(got, want):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape
    diff = got != want
    if not diff.any():
        return 0.0
    g = got[diff].astype(np.float64)
    w = want[diff].astype(np.float64)
    return float(np.max(np.abs(g - w) / np.maximum(np.abs(w), 1e-30)))


def assert_f32(got, want, what=""):
    err = f32_max_rel(got, want)
    assert err <= F32_RTOL, f"{what}: max rel err {err:.3e} > {F32_RTOL}"


def bf16_max_ulp(got, want):
    g = np.asarray(got, np.uint16).astype(np.int64)
    w = np.asarray(want, np.uint16).astype(np.int64)
    assert g.shape == w.shape
    # map sign-magnitude bit patterns onto an ordered integer line
    def key(x):
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return int(np.max(np.abs(key(g) - key(w)))) if g.size else 0


def assert_bf16(got, want, what=""):
    u = bf16_max_ulp(got, want)
    assert u <= BF16_ULP, f"{what}: bf16 differs by {u} ulp"


def assert_bits(got, want, what=""):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, what
    assert got.tobytes() == want.tobytes(), f"{what}: not bit-exact"
