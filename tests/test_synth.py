"""The seeded input generator (not the method): its fp16 rounding against
numpy's, and that a stream regenerates the same values by range and by
index."""
import numpy as np

import synth


def test_f16_rounding_matches_numpy():
    lib = synth._host_lib()
    rng = np.random.default_rng(0)
    bits = np.concatenate([
        rng.integers(0, 2 ** 32, 100_000, dtype=np.uint64).astype(np.uint32),
        np.arange(0x33000000, 0x38900000, 4099, dtype=np.uint32),    # subnormal range
        np.arange(0x477F0000, 0x47810000, 7, dtype=np.uint32),       # around 65504 / 65520
        np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x33000000, 0x33000001], np.uint32)])
    x = bits.view(np.float32)
    ours = np.array([lib.synth_f32bits_to_f16(int(b)) for b in bits], dtype=np.uint16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    keep = ~np.isnan(x)
    assert np.array_equal(ours[keep], ref[keep])
    assert np.all((ours[~keep] & 0x7C00) == 0x7C00) and np.all((ours[~keep] & 0x3FF) != 0)


def test_range_and_index_agree():
    for dtype in ("bf16", "f16", "f32"):
        st = synth.normal_stream(3, (1, 2, 3), 65.0, outlier_p=0.05)
        a = synth.host_fill(st, 1000, 5000, dtype)
        idx = np.arange(1000, 6000)[::7]
        assert np.array_equal(synth.host_gather(st, idx, dtype), a[::7])
