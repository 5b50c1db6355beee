"""GPU parity: every entry point of the C ABI against the CPU oracle on the
same seeded inputs, element by element, at sizes that span several tiles,
ragged tails, misaligned pointers and the degenerate cases (N_d = 1, one
element, empty pieces).  Bar: bit-exact indexing and copies; fp32 state
within 1e-6 relative; bf16 within 1 ulp.  The fused step is also required to
be bit-exact, which its fixed operation order makes possible."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from tests._cmp import assert_bf16, assert_bits, assert_f32

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
HP = AdamWConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HPC = ss.AdamW(lr=HP.lr, beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps, weight_decay=HP.weight_decay)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    # no TMA-staged wait ran out during the module
    assert ss.device_status() == 0


@pytest.fixture(params=["auto", "register", "tma"])
def path(request):
    """Run a test under each kernel choice: auto (TMA-staged where it measured
    faster), register-staged only, and TMA-staged wherever the arguments
    allow (also at N_d = 1, 2 and on small buckets)."""
    prev = ss.set_fused_path(request.param)
    yield request.param
    ss.set_fused_path(prev)


def dev_bf16(u16, shift=0):
    """numpy bf16 bits -> CUDA bf16 tensor starting `shift` elements into its
    allocation (shift > 0 gives a misaligned pointer)."""
    buf = torch.empty(u16.size + shift + 8, dtype=torch.bfloat16, device=DEV)
    t = buf[shift:shift + u16.size]
    t.copy_(torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16))
    return t


def dev_f32(x, shift=0):
    buf = torch.empty(x.size + shift + 8, dtype=torch.float32, device=DEV)
    t = buf[shift:shift + x.size]
    t.copy_(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)))
    return t


def host_bf16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t):
    return t.contiguous().cpu().numpy()


def _grads(seed, nd, P, dtype, step):
    out = []
    for q in range(nd):
        st = synth.normal_stream(seed, (99, 1, step, q), 1e-3)
        out.append(synth.host_fill(st, 0, P, dtype))
    return out


# ------------------------------------------------------------ fused step

@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("S", [1, 13, 4099, 6151])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
@pytest.mark.parametrize("shift", [0, 1])
def test_fused_step_matches_oracle(nd, S, gdt, shift, path):
    seed = nd * 1000 + S + (7 if gdt == "f32" else 0)
    r = (S + 2 * nd) % nd
    P = nd * S
    p = synth.host_fill(synth.normal_stream(seed, (99, 2), 0.02), 0, S, "f32")
    m = np.zeros(S, np.float32)
    v = np.zeros(S, np.float32)
    dp, dm, dv = dev_f32(p, shift), dev_f32(m, shift), dev_f32(v, shift)
    out = torch.empty(S + 1, dtype=torch.bfloat16, device=DEV)[shift:shift + S]
    for t in (1, 2, 3):
        contribs = _grads(seed, nd, P, gdt, t)
        mk = dev_bf16 if gdt == "bf16" else dev_f32
        slices = [mk(c[r * S:(r + 1) * S], shift if q % 2 else 0) for q, c in enumerate(contribs)]
        ss.fsdp_rs_avg_adamw_cast(slices, dp, dm, dv, out, HPC, t)
        p, m, v, ob = oracle.fsdp_shard_step(contribs, r, S, p, m, v, HP, t)
        torch.cuda.synchronize()
        for name, got, want in (("master", host_f32(dp), p), ("m", host_f32(dm), m),
                                ("v", host_f32(dv), v)):
            assert_f32(got, want, f"{name} step {t}")
            assert_bits(got, want, f"{name} step {t}")
        assert_bf16(host_bf16(out), ob, f"bf16 step {t}")
        assert_bits(host_bf16(out), ob, f"bf16 step {t}")


@pytest.mark.parametrize("nd,gdt,S", [(8, "bf16", 152 * 256 * 8 * 2 + 5),
                                      (4, "f32", 152 * 256 * 8 + 8 * 37 + 3),
                                      (8, "bf16", 1 << 20),
                                      (8, "bf16", 2048 * 152 * 3 + 2048 + 8 * 5 + 7),
                                      (16, "bf16", 2048 * 200 + 1000),
                                      (8, "f32", 2048 * 160 + 16),
                                      (21, "bf16", 70001), (22, "bf16", 70001),
                                      (23, "bf16", 70001), (10, "f32", 70001),
                                      (11, "f32", 70001), (12, "f32", 70001)])
def test_fused_step_multi_tile(nd, gdt, S, path):
    seed = 5 + S
    P = nd * S
    r = 1 % nd
    contribs = _grads(seed, nd, P, gdt, 1)
    p = synth.host_fill(synth.normal_stream(seed, (99, 2), 0.02), 0, S, "f32")
    m = (synth.host_fill(synth.normal_stream(seed, (99, 3), 1e-4), 0, S, "f32"))
    v = np.abs(synth.host_fill(synth.normal_stream(seed, (99, 4), 1e-7), 0, S, "f32"))
    dp, dm, dv = dev_f32(p), dev_f32(m), dev_f32(v)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    mk = dev_bf16 if gdt == "bf16" else dev_f32
    slices = [mk(c[r * S:(r + 1) * S]) for c in contribs]
    ss.fsdp_rs_avg_adamw_cast(slices, dp, dm, dv, out, HPC, 7)
    p, m, v, ob = oracle.fsdp_shard_step(contribs, r, S, p, m, v, HP, 7)
    torch.cuda.synchronize()
    assert_bits(host_f32(dp), p, "master")
    assert_bits(host_f32(dm), m, "m")
    assert_bits(host_f32(dv), v, "v")
    assert_bits(host_bf16(out), ob, "bf16")


@pytest.mark.parametrize("nd,F", [(2, 1), (4, 2), (6, 3), (8, 1), (8, 2), (8, 4), (8, 8),
                                  (16, 8), (16, 4)])
@pytest.mark.parametrize("gdt,S,shift", [("bf16", 13, 0), ("bf16", 70001, 0), ("bf16", 4099, 1),
                                         ("f32", 6151, 0), ("f32", 4099, 1)])
def test_hybrid_step_matches_oracle(nd, F, gdt, S, shift, path):
    seed = 31 * nd + F + S
    f = (S + F - 1) % F
    p = synth.host_fill(synth.normal_stream(seed, (97, 2), 0.02), 0, S, "f32")
    m = np.zeros(S, np.float32)
    v = np.zeros(S, np.float32)
    dp, dm, dv = dev_f32(p, shift), dev_f32(m, shift), dev_f32(v, shift)
    out = torch.empty(S + 1, dtype=torch.bfloat16, device=DEV)[shift:shift + S]
    for t in (1, 2):
        contribs = _grads(seed, nd, F * S, gdt, t)
        mk = dev_bf16 if gdt == "bf16" else dev_f32
        slices = [mk(c[f * S:(f + 1) * S], shift if k % 2 else 0) for k, c in enumerate(contribs)]
        ss.fsdp_hybrid_rs_avg_adamw_cast(slices, F, dp, dm, dv, out, HPC, t)
        p, m, v, ob = oracle.hybrid_shard_step(contribs, F, f, S, p, m, v, HP, t)
        torch.cuda.synchronize()
        for name, got, want in (("master", host_f32(dp), p), ("m", host_f32(dm), m),
                                ("v", host_f32(dv), v)):
            assert_f32(got, want, f"{name} step {t}")
            assert_bits(got, want, f"{name} step {t}")
        assert_bits(host_bf16(out), ob, f"bf16 step {t}")


@pytest.mark.parametrize("nd,F,gdt", [(6, 6, "bf16"), (7, 7, "bf16"), (12, 12, "bf16"),
                                      (13, 13, "bf16"), (24, 24, "bf16"), (64, 64, "bf16"),
                                      (6, 6, "f32"), (13, 13, "f32"), (24, 8, "bf16"),
                                      (12, 4, "bf16"), (12, 3, "f32"), (64, 16, "bf16"),
                                      (5, 1, "bf16"), (7, 7, "f32"), (5, 5, "f32")])
def test_fused_step_any_nd_matches_oracle(nd, F, gdt, path):
    """N_d without a compiled register kernel (24, 64, and fp32 slices
    above 4 but 6 and 8): the slices are loaded in batches (8 16-bit or 4
    fp32 slices), the last batch partial, and with hybrid sharding the
    groups of F cross the batch boundaries; with 16-bit slices at 6, 7, 12
    and 13, the compiled and up-to-8 forms."""
    S = 6151
    seed = 77 * nd + F
    f = (S + F - 1) % F
    p = synth.host_fill(synth.normal_stream(seed, (96, 2), 0.02), 0, S, "f32")
    m = synth.host_fill(synth.normal_stream(seed, (96, 3), 1e-4), 0, S, "f32")
    v = np.abs(synth.host_fill(synth.normal_stream(seed, (96, 4), 1e-7), 0, S, "f32"))
    dp, dm, dv = dev_f32(p), dev_f32(m), dev_f32(v)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    contribs = _grads(seed, nd, F * S, gdt, 1)
    mk = dev_bf16 if gdt == "bf16" else dev_f32
    slices = [mk(c[f * S:(f + 1) * S]) for c in contribs]
    if F == nd:
        ss.fsdp_rs_avg_adamw_cast(slices, dp, dm, dv, out, HPC, 3)
        p, m, v, ob = oracle.fsdp_shard_step(contribs, f, S, p, m, v, HP, 3)
    else:
        ss.fsdp_hybrid_rs_avg_adamw_cast(slices, F, dp, dm, dv, out, HPC, 3)
        p, m, v, ob = oracle.hybrid_shard_step(contribs, F, f, S, p, m, v, HP, 3)
    torch.cuda.synchronize()
    assert_bits(host_f32(dp), p, "master")
    assert_bits(host_f32(dm), m, "m")
    assert_bits(host_f32(dv), v, "v")
    assert_bits(host_bf16(out), ob, "bf16")


@pytest.mark.parametrize("nd,F", [(9, 9), (10, 10), (11, 11), (13, 13), (14, 14), (15, 15),
                                  (10, 5), (14, 7), (15, 3), (9, 3)])
@pytest.mark.parametrize("S,shift", [(4099, 0), (152 * 512 + 13, 1)])
def test_fused_step_compiled_9_to_15_matches_oracle(nd, F, S, shift, path):
    """16-bit slices at N_d = 9..11 and 13..15: the register kernel compiled
    for each count, all N_d loads in flight; plain rank order and grouped
    (hybrid) order; ragged shards over many blocks, misaligned slices."""
    seed = 131 * nd + F + S
    f = (S + F - 1) % F
    p = synth.host_fill(synth.normal_stream(seed, (95, 2), 0.02), 0, S, "f32")
    m = synth.host_fill(synth.normal_stream(seed, (95, 3), 1e-4), 0, S, "f32")
    v = np.abs(synth.host_fill(synth.normal_stream(seed, (95, 4), 1e-7), 0, S, "f32"))
    dp, dm, dv = dev_f32(p, shift), dev_f32(m, shift), dev_f32(v, shift)
    out = torch.empty(S + 1, dtype=torch.bfloat16, device=DEV)[shift:shift + S]
    contribs = _grads(seed, nd, F * S, "bf16", 1)
    slices = [dev_bf16(c[f * S:(f + 1) * S], shift if q % 3 == 1 else 0)
              for q, c in enumerate(contribs)]
    if F == nd:
        ss.fsdp_rs_avg_adamw_cast(slices, dp, dm, dv, out, HPC, 2)
        p, m, v, ob = oracle.fsdp_shard_step(contribs, f, S, p, m, v, HP, 2)
    else:
        ss.fsdp_hybrid_rs_avg_adamw_cast(slices, F, dp, dm, dv, out, HPC, 2)
        p, m, v, ob = oracle.hybrid_shard_step(contribs, F, f, S, p, m, v, HP, 2)
    torch.cuda.synchronize()
    assert_bits(host_f32(dp), p, "master")
    assert_bits(host_f32(dm), m, "m")
    assert_bits(host_f32(dv), v, "v")
    assert_bits(host_bf16(out), ob, "bf16")
    if path != "tma" and shift == 0:
        assert ss.last_kernel().startswith(f"rs_adamw_cast_vec4<{nd}, bf16>"), ss.last_kernel()


def test_hybrid_group_order_is_not_the_flat_order(path):
    # the nested sum keeps what the flat rank-order sum rounds away
    S, nd, F = 4096, 4, 2
    vals = [2.0 ** 24, 1.0, 1.0, 1.0]
    slices = [torch.full((S,), x, dtype=torch.float32, device=DEV) for x in vals]
    res = {}
    for name, call in (("hybrid", lambda *a: ss.fsdp_hybrid_rs_avg_adamw_cast(slices, F, *a)),
                       ("flat", lambda *a: ss.fsdp_rs_avg_adamw_cast(slices, *a))):
        dp = torch.zeros(S, device=DEV)
        dm = torch.zeros(S, device=DEV)
        dv = torch.zeros(S, device=DEV)
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        # beta1 = 0, lr = 0: m = (1 - 0) * g holds the reduced gradient exactly
        call(dp, dm, dv, out, ss.AdamW(lr=0.0, beta1=0.0, beta2=0.5, eps=1.0, weight_decay=0.0), 1)
        res[name] = host_f32(dm)
    torch.cuda.synchronize()
    assert np.all(res["hybrid"] == np.float32(4194304.5))
    assert np.all(res["flat"] == np.float32(4194304.0))


def test_fused_step_padding_stays_zero(path):
    # zero gradients and zero master (the padding of a FlatParameter) stay zero
    S, nd = 10000, 4
    z = torch.zeros(S, dtype=torch.bfloat16, device=DEV)
    dp = torch.zeros(S, device=DEV)
    dm = torch.zeros(S, device=DEV)
    dv = torch.zeros(S, device=DEV)
    out = torch.full((S,), 1.0, dtype=torch.bfloat16, device=DEV)
    for t in (1, 2):
        ss.fsdp_rs_avg_adamw_cast([z] * nd, dp, dm, dv, out, HPC, t)
    torch.cuda.synchronize()
    assert not dp.any() and not dm.any() and not dv.any() and not out.float().any()


def test_fused_step_output_may_be_the_slot_of_the_full_buffer(path):
    nd, S, r = 4, 40960, 2
    contribs = _grads(11, nd, nd * S, "bf16", 1)
    p = synth.host_fill(synth.normal_stream(11, (99, 2), 0.02), 0, S, "f32")
    dp, dm, dv = dev_f32(p), torch.zeros(S, device=DEV), torch.zeros(S, device=DEV)
    full = torch.zeros(nd * S, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([dev_bf16(c[r * S:(r + 1) * S]) for c in contribs], dp, dm, dv,
                              full[r * S:(r + 1) * S], HPC, 1)
    _, _, _, ob = oracle.fsdp_shard_step(contribs, r, S, p, np.zeros(S, np.float32),
                                         np.zeros(S, np.float32), HP, 1)
    torch.cuda.synchronize()
    h = host_bf16(full)
    assert_bits(h[r * S:(r + 1) * S], ob, "slot")
    assert not h[:r * S].any() and not h[(r + 1) * S:].any()


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("nd", [1, 3, 8])
def test_flat_pack_matches_oracle(dtype, nd, path):
    rng = np.random.default_rng(nd)
    numels = [int(x) for x in rng.integers(0, 5000, size=150)] + [1 << 20, 3, 0, 77777]
    shifts = [int(s) for s in rng.integers(0, 4, size=len(numels))]
    host, dev = [], []
    for k, (n, sh) in enumerate(zip(numels, shifts)):
        st = synth.normal_stream(nd, (98, k), 0.02)
        h = synth.host_fill(st, 0, n, dtype)
        host.append(h)
        dev.append(dev_bf16(h, sh) if dtype == "bf16" else dev_f32(h, sh))
    flat = ss.fsdp_flat_pack(dev, nd)
    want, lay = oracle.flat_pack(host, nd)
    torch.cuda.synchronize()
    got = host_bf16(flat) if dtype == "bf16" else host_f32(flat)
    assert got.size == lay.padded
    assert_bits(got.view(np.uint8), want.view(np.uint8), "flat")
    # views of the packed buffer: whole tensors, and every rank's pieces
    shapes = [(n,) for n in numels]
    for t, v in enumerate(ss.fsdp_views(flat, shapes, nd)):
        assert v.numel() == numels[t]
    for r in range(nd):
        shard = flat[r * lay.shard:(r + 1) * lay.shard]
        pieces = ss.fsdp_views(shard, shapes, nd, r)
        want_pieces = oracle.sharded_views(oracle.shard_of(want, lay, r), lay, r)
        for a, b in zip(pieces, want_pieces):
            ha = host_bf16(a) if dtype == "bf16" else host_f32(a)
            assert_bits(ha.view(np.uint8), b.view(np.uint8), "piece")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flat_pack_every_source_and_destination_offset(dtype, path):
    """A tensor packed behind a filler of o elements (destination offset o)
    from a source that starts s elements into its allocation, for every o
    and s below 16 bytes and lengths around the 16-byte vector and the
    16 KB chunk: every pairing of source and destination alignment,
    including the ones the realigning copy takes."""
    es = 2 if dtype == "bf16" else 4
    per16 = 16 // es
    mk = dev_bf16 if dtype == "bf16" else dev_f32
    for n in (1, per16 - 1, per16 + 1, 8192 // es * 2 + 3, 70001):
        body = synth.host_fill(synth.normal_stream(n, (95, 1), 0.02), 0, n, dtype)
        for o in range(per16):
            filler = synth.host_fill(synth.normal_stream(n, (95, 2, o), 0.02), 0, o, dtype)
            for sh in range(per16):
                host = [filler, body] if o else [body]
                dev = [mk(filler)] if o else []
                dev.append(mk(body, sh))
                flat = ss.fsdp_flat_pack(dev, 1)
                want, _ = oracle.flat_pack(host, 1)
                torch.cuda.synchronize()
                got = host_bf16(flat) if dtype == "bf16" else host_f32(flat)
                assert_bits(got, want, f"n={n} o={o} s={sh}")


def test_flat_pack_misaligned_destination_segments(path):
    # element offsets that are odd make source and destination incongruent
    numels = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987, 1597, 2584]
    host = [synth.host_fill(synth.normal_stream(1, (97, k), 1.0), 0, n, "bf16")
            for k, n in enumerate(numels)]
    dev = [dev_bf16(h, k % 8) for k, h in enumerate(host)]
    flat = ss.fsdp_flat_pack(dev, 7)
    want, _ = oracle.flat_pack(host, 7)
    torch.cuda.synchronize()
    assert_bits(host_bf16(flat), want, "flat")


@pytest.mark.parametrize("dependent", [True, False])
def test_copy_launches_of_one_call_keep_stream_order(dependent):
    """A pack of 203 bf16 tensors at mixed offsets (congruent, realigned and
    byte-wise ranges, more than 64 of each kind, so every copy kernel runs
    several times and the later launches are programmatic dependents of the
    earlier ones) between a torch producer that writes its sources and a
    torch consumer that reads the packed buffer right after it, on the same
    stream; then the all-gather of shards at odd slot offsets the same way."""
    nd = 8
    rng = np.random.default_rng(5)
    numels = [1 << 20] + [int(x) for x in rng.integers(1, 20000, size=200)] + [3 << 20, 5]
    shifts = [int(s) for s in rng.integers(0, 8, size=len(numels))]
    host = [synth.host_fill(synth.normal_stream(6, (94, k), 0.02), 0, n, "bf16")
            for k, n in enumerate(numels)]
    staged = [dev_bf16(h, sh) for h, sh in zip(host, shifts)]
    srcs = [dev_bf16(np.zeros(n, np.uint16), sh) for n, sh in zip(numels, shifts)]
    want, lay = oracle.flat_pack(host, nd)
    S = lay.shard
    shards_h = [want[r * S:(r + 1) * S] for r in range(nd)]
    staged_sh = [dev_bf16(h, r % 8) for r, h in enumerate(shards_h)]
    shards = [dev_bf16(np.zeros(S, np.uint16), r % 8) for r in range(nd)]
    full = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    prev = ss.set_dependent_launch(dependent)
    try:
        for s, t in zip(srcs, staged):
            s.copy_(t)                      # the producer, on the same stream
        flat = ss.fsdp_flat_pack(srcs, nd)
        seen = flat.clone()                 # the consumer, on the same stream
        for s, t in zip(shards, staged_sh):
            s.copy_(t)
        ss.fsdp_ag_unpack(shards, full)
        seen_full = full.clone()
    finally:
        ss.set_dependent_launch(prev)
    torch.cuda.synchronize()
    assert_bits(host_bf16(seen), want, "flat")
    assert_bits(host_bf16(seen_full), want, "full")


def test_copy_launches_of_one_call_replay_from_a_cuda_graph():
    """A pack of 150 bf16 tensors at mixed offsets (several launches of each
    copy kernel, the later ones programmatic dependents) and the all-gather
    of its shards at odd slot offsets, captured once in a CUDA graph and
    replayed on fresh inputs: bit-exact against the oracle every time."""
    nd = 4
    rng = np.random.default_rng(9)
    numels = [int(x) for x in rng.integers(1, 9000, size=149)] + [1 << 18]
    shifts = [int(s) for s in rng.integers(0, 8, size=len(numels))]
    srcs = [dev_bf16(np.zeros(n, np.uint16), sh) for n, sh in zip(numels, shifts)]
    lay = oracle.layout(numels, nd)
    S = lay.shard
    flat = torch.empty(lay.padded, dtype=torch.bfloat16, device=DEV)
    shards = [dev_bf16(np.zeros(S, np.uint16), r % 8) for r in range(nd)]
    full = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm-up outside the capture
        ss.fsdp_flat_pack(srcs, nd, flat=flat)
        ss.fsdp_ag_unpack(shards, full)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ss.fsdp_flat_pack(srcs, nd, flat=flat)
        for r in range(nd):
            shards[r].copy_(flat[r * S:(r + 1) * S])
        ss.fsdp_ag_unpack(shards, full)
    for it in range(3):
        host = [synth.host_fill(synth.normal_stream(it, (93, k), 0.02), 0, n, "bf16")
                for k, n in enumerate(numels)]
        for s, h in zip(srcs, host):
            s.copy_(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16))
        g.replay()
        want, _ = oracle.flat_pack(host, nd)
        torch.cuda.synchronize()
        assert_bits(host_bf16(flat), want, f"flat, replay {it}")
        assert_bits(host_bf16(full), want, f"full, replay {it}")


def test_worked_example_on_gpu():
    tensors = [np.arange(1, 9, dtype=np.float32).reshape(4, 2) + 100 * (t + 1) for t in range(3)]
    flat = ss.fsdp_flat_pack([dev_f32(t.reshape(-1)).view(4, 2) for t in tensors], 2)
    want, lay = oracle.flat_pack(tensors, 2)
    torch.cuda.synchronize()
    assert_bits(host_f32(flat), want, "flat")
    sizes = [[v.numel() for v in ss.fsdp_views(flat[r * 12:(r + 1) * 12], [(4, 2)] * 3, 2, r)]
             for r in range(2)]
    assert sizes == [[8, 4, 0], [0, 4, 8]]


# ------------------------------------------------------------- all-gather

@pytest.mark.parametrize("nd", [1, 2, 3, 8])
@pytest.mark.parametrize("S", [1, 5, 1000, (1 << 20) + 3])
def test_ag_unpack_matches_oracle(nd, S, path):
    shards_h = [synth.host_fill(synth.normal_stream(nd, (96, q, S), 0.02), 0, S, "bf16")
                for q in range(nd)]
    shards = [dev_bf16(h, q % 3) for q, h in enumerate(shards_h)]
    full = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_ag_unpack(shards, full)
    lay = oracle.layout([nd * S], nd)
    want, _ = oracle.ag_unpack(shards_h, lay)
    torch.cuda.synchronize()
    assert_bits(host_bf16(full), want, "full")


def test_ag_unpack_skips_the_rank_already_in_place():
    nd, S = 4, 12345
    shards_h = [synth.host_fill(synth.normal_stream(3, (95, q), 0.02), 0, S, "bf16")
                for q in range(nd)]
    full = torch.zeros(nd * S, dtype=torch.bfloat16, device=DEV)
    full[2 * S:3 * S].copy_(dev_bf16(shards_h[2]))
    shards = [dev_bf16(h) for h in shards_h]
    shards[2] = full[2 * S:3 * S]
    before = ss.launch_count()
    ss.fsdp_ag_unpack(shards, full)
    # one launch per copy kind at most: the 16-byte copy of congruent bodies,
    # the realigning copy of the others, the vector copy of the rest (the
    # shard in place is in none)
    assert 1 <= ss.launch_count() - before <= 3
    torch.cuda.synchronize()
    assert_bits(host_bf16(full), np.concatenate(shards_h), "full")


def test_ag_unpack_views_are_the_unit_tensors(path):
    shapes = [(4096, 11008), (11008,), (3, 5), (4096,)]
    numels = [int(np.prod(s)) for s in shapes]
    nd = 8
    host = [synth.host_fill(synth.normal_stream(2, (94, k), 0.02), 0, n, "bf16")
            for k, n in enumerate(numels)]
    flat = ss.fsdp_flat_pack([dev_bf16(h) for h in host], nd)
    lay = ss.fsdp_layout(numels, nd)
    shards = [flat[r * lay.shard:(r + 1) * lay.shard].clone() for r in range(nd)]
    full = torch.empty(lay.padded, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_ag_unpack(shards, full)
    views = ss.fsdp_views(full, shapes, nd)
    torch.cuda.synchronize()
    for v, h, s in zip(views, host, shapes):
        assert tuple(v.shape) == s
        assert_bits(host_bf16(v).reshape(-1), h, "view")


@pytest.mark.parametrize("shift", [0, 3, 5])
def test_aligned_copy_with_congruent_unaligned_ends(shift, path):
    """Sources and destinations congruent modulo 16 bytes but not aligned:
    the 16-byte copy takes the aligned body, the vector copy the head and
    tail bytes; more than 64 aligned ranges in one call flush mid-way;
    ranges whose last 16 KB chunk is short."""
    nd = 8
    numels = [8 * 16384 + 8 * k + 5 for k in range(70)] + [3 * 1024 * 1024 + 1]
    host = [synth.host_fill(synth.normal_stream(5, (93, k), 0.02), 0, n, "bf16")
            for k, n in enumerate(numels)]
    # every source starts `shift` elements into its allocation; the
    # destination offsets follow the layout, so some ranges are congruent
    flat = ss.fsdp_flat_pack([dev_bf16(h, shift) for h in host], nd)
    want, lay = oracle.flat_pack(host, nd)
    shards = [flat[r * lay.shard:(r + 1) * lay.shard].clone() for r in range(nd)]
    full = torch.empty(lay.padded, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_ag_unpack(shards, full)
    torch.cuda.synchronize()
    assert_bits(host_bf16(flat), want, "flat")
    assert_bits(host_bf16(full), want, "gathered")
    assert ss.device_status() == 0


# ----------------------------------------------------------- accumulation

@pytest.mark.parametrize("n,shift", [(1, 0), (8, 0), (4099, 0), (4099, 1), (1 << 20, 0),
                                     (152 * 256 * 8 * 3 + 7, 0)])
def test_grad_accumulate_matches_oracle(n, shift):
    M = 4
    micro = [synth.host_fill(synth.normal_stream(n, (93, j), 1e-3, 0.01), 0, n, "bf16")
             for j in range(M)]
    acc = torch.full((n + shift + 4,), 7.0, device=DEV)[shift:shift + n]
    scale = np.float32(1.0 / M)
    for j in range(M):
        ss.fsdp_grad_accumulate(dev_bf16(micro[j], shift), acc, float(scale), j == 0)
    want = oracle.grad_accumulate(micro, scale)
    torch.cuda.synchronize()
    assert_bits(host_f32(acc), want, "acc")


# ---------------------------------------------------------------- buckets

@pytest.mark.parametrize("nd", [2, 3, 8, 9, 10, 11, 12, 13, 14, 15, 16, 17])
@pytest.mark.parametrize("cap", [64, 5000, 1 << 22])
def test_ddp_bucketed_step_matches_oracle(nd, cap):
    numels = [768, 3, 768 * 30, 5, 4096 * 3, 768, 1, 2000]
    off, of, boff = ss.ddp_bucket_plan(numels, 2, cap)
    assert (off, of, boff) == tuple(list(x) for x in oracle.bucket_plan(numels, 2, cap))
    total = boff[-1]
    grads_h = [synth.host_fill(synth.normal_stream(nd, (92, q), 1e-3), 0, total, "bf16")
               for q in range(nd)]
    grads = [dev_bf16(h, q % 2) for q, h in enumerate(grads_h)]
    out = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    # bucket by bucket, as each becomes ready
    for b in range(len(boff) - 1):
        ss.ddp_bucket_allreduce_avg(grads, boff, out, first=b, count=1)
    p = synth.host_fill(synth.normal_stream(nd, (92, 100), 0.02), 0, total, "f32")
    dp, dm, dv = dev_f32(p), torch.zeros(total, device=DEV), torch.zeros(total, device=DEV)
    pb = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([out], dp, dm, dv, pb, HPC, 1)
    z = np.zeros(total, np.float32)
    avg, p1, m1, v1, pb1 = oracle.ddp_step(grads_h, boff, p, z, z, HP, 1)
    torch.cuda.synchronize()
    assert_bits(host_bf16(out), avg, "avg")
    assert_bits(host_f32(dp), p1, "master")
    assert_bits(host_f32(dm), m1, "m")
    assert_bits(host_f32(dv), v1, "v")
    assert_bits(host_bf16(pb), pb1, "params")


def test_allreduce_equals_reduce_scatter_then_all_gather_on_gpu():
    nd, S = 8, 10007
    grads_h = [synth.host_fill(synth.normal_stream(4, (91, q), 1e-3), 0, nd * S, "bf16")
               for q in range(nd)]
    grads = [dev_bf16(h) for h in grads_h]
    ar = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
    ss.ddp_bucket_allreduce_avg(grads, [0, nd * S], ar)
    # the same average computed piece by piece, one rank slice per bucket, is
    # the reduce-scatter followed by the all-gather of the pieces
    ar2 = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
    ss.ddp_bucket_allreduce_avg(grads, [r * S for r in range(nd + 1)], ar2)
    torch.cuda.synchronize()
    want = np.concatenate([oracle.f32_to_bf16(oracle.rs_avg(grads_h, r, S)) for r in range(nd)])
    assert_bits(host_bf16(ar), want, "AR")
    assert_bits(host_bf16(ar2), want, "RS+AG")


# ------------------------------------- TMA-staged kernels under stage caps
# The stage count of a TMA-staged launch (chosen for ~128 KB in flight, or
# set) changes only how many tiles are in flight, never a result: every case is
# bit-exact against the oracle under each cap, with tiles dealt unevenly over
# the grid and a ragged tail of < 8 elements.

@pytest.fixture(params=[0, 2, 3, 16])
def stages(request):
    prev = ss.set_tma_stages(request.param)
    yield request.param
    ss.set_tma_stages(prev)


@pytest.mark.parametrize("nd,gdt,S", [(1, "bf16", 2048 * 152 * 2 + 8 * 3 + 5),
                                      (8, "bf16", 2048 * 152 + 2048 * 7 + 16 + 3),
                                      (3, "f32", 70001), (16, "bf16", 70001)])
def test_fused_step_under_stage_caps(nd, gdt, S, stages):
    seed = 11 + S + nd
    contribs = _grads(seed, nd, nd * S, gdt, 1)
    r = nd - 1
    p = synth.host_fill(synth.normal_stream(seed, (99, 2), 0.02), 0, S, "f32")
    m = synth.host_fill(synth.normal_stream(seed, (99, 3), 1e-4), 0, S, "f32")
    v = np.abs(synth.host_fill(synth.normal_stream(seed, (99, 4), 1e-7), 0, S, "f32"))
    dp, dm, dv = dev_f32(p), dev_f32(m), dev_f32(v)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    mk = dev_bf16 if gdt == "bf16" else dev_f32
    ss.fsdp_rs_avg_adamw_cast([mk(c[r * S:(r + 1) * S]) for c in contribs], dp, dm, dv, out,
                              HPC, 3)
    p, m, v, ob = oracle.fsdp_shard_step(contribs, r, S, p, m, v, HP, 3)
    torch.cuda.synchronize()
    assert_bits(host_f32(dp), p, "master")
    assert_bits(host_f32(dm), m, "m")
    assert_bits(host_f32(dv), v, "v")
    assert_bits(host_bf16(out), ob, "bf16")


@pytest.mark.parametrize("n", [4096, 2048 * 152 * 3 + 8 * 11 + 5, (1 << 21) + 7])
def test_grad_accumulate_under_stage_caps(n, stages, path):
    M = 3
    micro = [synth.host_fill(synth.normal_stream(n, (94, j), 1e-3, 0.01), 0, n, "bf16")
             for j in range(M)]
    acc = torch.full((n,), 7.0, device=DEV)
    scale = np.float32(1.0 / M)
    for j in range(M):
        ss.fsdp_grad_accumulate(dev_bf16(micro[j]), acc, float(scale), j == 0)
    want = oracle.grad_accumulate(micro, scale)
    torch.cuda.synchronize()
    assert_bits(host_f32(acc), want, "acc")


@pytest.mark.parametrize("nd", [1, 2, 8, 13])
def test_bucket_allreduce_under_stage_caps(nd, stages, path):
    # buckets: two TMA-eligible ones (16-byte aligned starts, >= 4096
    # elements, one with a ragged tail), a small one, and one whose start is
    # not 16-byte aligned (register-staged)
    boff = [0, 8192, 8192 + 70000, 8192 + 70000 + 4099, 8192 + 70000 + 4099 + 100,
            8192 + 70000 + 4099 + 100 + 9001]
    total = boff[-1]
    grads_h = [synth.host_fill(synth.normal_stream(nd, (95, q), 1e-3), 0, total, "bf16")
               for q in range(nd)]
    grads = [dev_bf16(h) for h in grads_h]
    out = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    for b in range(len(boff) - 1):
        ss.ddp_bucket_allreduce_avg(grads, boff, out, first=b, count=1)
    want = oracle.bucket_allreduce_avg(grads_h, boff)
    torch.cuda.synchronize()
    assert_bits(host_bf16(out), want, "avg")


@pytest.mark.parametrize("dependent", [True, False])
def test_bucket_allreduce_dependent_launches_keep_stream_order(dependent, path):
    """Later buckets of one call may start while the previous bucket's kernel
    drains; the first waits for the gradients' producer (a torch kernel just
    before the call) and a torch kernel right after the call sees every
    bucket's result."""
    nd = 4
    # buckets that take the TMA-staged kernel under path "tma" (>= 4096
    # elements, 16-byte aligned starts) between ones that cannot, two
    # consecutive large ones, a ragged tail
    sizes = [9_000_000, 104, 4096, 8_388_616, 8_388_608, 336, 70_000, 8, 8_388_608, 4099]
    boff = [0]
    for z in sizes:
        boff.append(boff[-1] + z)
    total = boff[-1]
    grads_h = [synth.host_fill(synth.normal_stream(17, (96, q), 1e-3), 0, total, "bf16")
               for q in range(nd)]
    staged = [dev_bf16(h) for h in grads_h]
    grads = [torch.empty_like(g) for g in staged]
    out = torch.full((total,), 5.0, dtype=torch.bfloat16, device=DEV)
    prev = ss.set_dependent_launch(dependent)
    try:
        for g, s in zip(grads, staged):
            g.copy_(s)                      # the producer, on the same stream
        ss.ddp_bucket_allreduce_avg(grads, boff, out)
        seen = out.clone()                  # the consumer, on the same stream
    finally:
        ss.set_dependent_launch(prev)
    want = oracle.bucket_allreduce_avg(grads_h, boff)
    torch.cuda.synchronize()
    assert_bits(host_bf16(seen), want, "avg")


# ------------------------------------------------- which kernel ran

def test_auto_path_names_the_kernel_it_launched():
    """The automatic choice, as shardstep_last_kernel reports it: the
    register-staged fused kernel at N_d = 8, 9 and 15 and its up-to-8 form
    at 7; the TMA-staged one at N_d = 17 and with 9 fp32 slices, the loop
    over any N_d with 16 fp32 slices; TMA-staged whenever forced; the all-reduce
    and the check on their register kernels at N_d = 1..16 (16-bit slices),
    on the TMA-staged ones above 16."""
    S = 8192
    master = torch.zeros(S, device=DEV)
    m = torch.zeros(S, device=DEV)
    v = torch.zeros(S, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    prev = ss.set_fused_path("auto")
    try:
        for nd, dt, want in [
                (8, torch.bfloat16, "rs_adamw_cast_vec4<8, bf16> (register-staged)"),
                (7, torch.bfloat16, "rs_adamw_cast_vec4<up to 8: 7, bf16> (register-staged)"),
                (9, torch.bfloat16, "rs_adamw_cast_vec4<9, bf16> (register-staged)"),
                (15, torch.bfloat16, "rs_adamw_cast_vec4<15, bf16> (register-staged)"),
                (17, torch.bfloat16, "staged_stream<AdamOp<bf16>> (TMA-staged)"),
                (9, torch.float32, "staged_stream<AdamOp<f32>> (TMA-staged)"),
                (16, torch.float32,
                 "rs_adamw_cast_vec4<any N_d = 16, f32> (register-staged)")]:
            g = [torch.zeros(S, dtype=dt, device=DEV) for _ in range(nd)]
            ss.fsdp_rs_avg_adamw_cast(g, master, m, v, out, HPC, 1)
            assert ss.last_kernel() == want, (nd, dt)
        g = [torch.zeros(S, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
        ss.set_fused_path("tma")
        ss.fsdp_rs_avg_adamw_cast(g, master, m, v, out, HPC, 1)
        assert ss.last_kernel() == "staged_stream<AdamOp<bf16>> (TMA-staged)"
        ss.set_fused_path("register")
        ss.fsdp_rs_avg_adamw_cast([x[1:] for x in g], master[1:], m[1:], v[1:], out[1:], HPC, 1)
        assert ss.last_kernel() == "rs_adamw_cast_scalar<bf16>"
        acc = torch.zeros(S, device=DEV)
        ss.set_fused_path("auto")
        ss.fsdp_grad_accumulate(g[0], acc, 0.25, True)
        assert ss.last_kernel() == "accumulate_vec8 (register-staged)"
        # the bucket all-reduce and the check by N_d
        g = g + [torch.zeros(S, dtype=torch.bfloat16, device=DEV) for _ in range(9)]
        out16 = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        for nd, want in [(3, "allreduce_avg_vec4<3> (register-staged)"),
                         (8, "allreduce_avg_vec4<8> (register-staged)"),
                         (6, "allreduce_avg_vec4<6> (register-staged)"),
                         (10, "allreduce_avg_vec4<10> (register-staged)"),
                         (16, "allreduce_avg_vec4<16> (register-staged)"),
                         (17, "staged_stream<MeanOutOp> (TMA-staged)")]:
            ss.ddp_bucket_allreduce_avg(g[:nd], [0, S], out16)
            assert ss.last_kernel() == want, nd
        h = [x.to(torch.float16) for x in g]
        sc = ss.GradScaler(1.0, device=DEV)
        for nd, want in [(1, "nonfinite_check_vec4<1, f16> (register-staged)"),
                         (3, "nonfinite_check_vec4<3, f16> (register-staged)"),
                         (8, "nonfinite_check_vec4<8, f16> (register-staged)"),
                         (5, "nonfinite_check_vec4<5, f16> (register-staged)"),
                         (10, "nonfinite_check_vec4<10, f16> (register-staged)"),
                         (16, "nonfinite_check_vec4<16, f16> (register-staged)"),
                         (17, "staged_stream<CheckOp<f16>> (TMA-staged)")]:
            sc.check(h[:nd])
            assert ss.last_kernel() == want, nd
        torch.cuda.synchronize()
    finally:
        ss.set_fused_path(prev)
