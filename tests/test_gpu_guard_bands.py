"""Out-of-bounds writes, caught without a sanitizer: every output of every
entry point lives inside a larger buffer whose bytes before and after it
hold a sentinel pattern, and the pattern must survive the call.  Sizes are
ragged (tails past the last tile, misaligned starts) and every kernel
choice runs (TMA-staged, register-staged, auto)."""
import numpy as np
import pytest
import torch

import sharded_optimizer_step_gb300 as ss
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096          # bytes of sentinel on each side of an output
PATTERN = 0xA5


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


class Guarded:
    """An output tensor of `n` elements at byte offset GUARD + shift*itemsize
    inside a buffer filled with the sentinel byte."""

    def __init__(self, n, dtype, shift=0, fill=None):
        isz = torch.empty(0, dtype=dtype).element_size()
        self.lo = GUARD + shift * isz
        self.nbytes = n * isz
        self.raw = torch.full((self.lo + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device=DEV)
        self.t = self.raw[self.lo:self.lo + self.nbytes].view(dtype)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, what):
        torch.cuda.synchronize()
        before = self.raw[:self.lo]
        after = self.raw[self.lo + self.nbytes:]
        assert bool((before == PATTERN).all()), f"{what}: bytes before the output were written"
        assert bool((after == PATTERN).all()), f"{what}: bytes after the output were written"


def _bf16(n, seed, sigma=1e-3, shift=0):
    h = synth.host_fill(synth.normal_stream(seed, (77, n), sigma), 0, n, "bf16")
    buf = torch.empty(n + shift + 8, dtype=torch.bfloat16, device=DEV)
    t = buf[shift:shift + n]
    t.copy_(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16))
    return t


@pytest.mark.parametrize("nd,S,shift", [(1, 4099, 0), (2, 2048 * 152 + 13, 0), (8, 70001, 0),
                                        (8, 70001, 1), (16, 2048 * 3 + 5, 0), (3, 13, 0)])
def test_fused_step_writes_only_its_outputs(nd, S, shift, path):
    grads = [_bf16(S, q) for q in range(nd)]
    master = Guarded(S, torch.float32, shift, torch.randn(S, device=DEV) * 0.02)
    m = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    v = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    out = Guarded(S, torch.bfloat16, shift)
    ss.fsdp_rs_avg_adamw_cast(grads, master.t, m.t, v.t, out.t, ss.AdamW(), 1)
    for name, g in (("master", master), ("m", m), ("v", v), ("bf16", out)):
        g.check(f"fused step {name}")


def _f16(n, seed, shift=0):
    h = synth.host_fill(synth.normal_stream(seed, (78, n), 0.3), 0, n, "f16")
    buf = torch.empty(n + shift + 8, dtype=torch.float16, device=DEV)
    t = buf[shift:shift + n]
    t.copy_(torch.from_numpy(h.view(np.int16)).view(torch.float16))
    return t


@pytest.mark.parametrize("variant", ["hybrid", "state", "scaled", "scaled_state"])
@pytest.mark.parametrize("nd,F,S,shift", [(8, 4, 70001, 0), (8, 4, 70001, 1), (6, 3, 2048 * 152 + 13, 0),
                                          (16, 8, 4099, 0), (4, 2, 13, 0)])
def test_fused_step_variants_write_only_their_outputs(variant, nd, F, S, shift, path):
    """The fused step's other instantiations (grouped reduce order, AdamW
    scalars from the device state, fp16 gradients under loss scaling): the
    same bands around master / m / v / out, and the scaler's words read,
    not written, by the step."""
    scaled = variant.startswith("scaled")
    grads = ([_f16(S, 30 + q, shift) for q in range(nd)] if scaled
             else [_bf16(S, 30 + q, shift=shift) for q in range(nd)])
    master = Guarded(S, torch.float32, shift, torch.randn(S, device=DEV) * 0.02)
    m = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    v = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    out = Guarded(S, torch.bfloat16, shift)
    group = None if variant == "scaled" else F
    hp = ss.AdamW()
    st = ss.AdamWState(hp, 1, device=DEV)
    if variant == "hybrid":
        ss.fsdp_hybrid_rs_avg_adamw_cast(grads, F, master.t, m.t, v.t, out.t, hp, 1)
    elif variant == "state":
        ss.fsdp_state_rs_avg_adamw_cast(grads, master.t, m.t, v.t, out.t, st, shard_group=group)
    else:
        sc = ss.GradScaler(init_scale=1024.0, device=DEV)
        sc.check(grads, shard_group=group)
        words = (sc.scale.clone(), sc.found_inf.clone())
        if variant == "scaled":
            sc.step(grads, master.t, m.t, v.t, out.t, hp, 1)
        else:
            sc.step_state(grads, master.t, m.t, v.t, out.t, st, shard_group=group)
        torch.cuda.synchronize()
        assert torch.equal(sc.scale, words[0]) and torch.equal(sc.found_inf, words[1])
        assert int(sc.found_inf.item()) == 0
    for name, g in (("master", master), ("m", m), ("v", v), ("bf16", out)):
        g.check(f"{variant} fused step {name}")


@pytest.mark.parametrize("n,shift", [(4096 + 3, 0), (2048 * 152 * 2 + 7, 0), (10001, 1), (5, 0)])
def test_accumulate_writes_only_the_accumulator(n, shift, path):
    acc = Guarded(n, torch.float32, shift)
    for j in range(3):
        ss.fsdp_grad_accumulate(_bf16(n, 10 + j), acc.t, 1.0 / 3, j == 0)
    acc.check("accumulate")


@pytest.mark.parametrize("nd", [2, 8])
def test_bucket_allreduce_writes_only_its_buckets(nd, path):
    boff = [0, 4096, 4096 + 70003, 4096 + 70003 + 5, 4096 + 70003 + 5 + 40000]
    total = boff[-1]
    grads = [_bf16(total, 20 + q) for q in range(nd)]
    out = Guarded(total, torch.bfloat16)
    ss.ddp_bucket_allreduce_avg(grads, boff, out.t)
    out.check("all-reduce")
    # a single bucket in the middle writes only its own range
    mid = Guarded(total, torch.bfloat16)
    ss.ddp_bucket_allreduce_avg(grads, boff, mid.t, first=1, count=1)
    torch.cuda.synchronize()
    raw = mid.raw.cpu().numpy()
    a, e = mid.lo + boff[1] * 2, mid.lo + boff[2] * 2
    assert (raw[:a] == PATTERN).all() and (raw[e:] == PATTERN).all()


def test_check_writes_only_the_found_word(path):
    S, nd = 2048 * 152 + 11, 8
    grads = [_bf16(S, 30 + q, sigma=300.0) for q in range(nd)]
    sc = ss.GradScaler(init_scale=65536.0, device=DEV)
    found = Guarded(1, torch.int32, fill=torch.zeros(1, dtype=torch.int32, device=DEV))
    sc.found_inf = found.t
    sc.check([g.to(torch.float16) for g in grads])
    found.check("found_inf")


@pytest.mark.parametrize("S", [1000, (1 << 17) + 3, 2048 * 152 * 4 + 8])
def test_all_gather_writes_only_the_full_buffer(S, path):
    nd = 8
    shards = [_bf16(S, 40 + q, 0.02, shift=q % 2) for q in range(nd)]
    full = Guarded(nd * S, torch.bfloat16, shift=3)
    ss.fsdp_ag_unpack(shards, full.t)
    full.check("all-gather")


def test_flat_pack_writes_only_the_flat_buffer(path):
    nd = 8
    numels = [1 << 18, 5, (1 << 16) + 1, 3, 70001]
    tensors = [_bf16(n, 50 + k, 0.02, shift=k % 3) for k, n in enumerate(numels)]
    lay = ss.fsdp_layout(numels, nd)
    flat = Guarded(lay.padded, torch.bfloat16)
    ss.fsdp_flat_pack(tensors, nd, flat=flat.t)
    flat.check("flat_pack")


def test_fsdp2_copies_write_only_their_buffers(path):
    nd = 4
    shapes = [(1023, 130), (7,), (300, 512)]
    grads = [_bf16(int(np.prod(s)), 60 + k).view(s) for k, s in enumerate(shapes)]
    lay = ss.fsdp2_layout(shapes, nd)
    buf = Guarded(nd * lay.local, torch.bfloat16)
    ss.fsdp2_chunk_cat(grads, nd, out=buf.t)
    buf.check("chunk-cat")
    outs = [Guarded(int(np.prod(s)), torch.bfloat16, shift=k) for k, s in enumerate(shapes)]
    locals_ = [buf.t[r * lay.local:(r + 1) * lay.local] for r in range(nd)]
    ss.fsdp2_all_gather_copy_out(locals_, [o.t.view(s) for o, s in zip(outs, shapes)])
    for k, o in enumerate(outs):
        o.check(f"copy-out {k}")


def _f32(n, seed, sigma=1e-3, shift=0):
    h = synth.host_fill(synth.normal_stream(seed, (78, n), sigma), 0, n, "f32")
    buf = torch.empty(n + shift + 8, dtype=torch.float32, device=DEV)
    t = buf[shift:shift + n]
    t.copy_(torch.from_numpy(h))
    return t


@pytest.mark.parametrize("nd,F", [(8, 8), (8, 4), (9, 3), (2, 2), (6, 2)])
@pytest.mark.parametrize("S,shift", [(4099, 0), (2048 * 152 + 13, 0), (70001, 1), (13, 0)])
@pytest.mark.parametrize("state", [False, True])
def test_fused_last_micro_batch_writes_only_its_outputs(nd, F, S, shift, state, path):
    """The last micro-batch accumulated inside the fused step, plain and
    hybrid, host scalars and device step state: master / m / v / out inside
    sentinel bands, and the accumulator and last-gradient slices (also in
    bands) read, never written."""
    acc = [Guarded(S, torch.float32, shift, _f32(S, 80 + q)) for q in range(nd)]
    last = [Guarded(S, torch.bfloat16, shift, _bf16(S, 90 + q)) for q in range(nd)]
    before = [a.t.clone() for a in acc] + [g.t.clone() for g in last]
    master = Guarded(S, torch.float32, shift, torch.randn(S, device=DEV) * 0.02)
    m = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    v = Guarded(S, torch.float32, shift, torch.zeros(S, device=DEV))
    out = Guarded(S, torch.bfloat16, shift)
    hp = ss.AdamW()
    args = ([a.t for a in acc], [g.t for g in last], 0.25, master.t, m.t, v.t, out.t)
    if state:
        st = ss.AdamWState(hp, 0, device=DEV)
        st.advance()
        ss.fsdp_state_accumulate_rs_avg_adamw_cast(*args, st, shard_group=F)
    else:
        ss.fsdp_accumulate_rs_avg_adamw_cast(*args, hp, 1, shard_group=F)
    for name, g in (("master", master), ("m", m), ("v", v), ("bf16", out)):
        g.check(f"fused last micro-batch {name}")
    for k, (g, b) in enumerate(zip(acc + last, before)):
        g.check(f"input slice {k}")
        assert torch.equal(g.t.view(torch.uint8), b.view(torch.uint8)), f"input slice {k} written"


@pytest.mark.parametrize("nd", [1, 3, 8])
@pytest.mark.parametrize("keep_mean", [False, True])
def test_fused_ddp_step_writes_only_its_outputs(nd, keep_mean):
    boff = [0, 4096, 4096 + 70003, 4096 + 70003 + 5, 4096 + 70003 + 5 + 40000]
    total = boff[-1]
    grads = [Guarded(total, torch.bfloat16, q % 2, _bf16(total, 100 + q)) for q in range(nd)]
    before = [g.t.clone() for g in grads]
    master = Guarded(total, torch.float32, 1, torch.randn(total, device=DEV) * 0.02)
    m = Guarded(total, torch.float32, 1, torch.zeros(total, device=DEV))
    v = Guarded(total, torch.float32, 1, torch.zeros(total, device=DEV))
    pb = Guarded(total, torch.bfloat16, 1)
    mean = Guarded(total, torch.bfloat16, 3) if keep_mean else None
    ss.ddp_bucket_allreduce_avg_adamw_cast([g.t for g in grads], boff, master.t, m.t, v.t, pb.t,
                                           ss.AdamW(), 1, mean_out=mean.t if mean else None)
    # one bucket in the middle touches only its own range of every output
    ss.ddp_bucket_allreduce_avg_adamw_cast([g.t for g in grads], boff, master.t, m.t, v.t, pb.t,
                                           ss.AdamW(), 2, first=2, count=1)
    for name, g in (("master", master), ("m", m), ("v", v), ("params", pb)) + \
            ((("mean", mean),) if mean else ()):
        g.check(f"fused DDP {name}")
    for q, (g, b) in enumerate(zip(grads, before)):
        g.check(f"gradient {q}")
        assert torch.equal(g.t.view(torch.uint8), b.view(torch.uint8)), f"gradient {q} written"


@pytest.mark.parametrize("nd", [1, 3, 8])
def test_fsdp2_step_without_chunk_cat_writes_only_its_outputs(nd, path):
    """The FSDP2 step read straight from the gradients (uneven dim 0, so
    padding rows get their own launch): master / m / v / out inside bands,
    the gradients (also in bands) read, never written."""
    shapes = [(1023, 130), (7,), (300, 512), (5, 3)]
    L = ss.fsdp2_layout(shapes, nd).local
    grads = [[Guarded(int(np.prod(s)), torch.bfloat16, (q + k) % 3,
                      _bf16(int(np.prod(s)), 200 + 10 * q + k)) for k, s in enumerate(shapes)]
             for q in range(nd)]
    before = [g.t.clone() for gs in grads for g in gs]
    outs = [Guarded(L, torch.float32, 1, torch.randn(L, device=DEV) * 0.02),
            Guarded(L, torch.float32, 1, torch.zeros(L, device=DEV)),
            Guarded(L, torch.float32, 1, torch.zeros(L, device=DEV)),
            Guarded(L, torch.bfloat16, 3)]
    for r in range(nd):
        ss.fsdp2_rs_avg_adamw_cast([[g.t.view(s) for g, s in zip(gs, shapes)] for gs in grads], r,
                                   *[o.t for o in outs], ss.AdamW(), 1)
        for name, o in zip(("master", "m", "v", "bf16"), outs):
            o.check(f"FSDP2 step rank {r} {name}")
    for k, (g, b) in enumerate(zip([g for gs in grads for g in gs], before)):
        g.check(f"gradient {k}")
        assert torch.equal(g.t.view(torch.uint8), b.view(torch.uint8)), f"gradient {k} written"
