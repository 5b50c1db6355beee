"""Reads stay inside their inputs, checked without a sanitizer.

Every input of a call (gradient slices, accumulators, the fp32 state, the
shards and tensors a copy reads) sits inside a larger buffer whose bytes
before and after it hold a poison byte; the call runs three times, with the
poison 0x00, 0xFF (NaN in bf16, fp16 and fp32) and 0x7F (NaN in fp16, the
largest finite magnitudes in bf16 and fp32), and the outputs must be the
same bytes each time.  A kernel that used a byte outside an input would
turn it into a different sum, a NaN or an overflow; the gradient scaler's
check would report a non-finite value that is not there.  Sizes are ragged
(tails past the last tile and vector, misaligned starts) and every kernel
choice runs."""
import numpy as np
import pytest
import torch

import sharded_optimizer_step_gb300 as ss
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096
POISONS = (0x00, 0xFF, 0x7F)


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


def _host(kind, n, seed, sigma):
    return synth.host_fill(synth.normal_stream(seed, (79, n), sigma), 0, n, kind)


_TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _poisoned(h, kind, shift, poison):
    """Device copy of host bits ``h`` at byte offset GUARD + shift * size in a
    buffer whose other bytes are ``poison``."""
    dt = _TORCH[kind]
    isz = torch.empty(0, dtype=dt).element_size()
    lo = GUARD + shift * isz
    raw = torch.full((lo + h.size * isz + GUARD,), poison, dtype=torch.uint8, device=DEV)
    raw[lo:lo + h.size * isz].copy_(torch.from_numpy(np.ascontiguousarray(h).view(np.uint8)))
    return raw[lo:lo + h.size * isz].view(dt)


def _bytes(*ts):
    torch.cuda.synchronize()
    return [t.contiguous().view(torch.uint8).cpu().numpy().copy() for t in ts]


def _same_for_every_poison(run):
    ref = run(POISONS[0])
    for p in POISONS[1:]:
        got = run(p)
        for k, (a, b) in enumerate(zip(ref, got)):
            assert np.array_equal(a, b), f"output {k} depends on the bytes around an input " \
                                         f"(poison {p:#04x})"


@pytest.mark.parametrize("nd,F,kind", [(8, 8, "bf16"), (3, 3, "bf16"), (8, 4, "bf16"),
                                       (4, 4, "f32"), (12, 12, "bf16"), (16, 8, "bf16"),
                                       (5, 5, "f32")])
@pytest.mark.parametrize("S,shift", [(4099, 0), (2048 * 152 + 13, 1), (70001, 3), (7, 0)])
def test_fused_step_reads_only_its_inputs(nd, F, kind, S, shift, path):
    gh = [_host(kind, S, 10 + q, 1e-3) for q in range(nd)]
    ph = _host("f32", S, 30, 0.02)
    mh = _host("f32", S, 31, 1e-4)
    vh = np.abs(_host("f32", S, 32, 1e-6)).astype(np.float32)

    def run(poison):
        g = [_poisoned(h, kind, shift * (q % 2), poison) for q, h in enumerate(gh)]
        p, m, v = (_poisoned(x, "f32", shift, poison) for x in (ph, mh, vh))
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        ss.fsdp_hybrid_rs_avg_adamw_cast(g, F, p, m, v, out, ss.AdamW(), 3)
        return _bytes(p, m, v, out)

    _same_for_every_poison(run)


@pytest.mark.parametrize("nd", [1, 3, 8, 13])
@pytest.mark.parametrize("S,shift", [(4099, 0), (2048 * 152 + 13, 1), (7, 0)])
def test_scaler_check_and_step_read_only_their_inputs(nd, S, shift, path):
    gh = [_host("f16", S, 40 + q, 0.3) for q in range(nd)]
    ph = _host("f32", S, 41, 0.02)

    def run(poison):
        g = [_poisoned(h, "f16", shift * (q % 2), poison) for q, h in enumerate(gh)]
        p = _poisoned(ph, "f32", shift, poison)
        m = _poisoned(np.zeros(S, np.float32), "f32", shift, poison)
        v = _poisoned(np.zeros(S, np.float32), "f32", shift, poison)
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        sc = ss.GradScaler(init_scale=256.0, device=DEV)
        sc.check(g)
        sc.step(g, p, m, v, out, ss.AdamW(), 1)
        torch.cuda.synchronize()
        assert int(sc.found_inf.item()) == 0, f"a non-finite value found (poison {poison:#04x})"
        return _bytes(p, m, v, out)

    _same_for_every_poison(run)


@pytest.mark.parametrize("nd,F", [(8, 8), (4, 2), (7, 7)])
@pytest.mark.parametrize("S,shift", [(4099, 0), (2048 * 152 + 13, 1), (9, 0)])
def test_fused_last_micro_batch_reads_only_its_inputs(nd, F, S, shift, path):
    ah = [_host("f32", S, 50 + q, 1e-3) for q in range(nd)]
    lh = [_host("bf16", S, 60 + q, 1e-3) for q in range(nd)]
    ph = _host("f32", S, 70, 0.02)

    def run(poison):
        acc = [_poisoned(h, "f32", shift, poison) for h in ah]
        last = [_poisoned(h, "bf16", shift * (q % 2), poison) for q, h in enumerate(lh)]
        p = _poisoned(ph, "f32", shift, poison)
        m = _poisoned(np.zeros(S, np.float32), "f32", shift, poison)
        v = _poisoned(np.zeros(S, np.float32), "f32", shift, poison)
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        ss.fsdp_accumulate_rs_avg_adamw_cast(acc, last, 0.25, p, m, v, out, ss.AdamW(), 1,
                                             shard_group=F)
        return _bytes(p, m, v, out)

    _same_for_every_poison(run)


@pytest.mark.parametrize("n,shift", [(4096 + 3, 0), (2048 * 152 * 2 + 7, 1), (5, 0)])
def test_accumulate_reads_only_its_inputs(n, shift, path):
    gh = [_host("bf16", n, 80 + j, 1e-3) for j in range(3)]

    def run(poison):
        acc = _poisoned(np.zeros(n, np.float32), "f32", shift, poison)
        for j, h in enumerate(gh):
            ss.fsdp_grad_accumulate(_poisoned(h, "bf16", shift if j == 1 else 0, poison), acc,
                                    1.0 / 3, j == 0)
        return _bytes(acc)

    _same_for_every_poison(run)


@pytest.mark.parametrize("nd", [1, 3, 8, 11])
def test_bucket_allreduce_and_fused_ddp_read_only_their_inputs(nd, path):
    boff = [0, 4096, 4096 + 70003, 4096 + 70003 + 5, 4096 + 70003 + 5 + 40001]
    total = boff[-1]
    gh = [_host("bf16", total, 90 + q, 1e-3) for q in range(nd)]
    ph = _host("f32", total, 99, 0.02)

    def run(poison):
        g = [_poisoned(h, "bf16", q % 2, poison) for q, h in enumerate(gh)]
        mean = torch.empty(total, dtype=torch.bfloat16, device=DEV)
        ss.ddp_bucket_allreduce_avg(g, boff, mean)
        p = _poisoned(ph, "f32", 1, poison)
        m = _poisoned(np.zeros(total, np.float32), "f32", 1, poison)
        v = _poisoned(np.zeros(total, np.float32), "f32", 1, poison)
        params = torch.empty(total, dtype=torch.bfloat16, device=DEV)
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, boff, p, m, v, params, ss.AdamW(), 1)
        return _bytes(mean, p, m, v, params)

    _same_for_every_poison(run)


def test_copies_read_only_their_sources(path):
    nd = 8
    numels = [1 << 18, 5, (1 << 16) + 1, 3, 70001]
    th = [_host("bf16", n, 110 + k, 0.02) for k, n in enumerate(numels)]
    S = 70001
    sh = [_host("bf16", S, 120 + q, 0.02) for q in range(nd)]
    shapes = [(1023, 130), (7,), (300, 512)]
    fh = [_host("bf16", int(np.prod(s)), 130 + k, 0.02) for k, s in enumerate(shapes)]
    flay = ss.fsdp2_layout(shapes, 4)

    def run(poison):
        tensors = [_poisoned(h, "bf16", k % 3, poison) for k, h in enumerate(th)]
        flat = ss.fsdp_flat_pack(tensors, nd)
        shards = [_poisoned(h, "bf16", q % 2, poison) for q, h in enumerate(sh)]
        full = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
        ss.fsdp_ag_unpack(shards, full)
        grads = [_poisoned(h, "bf16", k, poison).view(s) for k, (h, s) in enumerate(zip(fh, shapes))]
        cc = ss.fsdp2_chunk_cat(grads, 4)
        locals_ = [_poisoned(cc[r * flay.local:(r + 1) * flay.local].contiguous().view(
            torch.int16).cpu().numpy().view(np.uint16), "bf16", r % 2, poison) for r in range(4)]
        outs = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
        ss.fsdp2_all_gather_copy_out(locals_, outs)
        return _bytes(flat, full, cc, *outs)

    _same_for_every_poison(run)


@pytest.mark.parametrize("nd", [1, 3, 8])
def test_fsdp2_step_without_chunk_cat_reads_only_its_inputs(nd, path):
    shapes = [(1023, 130), (7,), (300, 512), (5, 3)]
    L = ss.fsdp2_layout(shapes, nd).local
    gh = [[_host("bf16", int(np.prod(s)), 140 + 10 * q + k, 1e-3) for k, s in enumerate(shapes)]
          for q in range(nd)]
    ph = _host("f32", L, 150, 0.02)

    def run(poison):
        grads = [[_poisoned(h, "bf16", (q + k) % 3, poison).view(s)
                  for k, (h, s) in enumerate(zip(gs, shapes))] for q, gs in enumerate(gh)]
        res = []
        for r in range(nd):
            p = _poisoned(ph, "f32", 1, poison)
            m = _poisoned(np.zeros(L, np.float32), "f32", 1, poison)
            v = _poisoned(np.zeros(L, np.float32), "f32", 1, poison)
            out = torch.empty(L, dtype=torch.bfloat16, device=DEV)
            ss.fsdp2_rs_avg_adamw_cast(grads, r, p, m, v, out, ss.AdamW(), 1)
            res += _bytes(p, m, v, out)
        return res

    _same_for_every_poison(run)
