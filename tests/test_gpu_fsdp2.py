"""GPU parity of the FSDP2 per-parameter Shard(0) path against the oracle:
chunk-cat (the reduce-scatter input), the fused step on the padded local
buffers, and the all-gather straight into full per-parameter tensors, on
uneven dim 0, misaligned tensors and the model-shaped groups."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from synth import workloads as W
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = AdamWConfig()
HPC = ss.AdamW()

SHAPE_SETS = [
    [(4, 2), (4, 2), (4, 2)],
    [(8, 4)],
    [(7, 3), (5,), (9, 2), (1, 17), (0, 4), (3,)],
    [(2304, 768), (2304,), (768, 768), (768,), (3072, 768), (3072,), (768, 3072), (768,),
     (768,), (768,), (768,), (768,)],
    [(4097, 5), (13,), (1030, 3)],
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()


@pytest.fixture(params=["auto", "register", "tma"])
def path(request):
    """Each kernel choice: auto and tma (aligned copy bodies on the 16-byte
    copy), and register-staged only (every copy on the generic vector
    copy)."""
    prev = ss.set_fused_path(request.param)
    yield request.param
    ss.set_fused_path(prev)


def _dev(h, shift=0):
    dt = torch.bfloat16 if h.dtype == np.uint16 else torch.float32
    buf = torch.empty(h.size + shift + 8, dtype=dt, device=DEV)
    t = buf[shift:shift + h.size]
    src = torch.from_numpy(np.ascontiguousarray(h).view(np.int16 if h.dtype == np.uint16
                                                        else np.float32))
    t.copy_(src.view(dt))
    return t


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def _tensors(shapes, seed, dtype):
    return [synth.host_fill(synth.normal_stream(seed, (90, t), 1e-3), 0, int(np.prod(s)),
                            dtype).reshape(s) for t, s in enumerate(shapes)]


@pytest.mark.parametrize("shapes", SHAPE_SETS, ids=lambda s: f"{len(s)}params")
@pytest.mark.parametrize("nd", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_cat_and_copy_out_match_oracle(shapes, nd, dtype, path):
    host = _tensors(shapes, nd, dtype)
    dev = [_dev(h.reshape(-1), t % 3).view(s) for t, (h, s) in enumerate(zip(host, shapes))]
    lay = oracle.fsdp2_layout(shapes, nd)
    cc = ss.fsdp2_chunk_cat(dev, nd)
    want = oracle.chunk_cat(host, lay)
    torch.cuda.synchronize()
    assert_bits(_host(cc), want, "chunk_cat")
    # local views have the DTensor local shapes
    for r in range(nd):
        loc = ss.fsdp2_local_views(cc[r * lay.local:(r + 1) * lay.local], shapes, nd, r)
        for t, (a, b) in enumerate(zip(loc, oracle.local_shards(host, lay, r))):
            assert tuple(a.shape) == b.shape
            assert_bits(_host(a).reshape(-1), b.reshape(-1), f"local {r} {t}")
    # all-gather the rank pieces back into full tensors
    bufs = [cc[r * lay.local:(r + 1) * lay.local].clone() for r in range(nd)]
    outs = [torch.full(s, 7.0, dtype=dev[0].dtype, device=DEV) for s in shapes]
    ss.fsdp2_all_gather_copy_out(bufs, outs)
    torch.cuda.synchronize()
    for o, h in zip(outs, host):
        assert_bits(_host(o).reshape(-1), h.reshape(-1), "copy-out")


@pytest.mark.parametrize("shapes", SHAPE_SETS[2:], ids=lambda s: f"{len(s)}params")
@pytest.mark.parametrize("nd", [2, 8])
def test_fsdp2_step_matches_oracle(shapes, nd, path):
    # every rank: chunk-cat its gradients; rank r: fused step on its padded
    # local buffer with the nd pieces r; then the all-gather copy-out
    lay = oracle.fsdp2_layout(shapes, nd)
    masters = [synth.host_fill(synth.normal_stream(3, (89, t), 0.02), 0, int(np.prod(s)),
                               "f32").reshape(s) for t, s in enumerate(shapes)]
    state = []
    for r in range(nd):
        p = oracle.local_buffer(masters, lay, r)
        state.append(dict(p=p, m=np.zeros(lay.local, np.float32), v=np.zeros(lay.local, np.float32),
                          dp=_dev(p), dm=torch.zeros(lay.local, device=DEV),
                          dv=torch.zeros(lay.local, device=DEV),
                          out=torch.empty(lay.local, dtype=torch.bfloat16, device=DEV)))
    for t in (1, 2):
        grads = [_tensors(shapes, 100 * t + q, "bf16") for q in range(nd)]
        cc_h = [oracle.chunk_cat(g, lay) for g in grads]
        cc = [ss.fsdp2_chunk_cat([_dev(x.reshape(-1)).view(x.shape) for x in g], nd) for g in grads]
        for r, st in enumerate(state):
            ss.fsdp_rs_avg_adamw_cast([c[r * lay.local:(r + 1) * lay.local] for c in cc],
                                      st["dp"], st["dm"], st["dv"], st["out"], HPC, t)
            st["p"], st["m"], st["v"], st["ob"] = oracle.fsdp_shard_step(
                cc_h, r, lay.local, st["p"], st["m"], st["v"], HP, t)
    params = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    ss.fsdp2_all_gather_copy_out([st["out"] for st in state], params)
    want_params = oracle.all_gather_copy_out([st["ob"] for st in state], lay)
    torch.cuda.synchronize()
    for st in state:
        assert_bits(_host(st["dp"]), st["p"], "master")
        assert_bits(_host(st["dm"]), st["m"], "m")
        assert_bits(_host(st["dv"]), st["v"], "v")
        assert_bits(_host(st["out"]), st["ob"], "bf16 local")
    for a, b in zip(params, want_params):
        assert_bits(_host(a).reshape(-1), b.reshape(-1), "gathered parameter")


def test_fsdp2_llama_layer_group_full_size():
    # one Llama-7B layer as an FSDP2 group on 8 ranks, every rank emulated:
    # chunk-cat of each rank's full gradients, 8 fused steps, copy-out
    w = W.llama_7b_rank_view()
    shapes = w.units[0]
    nd = 8
    lay = ss.fsdp2_layout(shapes, nd)
    assert lay.local == 202_383_360 // 8
    olay = oracle.fsdp2_layout(shapes, nd)
    grads = [[torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes] for _ in range(nd)]
    for q in range(nd):
        for t, g in enumerate(grads[q]):
            synth.dev_fill(w.grad_stream(1, q, 0, 100, t), g)
    cc = [ss.fsdp2_chunk_cat(grads[q], nd) for q in range(nd)]
    rng = np.random.default_rng(5)
    masters = [torch.empty(s, dtype=torch.float32, device=DEV) for s in shapes]
    for t, mt in enumerate(masters):
        synth.dev_fill(w.master_stream(100, t), mt)
    local_master = ss.fsdp2_chunk_cat(masters, nd)
    outs = []
    for r in range(nd):
        sl = slice(r * lay.local, (r + 1) * lay.local)
        mm = torch.zeros(lay.local, device=DEV)
        vv = torch.zeros(lay.local, device=DEV)
        out = torch.empty(lay.local, dtype=torch.bfloat16, device=DEV)
        ss.fsdp_rs_avg_adamw_cast([c[sl] for c in cc], local_master[sl], mm, vv, out, HPC, 1)
        outs.append(out)
    params = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    ss.fsdp2_all_gather_copy_out(outs, params)
    torch.cuda.synchronize()
    # oracle on sampled rows of every parameter
    for t, s in enumerate(shapes):
        rows = np.unique(np.concatenate([rng.integers(0, s[0], 24), [0, s[0] - 1]]))
        row = int(np.prod(s[1:]))
        cols = np.unique(np.concatenate([rng.integers(0, row, 16), [0, row - 1]]))
        flat_idx = (rows[:, None] * row + cols[None, :]).reshape(-1)
        gq = [synth.host_gather(w.grad_stream(1, q, 0, 100, t), flat_idx, "bf16")
              for q in range(nd)]
        p0 = synth.host_gather(w.master_stream(100, t), flat_idx, "f32")
        z = np.zeros(flat_idx.size, np.float32)
        _, _, _, ob = oracle.fsdp_shard_step(gq, 0, flat_idx.size, p0, z, z, HP, 1)
        got = _host(params[t].reshape(-1)[torch.from_numpy(flat_idx).to(DEV)])
        assert_bits(got, ob, f"param {t}")
    del olay


# ------------------------------------ the step read straight from the gradients

def _f32_dev(h):
    return torch.from_numpy(np.ascontiguousarray(h, dtype=np.float32)).to(DEV)


def _dev_grad(h, gdt):
    if gdt == "f16":
        return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(DEV).view(
            torch.float16)
    return _dev(h)


def _oracle_contribs(cc, gdt):
    """fp16 contributions widened to fp32 (exact) for the oracle's shard step,
    which reads bf16 bits or fp32 values."""
    return [oracle.f16_to_f32(c) for c in cc] if gdt == "f16" else cc


# every compiled count with every slice type, and the 16-bit counts 9..15
# (compiled for 16-bit slices only)
ND_GDT = ([(nd, g) for nd in (1, 2, 3, 4, 8, 12, 16) for g in ("bf16", "f32", "f16")] +
          [(9, "bf16"), (10, "f16"), (11, "bf16"), (13, "f16"), (14, "bf16"), (15, "bf16"),
           (11, "f32")])


@pytest.mark.parametrize("shapes", SHAPE_SETS, ids=lambda s: f"{len(s)}params")
@pytest.mark.parametrize("nd,gdt", ND_GDT)
def test_fsdp2_step_without_chunk_cat_matches_oracle(shapes, nd, gdt, path):
    """fsdp2_rs_avg_adamw_cast on every rank, two steps, against the oracle's
    chunk-cat + shard step.  The local state starts non-zero everywhere,
    padding rows included, so that the padding rows' update (AdamW on a
    zero gradient) is checked too."""
    lay = oracle.fsdp2_layout(shapes, nd)
    L = lay.local
    state = []
    for r in range(nd):
        p = synth.host_fill(synth.normal_stream(5, (88, r), 0.02), 0, L, "f32")
        m0 = synth.host_fill(synth.normal_stream(5, (87, r), 1e-4), 0, L, "f32")
        v0 = np.abs(synth.host_fill(synth.normal_stream(5, (86, r), 1e-6), 0, L, "f32"))
        state.append(dict(p=p, m=m0, v=v0, dp=_f32_dev(p), dm=_f32_dev(m0), dv=_f32_dev(v0),
                          out=torch.empty(L, dtype=torch.bfloat16, device=DEV)))
    for t in (1, 2):
        grads_h = [_tensors(shapes, 300 * t + q, gdt) for q in range(nd)]
        grads = [[_dev_grad(x.reshape(-1), gdt).view(x.shape) for x in g] for g in grads_h]
        cc_h = _oracle_contribs([oracle.chunk_cat(g, lay) for g in grads_h], gdt)
        for r, st in enumerate(state):
            ss.fsdp2_rs_avg_adamw_cast(grads, r, st["dp"], st["dm"], st["dv"], st["out"], HPC, t)
            st["p"], st["m"], st["v"], st["ob"] = oracle.fsdp_shard_step(
                cc_h, r, L, st["p"], st["m"], st["v"], HP, t)
        torch.cuda.synchronize()
        for r, st in enumerate(state):
            assert_bits(_host(st["dp"]), st["p"], f"step {t} rank {r} master")
            assert_bits(_host(st["dm"]), st["m"], f"step {t} rank {r} m")
            assert_bits(_host(st["dv"]), st["v"], f"step {t} rank {r} v")
            assert_bits(_host(st["out"]), st["ob"], f"step {t} rank {r} bf16")


@pytest.mark.parametrize("nd", [8, 12])
def test_fsdp2_step_without_chunk_cat_equals_the_chunk_cat_path(nd):
    """On the GPU both compositions give the same bits on one Llama-7B layer
    group at 8 ranks (a rank's 9 parameters, 25.3M local elements) and at
    12 (every parameter with padding rows: 18 segments).  One segment table
    holds them all; at 8 ranks that is the only launch, at 12 the rows that
    start 2 elements off a 16-byte boundary (after a norm vector's
    342-element chunk) take the per-parameter fallback."""
    w = W.llama_7b_rank_view()
    shapes = w.units[0]
    r = 3
    lay = ss.fsdp2_layout(shapes, nd)
    L = lay.local
    grads = [[torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes] for _ in range(nd)]
    for q in range(nd):
        for k, g in enumerate(grads[q]):
            synth.dev_fill(w.grad_stream(1, q, 0, 0, k), g)
    p0 = torch.empty(L, device=DEV)
    synth.dev_fill(synth.normal_stream(7, (85,), 0.02), p0)
    a = [p0.clone(), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV),
         torch.empty(L, dtype=torch.bfloat16, device=DEV)]
    b = [p0.clone(), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV),
         torch.empty(L, dtype=torch.bfloat16, device=DEV)]
    cc = [ss.fsdp2_chunk_cat(grads[q], nd) for q in range(nd)]
    ss.fsdp_rs_avg_adamw_cast([c[r * L:(r + 1) * L] for c in cc], *a, HPC, 1)
    torch.cuda.synchronize()
    before = ss.launch_count()
    ss.fsdp2_rs_avg_adamw_cast(grads, r, *b, HPC, 1)
    torch.cuda.synchronize()
    if nd == 8:
        assert ss.launch_count() - before == 1
    assert ss.last_kernel() == f"rs_adamw_cast_segs<{nd}, bf16> (register-staged, 1 launch)"
    for x, y, name in zip(a, b, ("master", "m", "v", "bf16")):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), name


def test_fsdp2_step_without_chunk_cat_rejects_bad_arguments():
    shapes = [(5, 3), (2,)]
    nd = 2
    L = ss.fsdp2_layout(shapes, nd).local
    grads = [[torch.zeros(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
             for _ in range(nd)]
    st = [torch.zeros(L, device=DEV) for _ in range(3)]
    out = torch.empty(L, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ss.ShardstepError):
        ss.fsdp2_rs_avg_adamw_cast(grads, 2, *st, out, HPC, 1)          # rank out of range
    with pytest.raises(ValueError):
        ss.fsdp2_rs_avg_adamw_cast(grads, 0, *st, out[:-1], HPC, 1)     # wrong local length
    # a gradient that overlaps the local state
    big = torch.zeros(4 * L + 64, device=DEV)
    with pytest.raises(ss.ShardstepError):
        ss.fsdp2_rs_avg_adamw_cast([[big[:15].view(5, 3), torch.zeros(2, device=DEV)]] * nd, 0,
                                   big[:L], big[L:2 * L], big[2 * L:3 * L],
                                   torch.empty(L, dtype=torch.bfloat16, device=DEV), HPC, 1)


def test_fsdp2_step_object_gives_the_same_bits_and_checks_its_buffers():
    """Fsdp2Step (gradient buffers checked once) equals the function form,
    step after step, and still rejects local buffers of the wrong kind."""
    shapes = SHAPE_SETS[2]
    nd = 4
    L = ss.fsdp2_layout(shapes, nd).local
    grads = [[_dev(x.reshape(-1)).view(x.shape) for x in _tensors(shapes, 400 + q, "bf16")]
             for q in range(nd)]
    p0 = _f32_dev(synth.host_fill(synth.normal_stream(9, (84,), 0.02), 0, L, "f32"))
    a = [p0.clone(), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV),
         torch.empty(L, dtype=torch.bfloat16, device=DEV)]
    b = [p0.clone(), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV),
         torch.empty(L, dtype=torch.bfloat16, device=DEV)]
    step = ss.Fsdp2Step(grads)
    assert step.local == L
    for t in (1, 2, 3):
        ss.fsdp2_rs_avg_adamw_cast(grads, 2, *a, HPC, t)
        step(2, *b, HPC, t)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    with pytest.raises(ValueError):
        step(0, b[0][:-1], b[1], b[2], b[3], HPC, 1)
    with pytest.raises(ValueError):
        step(0, b[0], b[1], b[2], b[0], HPC, 1)        # fp32 where bf16 goes
    with pytest.raises(ValueError):
        ss.Fsdp2Step([grads[0], grads[1][:-1]])         # ranks disagree on the parameters
    # a gradient's storage moved by an in-place resize: refused, not read
    g = torch.zeros(shapes[0], dtype=torch.bfloat16, device=DEV)
    moved = ss.Fsdp2Step([[g] + grads[q][1:] for q in range(nd)])
    g.resize_(4096, 4096)
    with pytest.raises(ValueError):
        moved(0, *b, HPC, 1)


@pytest.mark.parametrize("nd", [3, 8])
def test_fsdp2_step_replayed_from_a_cuda_graph(nd):
    """The whole FSDP2 step -- the step count advanced on the device, every
    rank's step read straight from the gradients, the copy-out -- captured
    once and replayed three times gives the bits of three host-scalar steps
    (steps 1, 2, 3), padding rows included."""
    shapes = SHAPE_SETS[4]                     # uneven dim 0: padding rows
    L = ss.fsdp2_layout(shapes, nd).local
    grads = [[_dev(x.reshape(-1)).view(x.shape) for x in _tensors(shapes, 500 + q, "bf16")]
             for q in range(nd)]
    step = ss.Fsdp2Step(grads)

    def fresh():
        bufs = []
        for r in range(nd):
            p = _f32_dev(synth.host_fill(synth.normal_stream(9, (83, r), 0.02), 0, L, "f32"))
            bufs.append([p, torch.zeros(L, device=DEV), torch.zeros(L, device=DEV),
                         torch.empty(L, dtype=torch.bfloat16, device=DEV)])
        return bufs

    a, b = fresh(), fresh()
    pa = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    pb = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    for t in (1, 2, 3):
        for r in range(nd):
            step(r, *a[r], HPC, t)
        ss.fsdp2_all_gather_copy_out([x[3] for x in a], pa)
    state = ss.AdamWState(HPC, 0, device=DEV)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        state.advance()
        for r in range(nd):
            step.step_state(r, *b[r], state)
        ss.fsdp2_all_gather_copy_out([x[3] for x in b], pb)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert state.step() == 3
    for r in range(nd):
        for x, y in zip(a[r], b[r]):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), r
    for x, y in zip(pa, pb):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("nd", [33, 64])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_fsdp2_step_without_chunk_cat_at_large_nd(nd, gdt):
    """Past the compiled counts (the kernel's loop over batches of slices) and
    with the 128-pointer table holding only 3 or 2 segments (a rank's
    segments split over several launches), against the oracle."""
    shapes = SHAPE_SETS[3]                     # 12 parameters: 24 segments at most
    lay = oracle.fsdp2_layout(shapes, nd)
    L = lay.local
    grads_h = [_tensors(shapes, 600 + q, gdt) for q in range(nd)]
    grads = [[_dev(x.reshape(-1)).view(x.shape) for x in g] for g in grads_h]
    cc_h = [oracle.chunk_cat(g, lay) for g in grads_h]
    step = ss.Fsdp2Step(grads)
    for r in (0, 1, nd // 2, nd - 1):
        p = synth.host_fill(synth.normal_stream(9, (82, r), 0.02), 0, L, "f32")
        dp, dm, dv = _f32_dev(p), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV)
        out = torch.empty(L, dtype=torch.bfloat16, device=DEV)
        before = ss.launch_count()
        step(r, dp, dm, dv, out, HPC, 1)
        torch.cuda.synchronize()
        assert ss.launch_count() - before >= 2      # the table filled at least once
        z = np.zeros(L, np.float32)
        p1, m1, v1, o1 = oracle.fsdp_shard_step(cc_h, r, L, p, z, z, HP, 1)
        assert_bits(_host(dp), p1, f"rank {r} master")
        assert_bits(_host(dm), m1, f"rank {r} m")
        assert_bits(_host(dv), v1, f"rank {r} v")
        assert_bits(_host(out), o1, f"rank {r} bf16")


def test_fsdp2_rank_optimizer_steps_and_gathers_like_the_oracle():
    """Fsdp2RankOptimizer: every rank's local state, two host-scalar steps and
    a third on the device step state, then the gather into the full
    parameters, against the oracle; the local views have DTensor's local
    shapes."""
    from sharded_optimizer_step_gb300.engine import Fsdp2RankOptimizer
    shapes, nd = SHAPE_SETS[2], 4
    lay = oracle.fsdp2_layout(shapes, nd)
    masters = [synth.host_fill(synth.normal_stream(11, (81, t), 0.02), 0, int(np.prod(s)),
                               "f32").reshape(s) for t, s in enumerate(shapes)]
    grads_h = [_tensors(shapes, 700 + q, "bf16") for q in range(nd)]
    grads = [[_dev(x.reshape(-1)).view(x.shape) for x in g] for g in grads_h]
    opts = [Fsdp2RankOptimizer(grads, r, HPC, device=DEV) for r in range(nd)]
    want = []
    for r, o in enumerate(opts):
        p = oracle.local_buffer(masters, lay, r)
        o.master.copy_(_f32_dev(p))
        views = o.local_views(o.master)
        assert [tuple(x.shape) for x in views] == \
            [tuple(x.shape) for x in oracle.local_shards(masters, lay, r)]
        want.append([p, np.zeros(lay.local, np.float32), np.zeros(lay.local, np.float32), None])
    cc = [oracle.chunk_cat(g, lay) for g in grads_h]
    for t in (1, 2, 3):
        for r, o in enumerate(opts):
            if t < 3:
                o.step()
            else:
                o.device_step_state()
                o.step_on_device()
            want[r][0], want[r][1], want[r][2], want[r][3] = oracle.fsdp_shard_step(
                cc, r, lay.local, want[r][0], want[r][1], want[r][2], HP, t)
    params = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    opts[0].gather([o.params for o in opts], params)
    torch.cuda.synchronize()
    for r, o in enumerate(opts):
        assert o.state.step() == 3
        assert_bits(_host(o.master), want[r][0], f"rank {r} master")
        assert_bits(_host(o.params), want[r][3], f"rank {r} bf16")
    for got, w in zip(params, oracle.all_gather_copy_out([x[3] for x in want], lay)):
        assert_bits(_host(got).reshape(-1), w.reshape(-1), "gathered parameter")
