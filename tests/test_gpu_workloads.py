"""GPU parity on the model-shaped workloads at full size.

The 9.4M-parameter unit (N_d = 4, M = 4) is compared element by element with
the oracle.  The larger workloads run in full on the GPU and are checked on
sampled outputs that the oracle computes one by one from the same seeded
inputs (every step, every micro-batch, every rank), plus properties that hold
at any size.  The two sides lay the FlatParameters out independently: the
GPU side packs each unit from its per-tensor inputs with ``fsdp_flat_pack``,
takes the shards from ``fsdp_layout``, fills a rank's buffers at the places
``fsdp_shard_pieces`` gives and reads the gathered tensors through
``fsdp_views``; the oracle traces every sampled position back to its tensor
element with its own layout.  GPT-2 small also runs at N_d = 7, where every
unit is padded.  The Llama-7B rank view runs in the launch configuration the
benchmark times: one fused launch over the rank's 842,301,952-element shard
and one all-gather of a 202,383,360-parameter layer unit; so does the
Llama-1B accumulation view (three accumulate launches over the 8
contributions, the fourth micro-batch inside one fused launch)."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from sharded_optimizer_step_gb300.engine import RankShardOptimizer
from synth import workloads as W
from tests._cmp import assert_bf16, assert_bits, assert_f32
from tests._views import gpu_fill_rank, oracle_rank_total, oracle_rank_values

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    torch.cuda.empty_cache()


def _hp(w):
    return (AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay),
            ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay))


def _host_bf16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _sample(n, k, rng, extra=()):
    idx = set(int(i) for i in rng.integers(0, n, size=min(k, n)))
    idx.update(i for i in range(min(n, 16)))
    idx.update(i for i in range(max(0, n - 16), n))
    idx.update(int(i) for i in extra if 0 <= i < n)
    return np.array(sorted(idx), dtype=np.int64)


def _gpu_pack(tensors, streams, nd, flat):
    """Fill each device tensor of a unit from its stream and pack them with
    the library into ``flat`` (its padding zeroed by the pack)."""
    for x, st in zip(tensors, streams):
        synth.dev_fill(st, x.view(-1))
    ss.fsdp_flat_pack(tensors, nd, flat=flat)


# --------------------------------------------------- 9.4M unit, every element

def test_unit_9m_every_element():
    w = W.unit_9m()
    hp, hpc = _hp(w)
    nd, M = w.nd, w.micro
    shapes = w.units[0]
    numels = w.unit_numels(0)
    # master weights: the unit's tensors packed into the fp32 FlatParameter
    host_t = [synth.host_fill(w.master_stream(0, t), 0, n, "f32").reshape(s)
              for t, (n, s) in enumerate(zip(numels, shapes))]
    dev_t = [torch.from_numpy(h).to(DEV) for h in host_t]
    flat = ss.fsdp_flat_pack(dev_t, nd)
    want_flat, lay = oracle.flat_pack(host_t, nd)
    S, P = lay.shard, lay.padded
    torch.cuda.synchronize()
    assert_bits(flat.cpu().numpy(), want_flat, "packed master")

    accs, accs_h = [], []
    g = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    gt = [torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes]
    for q in range(nd):
        acc = torch.empty(P, dtype=torch.float32, device=DEV)
        micro_h = []
        for j in range(M):
            streams = [w.grad_stream(1, q, j, 0, t) for t in range(len(shapes))]
            _gpu_pack(gt, streams, nd, g)
            micro_h.append(oracle.flat_pack(
                [synth.host_fill(st, 0, n, "bf16") for st, n in zip(streams, numels)], nd)[0])
            ss.fsdp_grad_accumulate(g, acc, float(np.float32(1.0 / M)), j == 0)
        torch.cuda.synchronize()
        assert_bits(_host_bf16(g), micro_h[-1], "packed gradient")
        accs.append(acc)
        accs_h.append(oracle.grad_accumulate(micro_h, np.float32(1.0 / M)))
        assert_bits(acc.cpu().numpy(), accs_h[-1], f"accumulator rank {q}")

    shards = []
    for r in range(nd):
        master = flat[r * S:(r + 1) * S].clone()
        m = torch.zeros(S, device=DEV)
        v = torch.zeros(S, device=DEV)
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        ss.fsdp_rs_avg_adamw_cast([a[r * S:(r + 1) * S] for a in accs], master, m, v, out, hpc, 1)
        z = np.zeros(S, np.float32)
        p1, m1, v1, o1 = oracle.fsdp_shard_step(accs_h, r, S, want_flat[r * S:(r + 1) * S], z, z,
                                                hp, 1)
        torch.cuda.synchronize()
        for name, got, want in (("master", master, p1), ("m", m, m1), ("v", v, v1)):
            gh = got.cpu().numpy()
            assert_f32(gh, want, f"{name} rank {r}")
            assert_bits(gh, want, f"{name} rank {r}")
        assert_bf16(_host_bf16(out), o1, f"bf16 rank {r}")
        assert_bits(_host_bf16(out), o1, f"bf16 rank {r}")
        shards.append((out, o1))

    full = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_ag_unpack([s for s, _ in shards], full)
    want_full, want_views = oracle.ag_unpack([o for _, o in shards], lay, shapes)
    views = ss.fsdp_views(full, shapes, nd)
    torch.cuda.synchronize()
    assert_bits(_host_bf16(full), want_full, "gathered unit")
    for v, wv in zip(views, want_views):
        assert tuple(v.shape) == wv.shape
        assert_bits(_host_bf16(v), wv, "view")


# ------------------------------------- per-unit emulation of all N_d ranks

def _run_all_ranks(w, sample_per_unit=1024, seed=0):
    """Every rank of every unit, all steps; oracle on sampled shard positions
    (the last ones of every shard among them, so the padding of a padded
    unit is sampled).  Each unit's inputs are packed on the GPU from its
    per-tensor fills by the library; the fused outputs land in per-rank
    shard buffers that the all-gather copies into the unit's full flat
    buffer, whose tensor views are compared with the oracle."""
    hp, hpc = _hp(w)
    nd, M = w.nd, w.micro
    rng = np.random.default_rng(seed)
    glays = [ss.fsdp_layout(w.unit_numels(u), nd) for u in range(len(w.units))]
    olays = [oracle.layout(w.unit_numels(u), nd) for u in range(len(w.units))]
    maxP = max(g.padded for g in glays)
    g = torch.empty(maxP, dtype=torch.bfloat16, device=DEV)
    acc = [torch.empty(maxP, dtype=torch.float32 if M > 1 else torch.bfloat16, device=DEV)
           for _ in range(nd)]
    state = []
    for u, shapes in enumerate(w.units):
        glay, olay = glays[u], olays[u]
        assert (glay.shard, glay.padded, glay.total) == (olay.shard, olay.padded, olay.total)
        S, P = glay.shard, glay.padded
        master = torch.empty(P, dtype=torch.float32, device=DEV)
        mt = [torch.empty(s, dtype=torch.float32, device=DEV) for s in shapes]
        _gpu_pack(mt, [w.master_stream(u, t) for t in range(len(shapes))], nd, master)
        del mt
        ranks = []
        for r in range(nd):
            idx = _sample(S, sample_per_unit, rng)
            tt, kk = oracle.element_source(olay, r * olay.shard + idx)
            p0 = synth.host_gather_sources(np.full(idx.size, u), tt, kk,
                                           lambda uu, t: w.master_stream(uu, t), "f32")
            ranks.append(dict(master=master[r * S:(r + 1) * S], m=torch.zeros(S, device=DEV),
                              v=torch.zeros(S, device=DEV),
                              out=torch.empty(S, dtype=torch.bfloat16, device=DEV),
                              idx=idx, tt=tt, kk=kk, p=p0, mm=np.zeros(idx.size, np.float32),
                              vv=np.zeros(idx.size, np.float32), ob=None))
        state.append(dict(S=S, P=P, ranks=ranks,
                          gt=[torch.empty(s, dtype=torch.bfloat16, device=DEV) for s in shapes],
                          full=torch.empty(P, dtype=torch.bfloat16, device=DEV)))

    for t in range(1, w.steps + 1):
        for u, us in enumerate(state):
            S, P = us["S"], us["P"]
            nt = len(w.units[u])
            for q in range(nd):
                for j in range(M):
                    dst = (g if M > 1 else acc[q])[:P]
                    _gpu_pack(us["gt"], [w.grad_stream(t, q, j, u, k) for k in range(nt)], nd,
                              dst)
                    if M > 1:
                        ss.fsdp_grad_accumulate(dst, acc[q][:P], float(np.float32(1.0 / M)),
                                                j == 0)
            for r, rs in enumerate(us["ranks"]):
                ss.fsdp_rs_avg_adamw_cast([a[r * S:(r + 1) * S] for a in acc], rs["master"],
                                          rs["m"], rs["v"], rs["out"], hpc, t)
            ss.fsdp_ag_unpack([rs["out"] for rs in us["ranks"]], us["full"])
            # oracle on the sampled positions of every rank
            for r, rs in enumerate(us["ranks"]):
                uu = np.full(rs["idx"].size, u)
                contribs = []
                for q in range(nd):
                    micro = [synth.host_gather_sources(
                        uu, rs["tt"], rs["kk"],
                        lambda a, b, q=q, j=j: w.grad_stream(t, q, j, a, b), "bf16")
                        for j in range(M)]
                    contribs.append(oracle.grad_accumulate(micro, np.float32(1.0 / M))
                                    if M > 1 else micro[0])
                rs["p"], rs["mm"], rs["vv"], rs["ob"] = oracle.fsdp_shard_step(
                    contribs, 0, rs["idx"].size, rs["p"], rs["mm"], rs["vv"], hp, t)
    torch.cuda.synchronize()
    for u, us in enumerate(state):
        shapes = w.units[u]
        views = ss.fsdp_views(us["full"], shapes, nd)
        assert [tuple(x.shape) for x in views] == [tuple(s) for s in shapes]
        for r, rs in enumerate(us["ranks"]):
            it = torch.from_numpy(rs["idx"]).to(DEV)
            assert_f32(rs["master"][it].cpu().numpy(), rs["p"], f"unit {u} rank {r} master")
            assert_bits(rs["master"][it].cpu().numpy(), rs["p"], f"unit {u} rank {r} master")
            assert_bits(rs["m"][it].cpu().numpy(), rs["mm"], f"unit {u} rank {r} m")
            assert_bits(rs["v"][it].cpu().numpy(), rs["vv"], f"unit {u} rank {r} v")
            assert_bits(_host_bf16(rs["out"][it]), rs["ob"], f"unit {u} rank {r} bf16")
            # the gathered tensors: each sampled element, found through the
            # library's views, is the oracle's value of the tensor element
            # the oracle's layout puts there
            for k in np.unique(rs["tt"][rs["tt"] >= 0]):
                sel = np.nonzero(rs["tt"] == k)[0]
                got = _host_bf16(views[k].reshape(-1)[torch.from_numpy(rs["kk"][sel]).to(DEV)])
                assert_bits(got, rs["ob"][sel], f"unit {u} rank {r} view {k}")
            pad = np.nonzero(rs["tt"] < 0)[0]
            assert not rs["ob"][pad].any() and not rs["p"][pad].any()
        T = sum(w.unit_numels(u))
        assert not us["full"][T:].view(torch.int16).any(), f"unit {u}: padding not zero"


def test_gpt2_small_all_units_all_ranks():
    _run_all_ranks(W.gpt2_small(), sample_per_unit=512)


def test_gpt2_small_nd7_every_unit_padded():
    w = W.gpt2_small_nd7()
    pads = [ss.fsdp_layout(w.unit_numels(u), w.nd) for u in range(len(w.units))]
    assert [p.padded - p.total for p in pads] == [6] * 12 + [2]
    _run_all_ranks(w, sample_per_unit=512)


def test_llama_1b_all_units_all_ranks_with_accumulation_and_outliers():
    _run_all_ranks(W.llama_1b(), sample_per_unit=256)


# ------------------------------------------ Llama-7B rank view (bench launch)

def test_llama_7b_rank_view_as_benchmarked():
    w = W.llama_7b_rank_view()
    hp, hpc = _hp(w)
    r = w.extra["rank"]
    opt = RankShardOptimizer(w.units, w.nd, r, hpc, device=DEV)
    assert opt.shard_total == 842_301_952 == oracle_rank_total(w)
    gpu_fill_rank(opt, opt.master, w.master_stream)
    rng = np.random.default_rng(7)
    bounds = opt.starts[1:] + [s - 1 for s in opt.starts[1:]]
    idx = _sample(opt.shard_total, 200_000, rng, extra=bounds)
    p = oracle_rank_values(w, r, idx, w.master_stream, "f32")
    m = np.zeros(idx.size, np.float32)
    v = np.zeros(idx.size, np.float32)
    for t in range(1, w.steps + 1):
        for q in range(w.nd):
            gpu_fill_rank(opt, opt.grad_in[q], lambda u, k, q=q: w.grad_stream(t, q, 0, u, k))
        launches = ss.launch_count()
        opt.step()
        assert ss.launch_count() - launches == 1      # one fused launch over the shard
        contribs = [oracle_rank_values(w, r, idx, lambda u, k, q=q: w.grad_stream(t, q, 0, u, k),
                                       "bf16") for q in range(w.nd)]
        p, m, v, ob = oracle.fsdp_shard_step(contribs, 0, idx.size, p, m, v, hp, t)
    torch.cuda.synchronize()
    it = torch.from_numpy(idx).to(DEV)
    assert_f32(opt.master[it].cpu().numpy(), p, "master")
    assert_bits(opt.master[it].cpu().numpy(), p, "master")
    assert_bits(opt.m[it].cpu().numpy(), m, "m")
    assert_bits(opt.v[it].cpu().numpy(), v, "v")
    assert_bits(_host_bf16(opt.params[it]), ob, "bf16")

    # all-gather of one layer unit: the other ranks' shards are seeded inputs
    u = w.extra["ag_unit"]
    S, P = opt.layouts[u].shard, opt.layouts[u].padded
    assert P == 202_383_360
    peers = []
    for q in range(w.nd):
        s = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        if q != r:
            synth.dev_fill(w.peer_shard_stream(w.steps, q, u), s)
        peers.append(s)
    full = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    views = opt.gather_unit(u, peers, full)
    torch.cuda.synchronize()
    assert [tuple(x.shape) for x in views] == [tuple(s) for s in w.units[u]]
    for q in range(w.nd):
        src = opt.unit_slice(opt.params, u) if q == r else peers[q]
        assert torch.equal(full[q * S:(q + 1) * S].view(torch.int16), src.view(torch.int16))
    loc = _sample(S, 4096, rng)
    for q in range(w.nd):
        if q == r:
            continue
        want = synth.host_gather(w.peer_shard_stream(w.steps, q, u), loc, "bf16")
        assert_bits(_host_bf16(full[q * S + torch.from_numpy(loc).to(DEV)]), want, "peer shard")


def test_llama_1b_rank_view_accumulation_as_benchmarked():
    """The accumulation line's launches: per step M - 1 accumulate launches
    over the 8 contributions side by side, then the last micro-batch inside
    the fused step (one launch over the whole 150,610,176-element shard);
    the oracle accumulates all M micro-batches and steps, on sampled shard
    positions, and the accumulators still hold micro-batches 0..M-2."""
    w = W.llama_1b()
    hp, hpc = _hp(w)
    nd, M, r = w.nd, w.micro, 0
    opt = RankShardOptimizer(w.units, nd, r, hpc, device=DEV, grad_dtype=torch.float32)
    S = opt.shard_total
    assert S == 150_610_176 and M == 4
    acc = torch.empty(nd * S, dtype=torch.float32, device=DEV)
    opt.grad_in = [acc[q * S:(q + 1) * S] for q in range(nd)]
    micro = [torch.empty(nd * S, dtype=torch.bfloat16, device=DEV) for _ in range(M)]
    last = [micro[M - 1][q * S:(q + 1) * S] for q in range(nd)]
    gpu_fill_rank(opt, opt.master, w.master_stream)
    rng = np.random.default_rng(11)
    assert oracle_rank_total(w) == S
    bounds = opt.starts[1:] + [s - 1 for s in opt.starts[1:]]
    idx = _sample(S, 100_000, rng, extra=bounds)
    p = oracle_rank_values(w, r, idx, w.master_stream, "f32")
    m = np.zeros(idx.size, np.float32)
    v = np.zeros(idx.size, np.float32)
    inv_m = np.float32(1.0 / M)
    for t in range(1, 4):
        for j in range(M):
            for q in range(nd):
                gpu_fill_rank(opt, micro[j][q * S:(q + 1) * S],
                              lambda u, k, q=q, j=j: w.grad_stream(t, q, j, u, k))
        launches = ss.launch_count()
        for j in range(M - 1):
            ss.fsdp_grad_accumulate(micro[j], acc, float(inv_m), j == 0)
        opt.step_with_last_micro_batch(last, float(inv_m))
        assert ss.launch_count() - launches == M
        assert ss.last_kernel() == "accum_rs_adamw_cast_vec4<8> (register-staged)"
        grads = [[oracle_rank_values(w, r, idx,
                                     lambda u, k, q=q, j=j: w.grad_stream(t, q, j, u, k), "bf16")
                  for j in range(M)] for q in range(nd)]
        contribs = [oracle.grad_accumulate(grads[q], inv_m) for q in range(nd)]
        p, m, v, ob = oracle.fsdp_shard_step(contribs, 0, idx.size, p, m, v, hp, t)
    torch.cuda.synchronize()
    it = torch.from_numpy(idx).to(DEV)
    assert_f32(opt.master[it].cpu().numpy(), p, "master")
    assert_bits(opt.master[it].cpu().numpy(), p, "master")
    assert_bits(opt.m[it].cpu().numpy(), m, "m")
    assert_bits(opt.v[it].cpu().numpy(), v, "v")
    assert_bits(_host_bf16(opt.params[it]), ob, "bf16")
    for q in (0, nd - 1):
        assert_bits(opt.grad_in[q][it].cpu().numpy(),
                    oracle.grad_accumulate(grads[q][:M - 1], inv_m), f"accumulator {q}")


def test_llama_7b_rank_view_every_kernel_and_the_graph_agree_everywhere():
    """The register-staged kernel (the default, checked against the oracle
    on samples above), the TMA-staged kernel and the device-state step
    replayed from a CUDA graph give the same bits on every one of the 842M
    shard elements over two steps."""
    w = W.llama_7b_rank_view()
    _, hpc = _hp(w)
    r = w.extra["rank"]
    a = RankShardOptimizer(w.units, w.nd, r, hpc, device=DEV)
    b = RankShardOptimizer(w.units, w.nd, r, hpc, device=DEV)
    c = RankShardOptimizer(w.units, w.nd, r, hpc, device=DEV)
    b.grad_in = a.grad_in                 # one set of gradient buffers for all
    c.grad_in = a.grad_in
    gpu_fill_rank(a, a.master, w.master_stream)
    b.master.copy_(a.master)
    c.master.copy_(a.master)
    c.device_step_state()
    prev = ss.set_fused_path("auto")
    try:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):     # warm-up outside the capture, then undone
            c.step_on_device()
        torch.cuda.current_stream().wait_stream(side)
        c.master.copy_(a.master)
        c.m.zero_()
        c.v.zero_()
        c.state.init(0)
        with torch.cuda.graph(graph):
            c.step_on_device()
        for t in (1, 2):
            for q in range(w.nd):
                gpu_fill_rank(a, a.grad_in[q], lambda u, k, q=q: w.grad_stream(t, q, 0, u, k))
            ss.set_fused_path("auto")
            a.step()
            ss.set_fused_path("tma")
            b.step()
            graph.replay()
    finally:
        ss.set_fused_path(prev)
    torch.cuda.synchronize()
    assert c.state.step() == 2
    for other in (b, c):
        for name in ("master", "m", "v"):
            assert torch.equal(getattr(a, name).view(torch.int32),
                               getattr(other, name).view(torch.int32)), name
        assert torch.equal(a.params.view(torch.int16), other.params.view(torch.int16))
    assert ss.device_status() == 0


def test_llama_7b_hybrid_view_as_benchmarked():
    # N_d = 16 ranks in two groups of F = 8: rank (g=0, f=0)'s shard of every
    # unit, with all 16 contributions, one fused launch
    w = W.llama_7b_hybrid_view()
    hp, hpc = _hp(w)
    f = w.extra["rank"]
    opt = RankShardOptimizer(w.units, w.nd, f, hpc, device=DEV, shard_group=w.F)
    assert opt.shard_total == 842_301_952
    assert opt.shard_total == oracle_rank_total(w)
    gpu_fill_rank(opt, opt.master, w.master_stream)
    rng = np.random.default_rng(11)
    idx = _sample(opt.shard_total, 100_000, rng, extra=opt.starts)
    p = oracle_rank_values(w, f, idx, w.master_stream, "f32")
    m = np.zeros(idx.size, np.float32)
    v = np.zeros(idx.size, np.float32)
    for t in (1, 2):
        for k in range(w.nd):
            gpu_fill_rank(opt, opt.grad_in[k], lambda u, x, k=k: w.grad_stream(t, k, 0, u, x))
        launches = ss.launch_count()
        opt.step()
        assert ss.launch_count() - launches == 1
        contribs = [oracle_rank_values(w, f, idx, lambda u, x, k=k: w.grad_stream(t, k, 0, u, x),
                                       "bf16") for k in range(w.nd)]
        p, m, v, ob = oracle.hybrid_shard_step(contribs, w.F, 0, idx.size, p, m, v, hp, t)
    torch.cuda.synchronize()
    it = torch.from_numpy(idx).to(DEV)
    assert_bits(opt.master[it].cpu().numpy(), p, "master")
    assert_bits(opt.m[it].cpu().numpy(), m, "m")
    assert_bits(opt.v[it].cpu().numpy(), v, "v")
    assert_bits(_host_bf16(opt.params[it]), ob, "bf16")
    # all-gather inside the group of 8
    u = w.extra["ag_unit"]
    S, P = opt.layouts[u].shard, opt.layouts[u].padded
    peers = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(w.F)]
    for q in range(1, w.F):
        synth.dev_fill(w.peer_shard_stream(2, q, u), peers[q])
    full = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    views = opt.gather_unit(u, peers, full)
    torch.cuda.synchronize()
    assert [tuple(x.shape) for x in views] == [tuple(s) for s in w.units[u]]
    assert torch.equal(full[:S].view(torch.int16), opt.unit_slice(opt.params, u).view(torch.int16))
    for q in range(1, w.F):
        assert torch.equal(full[q * S:(q + 1) * S].view(torch.int16), peers[q].view(torch.int16))


# ------------------------------------------------------- DDP bucket sweep

def test_ddp_bucket_sweep_full_size():
    w = W.ddp_sweep()
    hp, hpc = _hp(w)
    nd = w.nd
    numels = w.unit_numels(0)
    total = sum(numels)
    rng = np.random.default_rng(3)
    grads = [torch.empty(total, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    outs = {}
    for mib in w.extra["caps_mib"]:
        off, of, boff = ss.ddp_bucket_plan(numels, 2, mib << 20)
        assert (off, of, boff) == tuple(list(x) for x in oracle.bucket_plan(numels, 2, mib << 20))
        # rank q's gradient of parameter i is seeded per parameter, so the
        # values do not depend on where the plan puts the parameter
        for q in range(nd):
            for i, n in enumerate(numels):
                synth.dev_fill(w.grad_stream(1, q, 0, 0, i), grads[q][off[i]:off[i] + n])
        out = torch.empty(total, dtype=torch.bfloat16, device=DEV)
        before = ss.launch_count()
        ss.ddp_bucket_allreduce_avg(grads, boff, out)
        assert ss.launch_count() - before == len(boff) - 1
        # back to registration order for the comparison across caps
        outs[mib] = torch.cat([out[off[i]:off[i] + n] for i, n in enumerate(numels)])
        # oracle on sampled elements of sampled parameters
        for i in rng.choice(len(numels), size=12, replace=False):
            loc = _sample(numels[i], 512, rng)
            gq = [synth.host_gather(w.grad_stream(1, q, 0, 0, int(i)), loc, "bf16")
                  for q in range(nd)]
            want = oracle.bucket_allreduce_avg(gq, [0, loc.size])
            got = _host_bf16(out[off[i] + torch.from_numpy(loc).to(DEV)])
            assert_bits(got, want, f"cap {mib} MiB param {i}")
    ref = outs[25]
    for mib, o in outs.items():
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), mib
    # replicated AdamW over every parameter (registration order, the library's
    # unsharded layout) with the averaged gradient
    glay = ss.fsdp_layout(numels, 1)
    master = torch.empty(total, dtype=torch.float32, device=DEV)
    for i, n in enumerate(numels):
        synth.dev_fill(w.master_stream(0, i), master[glay.offsets[i]:glay.offsets[i] + n])
    mm = torch.zeros(total, device=DEV)
    vv = torch.zeros(total, device=DEV)
    pb = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_rs_avg_adamw_cast([ref], master, mm, vv, pb, hpc, 1)
    # the oracle from the seeded inputs alone: each sampled position traced to
    # its parameter element by the oracle's layout
    loc = _sample(total, 100_000, rng)
    it = torch.from_numpy(loc).to(DEV)
    tt, kk = oracle.element_source(oracle.layout(numels, 1), loc)
    uu = np.zeros(loc.size, np.int64)
    p0 = synth.host_gather_sources(uu, tt, kk, w.master_stream, "f32")
    gq = [synth.host_gather_sources(uu, tt, kk, lambda u, i, q=q: w.grad_stream(1, q, 0, u, i),
                                    "bf16") for q in range(nd)]
    z = np.zeros(loc.size, np.float32)
    avg, p1, m1, v1, pb1 = oracle.ddp_step(gq, [0, loc.size], p0, z, z, hp, 1)
    torch.cuda.synchronize()
    assert_bits(_host_bf16(ref[it]), avg, "averaged gradient")
    assert_bits(master[it].cpu().numpy(), p1, "master")
    assert_bits(mm[it].cpu().numpy(), m1, "m")
    assert_bits(vv[it].cpu().numpy(), v1, "v")
    assert_bits(_host_bf16(pb[it]), pb1, "params")
