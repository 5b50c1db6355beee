"""GPU parity of fsdp_accumulate_rs_avg_adamw_cast: the last micro-batch's
accumulation fused into the sharded step.  The expected values are the
oracle's accumulation over all M micro-batches followed by its shard step;
the accumulators must still hold micro-batches 0..M-2 afterwards."""
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


def dev(x, shift=0):
    """numpy (bf16 bits as uint16, or fp32) -> CUDA tensor starting `shift`
    elements into its allocation."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        buf = torch.empty(x.size + shift + 8, dtype=torch.bfloat16, device=DEV)
        t = buf[shift:shift + x.size]
        t.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))
    else:
        buf = torch.empty(x.size + shift + 8, dtype=torch.float32, device=DEV)
        t = buf[shift:shift + x.size]
        t.copy_(torch.from_numpy(x.astype(np.float32)))
    return t


def host(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def _micro(seed, nd, M, S):
    """micro[q][j]: rank q's bf16 gradient slice of micro-batch j."""
    return [[synth.host_fill(synth.normal_stream(seed, (91, q, j), 1e-3), 0, S, "bf16")
             for j in range(M)] for q in range(nd)]


def _state(seed, S):
    p = synth.host_fill(synth.normal_stream(seed, (91, 100), 0.02), 0, S, "f32")
    m = synth.host_fill(synth.normal_stream(seed, (91, 101), 1e-4), 0, S, "f32")
    v = np.abs(synth.host_fill(synth.normal_stream(seed, (91, 102), 1e-7), 0, S, "f32"))
    return p, m, v


def _check(nd, S, M, step, shift, F=None):
    seed = 31 * nd + S + M + (F or 0)
    micro = _micro(seed, nd, M, S)
    scale = np.float32(1.0 / M)
    p, m, v = _state(seed, S)
    dp, dm, dv = dev(p, shift), dev(m, shift), dev(v, shift)
    out = torch.empty(S + 1, dtype=torch.bfloat16, device=DEV)[shift:shift + S]
    accs = []
    for q in range(nd):
        acc = dev(np.zeros(S, np.float32), shift if q % 2 else 0)
        for j in range(M - 1):
            ss.fsdp_grad_accumulate(dev(micro[q][j]), acc, float(scale), j == 0)
        accs.append(acc)
    last = [dev(micro[q][M - 1], shift if q % 3 == 1 else 0) for q in range(nd)]
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, float(scale), dp, dm, dv, out, HPC, step,
                                         shard_group=F)
    contribs = [oracle.grad_accumulate(micro[q], scale) for q in range(nd)]
    if F is None or F == nd:
        wp, wm, wv, wo = oracle.fsdp_shard_step(contribs, 0, S, p, m, v, HP, step)
    else:
        wp, wm, wv, wo = oracle.hybrid_shard_step(contribs, F, 0, S, p, m, v, HP, step)
    torch.cuda.synchronize()
    for name, got, want in (("master", host(dp), wp), ("m", host(dm), wm), ("v", host(dv), wv)):
        assert_f32(got, want, name)
        assert_bits(got, want, name)
    assert_bf16(host(out), wo, "bf16")
    assert_bits(host(out), wo, "bf16")
    for q in range(nd):  # the accumulators are read, not written
        assert_bits(host(accs[q]), oracle.grad_accumulate(micro[q][:M - 1], scale), "acc")


@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 6, 7, 8, 9, 16])
@pytest.mark.parametrize("S", [1, 13, 4099])
@pytest.mark.parametrize("shift", [0, 1])
def test_accumulate_step_matches_oracle(nd, S, shift):
    _check(nd, S, M=3, step=1 + nd % 3, shift=shift)


@pytest.mark.parametrize("nd,F", [(16, 8), (8, 4), (6, 3), (8, 2), (4, 1), (9, 3)])
@pytest.mark.parametrize("S", [13, 4099, 70001])
@pytest.mark.parametrize("shift", [0, 1])
def test_hybrid_accumulate_step_matches_oracle(nd, F, S, shift):
    """Hybrid sharding (sharding factor F): the contributions summed inside
    each group of F ranks, then across the groups, as the hybrid step does;
    with shift = 1 the slices are misaligned and the one-element kernel runs
    the grouped sum."""
    _check(nd, S, M=3, step=2, shift=shift, F=F)


@pytest.mark.parametrize("nd,F,rank", [(8, 4, 3), (9, 3, 2), (16, 8, 7)])
def test_engine_hybrid_last_micro_batch_in_a_cuda_graph(nd, F, rank):
    """RankShardOptimizer with sharding factor F < N_d and a rank other than
    0: step_with_last_micro_batch (host scalars) and its device-state form
    captured once in a CUDA graph and replayed, over three steps of a small
    model, against the oracle's accumulation and hybrid shard step."""
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    units = [[(37, 29), (29,), (301,)], [(64, 64), (5,)]]
    M, steps = 3, 3
    a = RankShardOptimizer(units, nd, rank, HPC, device=DEV, grad_dtype=torch.float32,
                           shard_group=F)
    b = RankShardOptimizer(units, nd, rank, HPC, device=DEV, grad_dtype=torch.float32,
                           shard_group=F)
    S = a.shard_total
    seed = 7 * nd + F + rank
    p, _, _ = _state(seed, S)
    a.master.copy_(torch.from_numpy(p))
    b.master.copy_(torch.from_numpy(p))
    last = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    scale = np.float32(1.0 / M)
    b.device_step_state()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # a warm-up outside the capture, then undone
        b.step_with_last_micro_batch_on_device(last, float(scale))
    torch.cuda.current_stream().wait_stream(side)
    b.master.copy_(torch.from_numpy(p))
    b.m.zero_()
    b.v.zero_()
    b.state.init(0)
    with torch.cuda.graph(graph):
        b.step_with_last_micro_batch_on_device(last, float(scale))
    wp, wm, wv = p, np.zeros(S, np.float32), np.zeros(S, np.float32)
    for t in range(1, steps + 1):
        micro = _micro(seed + t, nd, M, S)
        for q in range(nd):
            for j in range(M - 1):
                ss.fsdp_grad_accumulate(dev(micro[q][j]), a.grad_in[q], float(scale), j == 0)
            b.grad_in[q].copy_(a.grad_in[q])
            last[q].copy_(dev(micro[q][M - 1]))
        a.step_with_last_micro_batch(last, float(scale))
        graph.replay()
        contribs = [oracle.grad_accumulate(micro[q], scale) for q in range(nd)]
        wp, wm, wv, wo = oracle.hybrid_shard_step(contribs, F, 0, S, wp, wm, wv, HP, t)
    torch.cuda.synchronize()
    assert b.state.step() == steps and a.t == steps
    for o in (a, b):
        assert_bits(host(o.master), wp, "master")
        assert_bits(host(o.m), wm, "m")
        assert_bits(host(o.v), wv, "v")
        assert_bits(host(o.params), wo, "bf16")


@pytest.mark.parametrize("nd,S,M", [(8, 152 * 128 * 6 * 2 + 7, 4), (8, 1 << 18, 2),
                                    (4, 70001, 5), (6, 65537, 3), (7, 40003, 2),
                                    (64, 4099, 2), (33, 1031, 3)])
def test_accumulate_step_multi_wave(nd, S, M):
    _check(nd, S, M, step=7, shift=0)


@pytest.mark.parametrize("nd,S", [(8, (1 << 20) + 3), (3, 100003)])
def test_accumulate_step_equals_the_two_call_path(nd, S):
    """Same bits as fsdp_grad_accumulate on the last micro-batch followed by
    the fused step on the fp32 accumulators, on the device."""
    M = 4
    scale = np.float32(1.0 / M)
    micro = _micro(S, nd, M, S)
    p, m, v = _state(S, S)
    accs = []
    for q in range(nd):
        acc = torch.empty(S, dtype=torch.float32, device=DEV)
        for j in range(M - 1):
            ss.fsdp_grad_accumulate(dev(micro[q][j]), acc, float(scale), j == 0)
        accs.append(acc)
    last = [dev(micro[q][M - 1]) for q in range(nd)]
    a = [dev(x) for x in (p, m, v)] + [torch.empty(S, dtype=torch.bfloat16, device=DEV)]
    b = [t.clone() for t in a]
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, float(scale), *a, HPC, 3)
    for q in range(nd):
        ss.fsdp_grad_accumulate(last[q], accs[q], float(scale), False)
    ss.fsdp_rs_avg_adamw_cast(accs, *b, HPC, 3)
    torch.cuda.synchronize()
    for x, y, name in zip(a, b, ("master", "m", "v", "bf16")):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32
                           else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32
                           else y.view(torch.int16)), name


def test_accumulate_step_names_its_kernel():
    S = 4096
    accs = [torch.zeros(S, device=DEV) for _ in range(8)]
    last = [torch.zeros(S, dtype=torch.bfloat16, device=DEV) for _ in range(8)]
    st = [torch.zeros(S, device=DEV) for _ in range(3)] + [
        torch.empty(S, dtype=torch.bfloat16, device=DEV)]
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, 0.5, *st, HPC, 1)
    assert ss.last_kernel() == "accum_rs_adamw_cast_vec4<8> (register-staged)"
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs[:6], last[:6], 0.5, *st, HPC, 1)
    assert ss.last_kernel() == "accum_rs_adamw_cast_vec4<6> (register-staged)"
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs[:5], last[:5], 0.5, *st, HPC, 1)
    assert ss.last_kernel() == "accum_rs_adamw_cast_vec4<up to 8: 5> (register-staged)"
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, 0.5, *st, HPC, 1, shard_group=4)
    assert ss.last_kernel() == ("accum_rs_adamw_cast_vec4<any N_d = 8, groups of 4> "
                                "(register-staged)")
    more = accs + accs[:1]
    ss.fsdp_accumulate_rs_avg_adamw_cast(more, last + last[:1], 0.5, *st, HPC, 1)
    assert ss.last_kernel() == "accum_rs_adamw_cast_vec4<any N_d = 9> (register-staged)"
    ss.fsdp_accumulate_rs_avg_adamw_cast([a[1:] for a in accs[:2]], [t[1:] for t in last[:2]],
                                         0.5,
                                         *[t[1:] for t in st], HPC, 1)
    assert ss.last_kernel() == "accum_rs_adamw_cast_scalar"
    torch.cuda.synchronize()


def test_accumulation_step_on_device_captured_in_a_cuda_graph():
    """The accumulation step (M - 1 accumulate launches over the contributions,
    then the last micro-batch inside the fused step on the device step
    state) captured once in a CUDA graph and replayed over three steps
    equals the host-scalar path run eagerly, bit for bit."""
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    units = [[(300, 40), (40,)], [(97, 13), (5,)]]
    nd, M = 8, 4
    inv_m = float(np.float32(1.0 / M))
    a = RankShardOptimizer(units, nd, 2, HPC, device=DEV, grad_dtype=torch.float32)
    b = RankShardOptimizer(units, nd, 2, HPC, device=DEV, grad_dtype=torch.float32)
    S = a.shard_total
    synth.dev_fill(synth.normal_stream(5, (89, 1), 0.02), a.master)
    b.master.copy_(a.master)
    micro = [[torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
             for _ in range(M)]

    def accumulate(opt):
        for j in range(M - 1):
            for q in range(nd):
                ss.fsdp_grad_accumulate(micro[j][q], opt.grad_in[q], inv_m, j == 0)

    b.device_step_state()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm-up, then undone
        accumulate(b)
        b.step_with_last_micro_batch_on_device(micro[M - 1], inv_m)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    b.master.copy_(a.master)
    b.m.zero_()
    b.v.zero_()
    b.state.init(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        accumulate(b)
        b.step_with_last_micro_batch_on_device(micro[M - 1], inv_m)
    for t in range(1, 4):
        for j in range(M):
            for q in range(nd):
                synth.dev_fill(synth.normal_stream(5, (89, 2, t, j, q), 1e-3), micro[j][q])
        accumulate(a)
        a.step_with_last_micro_batch(micro[M - 1], inv_m)
        g.replay()
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16)), t
    assert b.state.step() == 3


def test_binding_passes_an_explicit_sharding_factor_through():
    """Only None means full sharding in the binding; 0 or a factor that does
    not divide N_d reaches the C ABI and is rejected there."""
    S, nd = 64, 4
    accs = [torch.zeros(S, device=DEV) for _ in range(nd)]
    last = [torch.zeros(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    st = (torch.zeros(S, device=DEV), torch.zeros(S, device=DEV), torch.zeros(S, device=DEV),
          torch.empty(S, dtype=torch.bfloat16, device=DEV))
    for bad in (0, -2, 3):
        with pytest.raises(ss.ShardstepError):
            ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, 0.5, *st, HPC, 1, shard_group=bad)
    sc = ss.GradScaler(1.0, device=DEV)
    with pytest.raises(ss.ShardstepError):
        sc.check([a.to(torch.float16) for a in accs], shard_group=0)
    ss.fsdp_accumulate_rs_avg_adamw_cast(accs, last, 0.5, *st, HPC, 1, shard_group=None)
    torch.cuda.synchronize()
