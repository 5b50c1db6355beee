"""GPU parity of the device-resident AdamW step state: the fused step that
reads its scalars from the state gives the bits of the host-scalar call at
the same step, also after a restore at a checkpoint's step, and a step
captured once in a CUDA graph (advance, fused update, all-gather) replays as
consecutive steps.  The host-scalar path itself is checked against the
oracle in test_gpu_parity."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = ss.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


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


class _Shard:
    """master / m / v / bf16 of S elements with seeded contents."""

    def __init__(self, S, seed):
        self.master = torch.empty(S, device=DEV)
        synth.dev_fill(synth.normal_stream(seed, (91, 1), 0.02), self.master)
        self.m = torch.empty(S, device=DEV)
        synth.dev_fill(synth.normal_stream(seed, (91, 2), 1e-4), self.m)
        self.v = torch.empty(S, device=DEV)
        synth.dev_fill(synth.normal_stream(seed, (91, 3), 1e-7), self.v)
        self.v.abs_()
        self.out = torch.empty(S, dtype=torch.bfloat16, device=DEV)

    def clone(self):
        c = _Shard.__new__(_Shard)
        c.master, c.m, c.v, c.out = (x.clone() for x in (self.master, self.m, self.v, self.out))
        return c

    def assert_equal(self, other, what):
        for a, b, name in ((self.master, other.master, "master"), (self.m, other.m, "m"),
                           (self.v, other.v, "v")):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"{what}: {name}"
        assert torch.equal(self.out.view(torch.int16), other.out.view(torch.int16)), what


def _grads(nd, S, dtype, seed, t):
    gs = []
    for q in range(nd):
        g = torch.empty(S, dtype=dtype, device=DEV)
        synth.dev_fill(synth.normal_stream(seed, (92, t, q), 1e-3), g)
        gs.append(g)
    return gs


@pytest.mark.parametrize("nd,F,dtype,S", [(8, 8, torch.bfloat16, 6151),
                                          (8, 8, torch.bfloat16, (1 << 20) + 3),
                                          (4, 4, torch.float32, 70001),
                                          (16, 8, torch.bfloat16, 40961),
                                          (6, 6, torch.bfloat16, 8191)])
def test_state_step_equals_host_step(nd, F, dtype, S, path):
    seed = nd * 31 + S
    a = _Shard(S, seed)
    b = a.clone()
    st = ss.AdamWState(HP, 0, device=DEV)
    for t in range(1, 6):
        g = _grads(nd, S, dtype, seed, t)
        if F == nd:
            ss.fsdp_rs_avg_adamw_cast(g, a.master, a.m, a.v, a.out, HP, t)
        else:
            ss.fsdp_hybrid_rs_avg_adamw_cast(g, F, a.master, a.m, a.v, a.out, HP, t)
        st.advance()
        ss.fsdp_state_rs_avg_adamw_cast(g, b.master, b.m, b.v, b.out, st, shard_group=F)
        torch.cuda.synchronize()
        a.assert_equal(b, f"step {t}")
    assert st.step() == 5


def test_state_matches_the_oracle_scalars():
    """A few elements through the state path against the oracle directly,
    at steps 1, 2 and 1000 (the bias corrections far from their start)."""
    nd, S = 2, 4099
    for t in (1, 2, 1000):
        seed = 5 + t
        contribs = [synth.host_fill(synth.normal_stream(seed, (90, q), 1e-3), 0, nd * S, "bf16")
                    for q in range(nd)]
        p = synth.host_fill(synth.normal_stream(seed, (90, 9), 0.02), 0, S, "f32")
        m = synth.host_fill(synth.normal_stream(seed, (90, 10), 1e-4), 0, S, "f32")
        v = np.abs(synth.host_fill(synth.normal_stream(seed, (90, 11), 1e-7), 0, S, "f32"))
        dp, dm, dv = (torch.from_numpy(x.copy()).to(DEV) for x in (p, m, v))
        out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
        g = [torch.from_numpy(c[S:2 * S].view(np.int16).copy()).to(DEV).view(torch.bfloat16)
             for c in contribs]
        st = ss.AdamWState(HP, t - 1, device=DEV)
        st.advance()
        ss.fsdp_state_rs_avg_adamw_cast(g, dp, dm, dv, out, st)
        hp = AdamWConfig(HP.lr, HP.beta1, HP.beta2, HP.eps, HP.weight_decay)
        wp, wm, wv, wo = oracle.fsdp_shard_step(contribs, 1, S, p, m, v, hp, t)
        torch.cuda.synchronize()
        assert_bits(dp.cpu().numpy(), wp, f"master t={t}")
        assert_bits(dm.cpu().numpy(), wm, f"m t={t}")
        assert_bits(dv.cpu().numpy(), wv, f"v t={t}")
        assert_bits(out.view(torch.int16).cpu().numpy().view(np.uint16), wo, f"bf16 t={t}")


@pytest.mark.parametrize("k", [1, 7, 250])
def test_state_restored_at_a_step_continues_exactly(k):
    nd, S = 8, 6151
    a = _Shard(S, 3)
    b = a.clone()
    g = _grads(nd, S, torch.bfloat16, 3, k)
    # init at step k carries step k's scalars; one advance gives step k + 1's
    st = ss.AdamWState(HP, k, device=DEV)
    ss.fsdp_rs_avg_adamw_cast(g, a.master, a.m, a.v, a.out, HP, k)
    ss.fsdp_state_rs_avg_adamw_cast(g, b.master, b.m, b.v, b.out, st)
    torch.cuda.synchronize()
    a.assert_equal(b, f"restored at {k}")
    st.advance()
    ss.fsdp_rs_avg_adamw_cast(g, a.master, a.m, a.v, a.out, HP, k + 1)
    ss.fsdp_state_rs_avg_adamw_cast(g, b.master, b.m, b.v, b.out, st)
    torch.cuda.synchronize()
    a.assert_equal(b, f"advanced to {k + 1}")
    assert st.step() == k + 1


@pytest.mark.parametrize("path_name", ["auto", "tma"])
def test_step_captured_in_a_cuda_graph_replays_as_consecutive_steps(path_name):
    """advance + fused update + all-gather of the rank's unit, captured once;
    four replays with fresh gradients copied in between give the four
    host-scalar steps bit for bit."""
    prev = ss.set_fused_path(path_name)
    try:
        nd, S = 8, 8192 * 3 + 8
        r = 3
        a = _Shard(S, 11)
        b = a.clone()
        peers = []
        for q in range(nd):
            s = torch.empty(S, dtype=torch.bfloat16, device=DEV)
            synth.dev_fill(synth.normal_stream(11, (89, q), 0.02), s)
            peers.append(s)
        full_a = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
        full_b = torch.empty(nd * S, dtype=torch.bfloat16, device=DEV)
        g_in = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
        st = ss.AdamWState(HP, 0, device=DEV)
        shards_b = [peers[q] if q != r else full_b[r * S:(r + 1) * S] for q in range(nd)]

        def step_b():
            st.advance()
            ss.fsdp_state_rs_avg_adamw_cast(g_in, b.master, b.m, b.v,
                                            full_b[r * S:(r + 1) * S], st)
            ss.fsdp_ag_unpack(shards_b, full_b)

        # warm up outside the capture (kernel attributes, caches), then undo
        # its step: restore b and the state
        b0 = b.clone()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step_b()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        b = b0
        st.init(0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_b()
        torch.cuda.synchronize()
        assert st.step() == 0                       # capture ran nothing
        shards_a = [peers[q] if q != r else full_a[r * S:(r + 1) * S] for q in range(nd)]
        for t in range(1, 5):
            fresh = _grads(nd, S, torch.bfloat16, 11, t)
            for q in range(nd):
                g_in[q].copy_(fresh[q])
            ss.fsdp_rs_avg_adamw_cast(fresh, a.master, a.m, a.v, full_a[r * S:(r + 1) * S], HP,
                                      t)
            ss.fsdp_ag_unpack(shards_a, full_a)
            g.replay()
            torch.cuda.synchronize()
            for x, y, name in ((a.master, b.master, "master"), (a.m, b.m, "m"),
                               (a.v, b.v, "v")):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), f"{name} {t}"
            assert torch.equal(full_a.view(torch.int16), full_b.view(torch.int16)), f"full {t}"
        assert st.step() == 4
    finally:
        ss.set_fused_path(prev)


def test_rank_optimizer_step_on_device_in_a_graph():
    """RankShardOptimizer.step_on_device captured once equals step() run
    eagerly, over three replays of a two-unit hybrid rank view."""
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    units = [[(300, 40), (40,)], [(97, 13)]]
    a = RankShardOptimizer(units, 8, 1, HP, device=DEV, shard_group=4)
    b = RankShardOptimizer(units, 8, 1, HP, device=DEV, shard_group=4)
    synth.dev_fill(synth.normal_stream(4, (88, 1), 0.02), a.master)
    b.master.copy_(a.master)
    b.device_step_state()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # warm-up, then undone
        b.step_on_device()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    b.master.copy_(a.master)
    b.m.zero_()
    b.v.zero_()
    b.state.init(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b.step_on_device()
    for t in range(1, 4):
        for q in range(8):
            synth.dev_fill(synth.normal_stream(4, (88, 2, t, q), 1e-3), a.grad_in[q])
            b.grad_in[q].copy_(a.grad_in[q])
        a.step()
        g.replay()
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.params.view(torch.int16), b.params.view(torch.int16)), t
    assert b.state.step() == 3


def test_loss_scaled_step_captured_in_a_cuda_graph():
    """check + advance (skipped with found_inf) + scaled update from the
    state + scale update, captured once and replayed over four iterations,
    the second with an inf in one gradient: equal to the host path in which
    the skipped step does not count (AdamW steps 1, -, 2, 3); the scale
    backs off once and the state's count ends at 3."""
    nd, S = 8, 6151 * 4
    a = _Shard(S, 21)
    b = a.clone()
    sa = ss.GradScaler(init_scale=1024.0, device=DEV)
    sb = ss.GradScaler(init_scale=1024.0, device=DEV)
    st = ss.AdamWState(HP, 0, device=DEV)
    g_in = [torch.empty(S, dtype=torch.float16, device=DEV) for _ in range(nd)]
    for q in range(nd):
        synth.dev_fill(synth.normal_stream(21, (87, 0, q), 1e-3 * 1024.0), g_in[q])

    def step_b():
        sb.check(g_in)
        st.advance(skip=sb.found_inf)
        sb.step_state(g_in, b.master, b.m, b.v, b.out, st)
        sb.update()

    b0 = b.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):            # warm-up, then undone
        step_b()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    b = b0
    sb.scale.fill_(1024.0)
    sb.tracker.zero_()
    sb.found_inf.zero_()
    st.init(0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step_b()
    t_host = 0
    for it in range(4):
        fresh = [torch.empty(S, dtype=torch.float16, device=DEV) for _ in range(nd)]
        for q in range(nd):
            synth.dev_fill(synth.normal_stream(21, (87, it + 1, q), 1e-3 * 1024.0), fresh[q])
        if it == 1:
            fresh[3][17] = float("inf")
        for q in range(nd):
            g_in[q].copy_(fresh[q])
        skipped = it == 1
        if not skipped:
            t_host += 1
        sa.check(fresh)
        sa.step(fresh, a.master, a.m, a.v, a.out, HP, max(t_host, 1))
        sa.update()
        graph.replay()
        torch.cuda.synchronize()
        a.assert_equal(b, f"iteration {it}")
        assert sa.scale.item() == sb.scale.item()
        assert st.step() == t_host
    assert sa.scale.item() == 512.0


@pytest.mark.parametrize("S", [1, 3, 5, 4097])
def test_state_step_on_ragged_and_tiny_shards(S, path):
    """Shards of a few elements (the tail that block 0 handles) and a ragged
    one, 3 steps, against the host-scalar call."""
    nd = 4
    a = _Shard(S, 40 + S)
    b = a.clone()
    st = ss.AdamWState(HP, 0, device=DEV)
    for t in range(1, 4):
        g = _grads(nd, S, torch.bfloat16, 40 + S, t)
        ss.fsdp_rs_avg_adamw_cast(g, a.master, a.m, a.v, a.out, HP, t)
        st.advance()
        ss.fsdp_state_rs_avg_adamw_cast(g, b.master, b.m, b.v, b.out, st)
        torch.cuda.synchronize()
        a.assert_equal(b, f"S={S} step {t}")


def test_state_at_a_late_step():
    """Restored at step 10^6 (the beta powers long underflowed or tiny) and
    advanced once: the bits of the host-scalar call at 10^6 + 1."""
    nd, S = 2, 8191
    a = _Shard(S, 77)
    b = a.clone()
    g = _grads(nd, S, torch.bfloat16, 77, 1)
    st = ss.AdamWState(HP, 10 ** 6, device=DEV)
    st.advance()
    ss.fsdp_rs_avg_adamw_cast(g, a.master, a.m, a.v, a.out, HP, 10 ** 6 + 1)
    ss.fsdp_state_rs_avg_adamw_cast(g, b.master, b.m, b.v, b.out, st)
    torch.cuda.synchronize()
    a.assert_equal(b, "late step")
    assert st.step() == 10 ** 6 + 1


def test_engine_mixes_host_and_device_steps():
    """RankShardOptimizer with its count on the device: device steps, then a
    host-scalar step (which takes the device count and moves it on), then a
    device step again give the bits of four host-scalar steps, and both
    counts agree at 4."""
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    units = [[(300, 7), (5,)], [(1000,)]]
    nd = 3
    a = RankShardOptimizer(units, nd, 1, HP, device=DEV)
    b = RankShardOptimizer(units, nd, 1, HP, device=DEV)
    for o in (a, b):
        torch.manual_seed(3)
        o.master.copy_(torch.randn(o.shard_total, device=DEV) * 0.02)
        for q in range(nd):
            o.grad_in[q].copy_((torch.randn(o.shard_total, device=DEV) * 1e-3).to(torch.bfloat16))
    for _ in range(4):
        a.step()
    b.device_step_state()
    b.step_on_device()
    b.step_on_device()
    b.step()
    b.step_on_device()
    torch.cuda.synchronize()
    assert a.t == 4 and b.state.step() == 4 and b.t == 3
    for name in ("master", "m", "v", "params"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), name
