"""The benchmark's whole-job steps compute the method's step.

``bench.py`` times the 9.4M-parameter unit (N_d = 4, M = 4) and GPT-2 small
(N_d = 8) as whole jobs: every emulated rank's accumulation, fused step and
the all-gather, laid out for few launches (the 9.4M unit's ranks side by
side, one fused launch over all their shards).  These tests build each job
exactly as the benchmark does, run one step with host scalars and one with
the step count on the device (captured in a CUDA graph and replayed), and
compare with the oracle: the 9.4M unit on every element of every rank's
state and of the gathered unit, GPT-2 small on sampled positions of every
rank and of the gathered unit.  The oracle side takes its layout from
``oracle.layout`` and its inputs from the seeded streams, never from the
GPU."""
import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig
from synth import workloads as W
from tests._cmp import assert_bits
from tests._views import oracle_layouts, oracle_rank_values

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
    assert ss.device_status() == 0


def _bench():
    import bench
    return bench


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _graph_step(job):
    """One step of ``job`` with the step count on the device, captured in a
    CUDA graph and replayed once (the benchmark's --graph form)."""
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        job.run(graph_form=True)
    g.replay()
    torch.cuda.synchronize()


def _unit9m_oracle(w, steps):
    nd, M = w.nd, w.micro
    numels = w.unit_numels(0)
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    g = [[oracle.flat_pack([synth.host_fill(w.grad_stream(1, q, j, 0, t), 0, n, "bf16")
                            for t, n in enumerate(numels)], nd)[0] for j in range(M)]
         for q in range(nd)]
    accs = [oracle.grad_accumulate(g[q], np.float32(1.0 / M)) for q in range(nd)]
    p, lay = oracle.flat_pack([synth.host_fill(w.master_stream(0, t), 0, n, "f32")
                               for t, n in enumerate(numels)], nd)
    S = lay.shard
    state = [(p[r * S:(r + 1) * S], np.zeros(S, np.float32), np.zeros(S, np.float32))
             for r in range(nd)]
    per_step = []
    for t in range(1, steps + 1):
        outs = []
        for r in range(nd):
            p1, m1, v1, o1 = oracle.fsdp_shard_step(accs, r, S, *state[r], hp, t)
            state[r] = (p1, m1, v1)
            outs.append(o1)
        per_step.append((np.concatenate([s[0] for s in state]),
                         np.concatenate([s[1] for s in state]),
                         np.concatenate([s[2] for s in state]),
                         oracle.ag_unpack(outs, lay)[0]))
    return per_step


@pytest.mark.parametrize("form", ["host_scalars", "device_state"])
def test_unit_9m_job_every_element(form):
    b = _bench()
    job = b._SmallJob(b.UNIT9M_WORKLOAD, torch, ss, torch.device(DEV))
    want = _unit9m_oracle(job.w, 2)
    if form == "device_state":
        job.device_state()
        job.run(graph_form=True)          # step 1, eager
    else:
        job.run()
    torch.cuda.synchronize()
    got = (job.master.cpu().numpy(), job.m.cpu().numpy(), job.v.cpu().numpy(), _u16(job.full))
    for name, gv, wv in zip(("master", "m", "v", "gathered unit"), got, want[0]):
        assert_bits(gv, wv, f"step 1 {name}")
    if form == "device_state":
        _graph_step(job)                  # step 2, replayed from a graph
    else:
        job.run()
    torch.cuda.synchronize()
    got = (job.master.cpu().numpy(), job.m.cpu().numpy(), job.v.cpu().numpy(), _u16(job.full))
    for name, gv, wv in zip(("master", "m", "v", "gathered unit"), got, want[1]):
        assert_bits(gv, wv, f"step 2 {name}")


def _gpt2_oracle_at(w, r, idx, steps):
    """Rank r's master and bf16 parameters at its positions idx after each
    of ``steps`` steps (the same gradients every step)."""
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    contribs = [oracle_rank_values(w, r, idx, lambda u, k, q=q: w.grad_stream(1, q, 0, u, k),
                                   "bf16") for q in range(w.nd)]
    p = oracle_rank_values(w, r, idx, w.master_stream, "f32")
    n = idx.size
    m = v = np.zeros(n, np.float32)
    out = []
    for t in range(1, steps + 1):
        p, m, v, o = oracle.fsdp_shard_step(contribs, 0, n, p, m, v, hp, t)
        out.append((p, o))
    return out


@pytest.mark.parametrize("form", ["host_scalars", "device_state"])
def test_gpt2_small_job_sampled(form):
    b = _bench()
    job = b._SmallJob(b.GPT2_WORKLOAD, torch, ss, torch.device(DEV))
    w = job.w
    lays = oracle_layouts(w)
    S = sum(lay.shard for lay in lays)
    rng = np.random.default_rng(11)
    # positions of each rank: random, the first and last of every unit's shard
    starts = np.cumsum([0] + [lay.shard for lay in lays])
    edges = np.concatenate([starts[:-1], starts[1:] - 1])
    idx_r = [np.unique(np.concatenate([rng.integers(0, S, 3000), edges])).astype(np.int64)
             for _ in range(w.nd)]
    # positions of the gathered unit 0: rank j // S0, position j % S0
    S0, P0 = lays[0].shard, lays[0].padded
    jg = np.unique(np.concatenate([rng.integers(0, P0, 4000), [0, P0 - 1],
                                   np.arange(1, w.nd) * S0 - 1, np.arange(1, w.nd) * S0]))
    want = [_gpt2_oracle_at(w, r, idx_r[r], 2) for r in range(w.nd)]
    want_g = []
    for t in range(2):
        row = np.zeros(jg.size, np.uint16)
        for r in range(w.nd):
            sel = (jg // S0) == r
            if sel.any():
                row[sel] = _gpt2_oracle_at(w, r, (jg[sel] % S0).astype(np.int64), t + 1)[t][1]
        want_g.append(row)

    if form == "device_state":
        job.device_state()
    for t in range(2):
        if form == "host_scalars":
            job.run()
        elif t == 0:
            job.run(graph_form=True)
        else:
            _graph_step(job)
        torch.cuda.synchronize()
        for r, o in enumerate(job.opts):
            ix = torch.from_numpy(idx_r[r]).to(DEV)
            assert_bits(o.master[ix].cpu().numpy(), want[r][t][0], f"step {t + 1} rank {r} master")
            assert_bits(_u16(o.params[ix]), want[r][t][1], f"step {t + 1} rank {r} bf16")
        gathered = _u16(job.full[torch.from_numpy(jg).to(DEV)])
        assert_bits(gathered, want_g[t], f"step {t + 1} gathered unit 0")
