"""Stream order under dependent launches.  The library's kernels may go out
as programmatic dependents of the kernel before them in the stream; a
first kernel of a call then waits for its predecessor before it touches
memory.  A whole step -- a torch kernel producing the gradients, the
accumulate launches, the fused step with the last micro-batch, the
all-gather, a torch kernel consuming the gathered unit -- must give the
oracle's bits with dependent launches on and off, eagerly and replayed
from a CUDA graph on the device step state.  The chains are read-after-
write on every link (an accumulator read by the next accumulation, the
step state read by the fused kernel, the shards read by the all-gather)."""
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
HP = AdamWConfig()
ND, M = 4, 3
S = 152 * 128 * 4 * 5 + 4 * 7 + 3       # several waves, a ragged tail


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    yield
    assert ss.device_status() == 0


@pytest.fixture(params=[True, False])
def dependent(request):
    prev = ss.set_dependent_launch(request.param)
    yield request.param
    ss.set_dependent_launch(prev)


def _inputs(t):
    return [[synth.host_fill(synth.normal_stream(t, (89, q, j), 1e-3), 0, ND * S, "bf16")
             for j in range(M)] for q in range(ND)]


def _oracle(steps, p0):
    p, m, v = p0, np.zeros(ND * S, np.float32), np.zeros(ND * S, np.float32)
    outs = None
    for t in range(1, steps + 1):
        micro = _inputs(t)
        accs = [oracle.grad_accumulate(micro[q], np.float32(1.0 / M)) for q in range(ND)]
        res = [oracle.fsdp_shard_step(accs, r, S, p[r * S:(r + 1) * S], m[r * S:(r + 1) * S],
                                      v[r * S:(r + 1) * S], HP, t) for r in range(ND)]
        p = np.concatenate([x[0] for x in res])
        m = np.concatenate([x[1] for x in res])
        v = np.concatenate([x[2] for x in res])
        outs = [x[3] for x in res]
    return p, m, v, np.concatenate(outs)


class _Job:
    def __init__(self):
        self.staged = [[torch.empty(ND * S, dtype=torch.bfloat16, device=DEV) for _ in range(M)]
                       for _ in range(ND)]
        self.g = [[torch.empty_like(x) for x in row] for row in self.staged]
        self.acc = [torch.empty(ND * S, device=DEV) for _ in range(ND)]
        self.p0 = synth.host_fill(synth.normal_stream(7, (89, 99), 0.02), 0, ND * S, "f32")
        self.master = torch.from_numpy(self.p0.copy()).to(DEV)
        self.m = torch.zeros(ND * S, device=DEV)
        self.v = torch.zeros(ND * S, device=DEV)
        self.outs = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(ND)]
        self.full = torch.full((ND * S,), 3.0, dtype=torch.bfloat16, device=DEV)
        self.seen = torch.empty_like(self.full)

    def stage(self, t):
        for q, row in enumerate(_inputs(t)):
            for j, h in enumerate(row):
                self.staged[q][j].copy_(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16))

    def step(self, t, state=None):
        for q in range(ND):                       # the producer: torch copies
            for j in range(M):
                self.g[q][j].copy_(self.staged[q][j])
        for q in range(ND):
            for j in range(M - 1):
                ss.fsdp_grad_accumulate(self.g[q][j], self.acc[q], float(1.0 / M), j == 0)
        if state is not None:
            state.advance()
        for r in range(ND):
            sl = slice(r * S, (r + 1) * S)
            args = ([a[sl] for a in self.acc], [row[M - 1][sl] for row in self.g],
                    float(1.0 / M), self.master[sl], self.m[sl], self.v[sl], self.outs[r])
            if state is None:
                ss.fsdp_accumulate_rs_avg_adamw_cast(*args, ss.AdamW(), t)
            else:
                ss.fsdp_state_accumulate_rs_avg_adamw_cast(*args, state)
        ss.fsdp_ag_unpack(self.outs, self.full)
        self.seen.copy_(self.full)                # the consumer: a torch copy

    def check(self, steps):
        p, m, v, out = _oracle(steps, self.p0)
        torch.cuda.synchronize()
        assert_bits(self.master.cpu().numpy(), p, "master")
        assert_bits(self.m.cpu().numpy(), m, "m")
        assert_bits(self.v.cpu().numpy(), v, "v")
        assert_bits(self.seen.view(torch.int16).cpu().numpy().view(np.uint16), out, "gathered")


def test_eager_step_chain_keeps_stream_order(dependent):
    job = _Job()
    for t in (1, 2, 3):
        job.stage(t)
        job.step(t)
    job.check(3)


def test_graph_step_chain_keeps_stream_order(dependent):
    job = _Job()
    state = ss.AdamWState(ss.AdamW(), 0, device=DEV)
    job.stage(1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                 # warm-up outside the capture, then undone
        job.step(1, state)
    torch.cuda.current_stream().wait_stream(side)
    job.master.copy_(torch.from_numpy(job.p0))
    job.m.zero_()
    job.v.zero_()
    state.init(0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        job.step(0, state)
    for t in (1, 2, 3):
        job.stage(t)
        graph.replay()
    assert state.step() == 3
    job.check(3)
