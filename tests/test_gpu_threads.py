"""Concurrent use of the library from several host threads, each on its own
CUDA stream and buffers: the entry points keep no per-call state (the
process-wide caches -- SM count, occupancy, shared-memory opt-in, the kernel
choice -- are written once and read thereafter), so every thread's results
must equal the oracle's, whatever the interleaving."""
import threading

import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from oracle.numerics import AdamWConfig

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HP = AdamWConfig()


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    assert ss.device_status() == 0


def _work(tid, nd, S, M, results):
    """One thread: accumulate M micro-batches per rank, fused step, bucket
    all-reduce and all-gather, all on its own stream."""
    try:
        s = torch.cuda.Stream(device=DEV)
        P = nd * S
        micro = [[synth.host_fill(synth.normal_stream(tid, (55, q, j), 1e-3), 0, P, "bf16")
                  for j in range(M)] for q in range(nd)]
        master = synth.host_fill(synth.normal_stream(tid, (56,), 0.02), 0, S, "f32")
        with torch.cuda.stream(s):
            accs = []
            for q in range(nd):
                acc = torch.empty(P, device=DEV)
                for j in range(M):
                    g = torch.from_numpy(micro[q][j].view(np.int16)).to(DEV).view(torch.bfloat16)
                    ss.fsdp_grad_accumulate(g, acc, float(np.float32(1 / M)), j == 0)
                accs.append(acc)
            r = tid % nd
            dp = torch.from_numpy(master.copy()).to(DEV)
            dm = torch.zeros(S, device=DEV)
            dv = torch.zeros(S, device=DEV)
            out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
            for t in (1, 2, 3):
                ss.fsdp_rs_avg_adamw_cast([a[r * S:(r + 1) * S] for a in accs], dp, dm, dv, out,
                                          ss.AdamW(), t)
            g16 = [torch.from_numpy(micro[q][0].view(np.int16)).to(DEV).view(torch.bfloat16)
                   for q in range(nd)]
            avg = torch.empty(P, dtype=torch.bfloat16, device=DEV)
            ss.ddp_bucket_allreduce_avg(g16, [0, S, 2 * S, P], avg)
            full = torch.empty(P, dtype=torch.bfloat16, device=DEV)
            ss.fsdp_ag_unpack([avg[q * S:(q + 1) * S] for q in range(nd)], full)
        s.synchronize()
        results[tid] = (dp.cpu().numpy(), dm.cpu().numpy(), dv.cpu().numpy(),
                        out.view(torch.int16).cpu().numpy().view(np.uint16),
                        avg.view(torch.int16).cpu().numpy().view(np.uint16),
                        full.view(torch.int16).cpu().numpy().view(np.uint16), micro, master, r)
    except Exception as e:  # reported by the test
        results[tid] = e


@pytest.mark.parametrize("n_threads", [4])
def test_threads_on_their_own_streams_match_the_oracle(n_threads):
    nd, S, M = 4, 2048 * 40 + 13, 2
    results = {}
    ts = [threading.Thread(target=_work, args=(k, nd, S, M, results)) for k in range(n_threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for k in range(n_threads):
        res = results[k]
        assert not isinstance(res, Exception), repr(res)
        dp, dm, dv, out, avg, full, micro, master, r = res
        accs = [oracle.grad_accumulate(micro[q], np.float32(1 / M)) for q in range(nd)]
        p, m, v = master.copy(), np.zeros(S, np.float32), np.zeros(S, np.float32)
        for t in (1, 2, 3):
            p, m, v, ob = oracle.fsdp_shard_step(accs, r, S, p, m, v, HP, t)
        assert dp.tobytes() == p.tobytes() and dm.tobytes() == m.tobytes()
        assert dv.tobytes() == v.tobytes() and out.tobytes() == ob.tobytes()
        want_avg = oracle.bucket_allreduce_avg([micro[q][0] for q in range(nd)],
                                               [0, S, 2 * S, nd * S])
        assert avg.tobytes() == want_avg.tobytes()
        assert full.tobytes() == want_avg.tobytes()
