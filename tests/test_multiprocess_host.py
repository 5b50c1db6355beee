"""The N > 1 path on CPU, with real processes and the gloo backend
(world_size 2): the bench's control plane (barrier, max / sum over ranks,
rank 0 alone printing), and the sharded step itself run across two
processes -- each rank holds only its own gradient, receives the other
rank's contribution to its shard through a collective, reduces it in rank
order, updates its shard and all-gathers the bf16 parameters -- which must
equal, bit for bit, the single-process emulation of N_d ranks that the
library's kernels implement ("Infra: Data Parallel", FSDP sections: the
reduce-scatter before the sharded update and the all-gather after it)."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)


def _control_plane(rank, world, port, q):
    _init(rank, world, port)
    import bench
    bench.init_dist(world)
    bench.barrier(world)
    mx = bench.allreduce_max(world, float(10 + rank))
    sm = bench.allreduce_sum(world, float(1 + rank))
    bench.barrier(world)
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_bench_control_plane_across_two_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_control_plane, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    assert got == [(0, 11.0, 3.0), (1, 11.0, 3.0)]


def _sharded_step(rank, world, port, q):
    _init(rank, world, port)
    import oracle
    import synth
    from oracle.numerics import AdamWConfig
    dist.init_process_group("gloo")
    hp = AdamWConfig()
    numels = [600, 7, 394]                         # T = 1001: one element of padding at N_d = 2
    lay = oracle.layout(numels, world)
    T, P, S = lay.total, lay.padded, lay.shard
    # this rank's own flat bf16 gradient (zero padding) and the shared master
    g = np.zeros(P, np.uint16)
    g[:T] = synth.host_fill(synth.normal_stream(7, (61, rank), 1e-3), 0, T, "bf16")
    master = np.zeros(P, np.float32)
    master[:T] = synth.host_fill(synth.normal_stream(7, (62,), 0.02), 0, T, "f32")
    # reduce-scatter input: every rank's gradient bits (gloo moves int32, so
    # the bf16 bits travel widened and come back unchanged)
    parts = [torch.empty(P, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(g.astype(np.int32)))
    contribs = [p.numpy().astype(np.uint16) for p in parts]
    p = master[rank * S:(rank + 1) * S].copy()
    m = np.zeros(S, np.float32)
    v = np.zeros(S, np.float32)
    p, m, v, ob = oracle.fsdp_shard_step(contribs, rank, S, p, m, v, hp, 1)
    # all-gather of the bf16 shards
    shards = [torch.empty(S, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(shards, torch.from_numpy(ob.astype(np.int32)))
    full = np.concatenate([s.numpy().astype(np.uint16) for s in shards])
    q.put((rank, p.tobytes(), m.tobytes(), v.tobytes(), full.tobytes()))
    dist.destroy_process_group()


def test_sharded_step_across_two_processes_equals_the_emulation():
    import oracle
    import synth
    from oracle.numerics import AdamWConfig
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_sharded_step, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = {r: rest for r, *rest in (q.get() for _ in range(world))}
    # one process emulating both ranks, as the GPU path does
    numels = [600, 7, 394]
    lay = oracle.layout(numels, world)
    T, P, S = lay.total, lay.padded, lay.shard
    contribs = []
    for r in range(world):
        g = np.zeros(P, np.uint16)
        g[:T] = synth.host_fill(synth.normal_stream(7, (61, r), 1e-3), 0, T, "bf16")
        contribs.append(g)
    master = np.zeros(P, np.float32)
    master[:T] = synth.host_fill(synth.normal_stream(7, (62,), 0.02), 0, T, "f32")
    obs = []
    for r in range(world):
        p = master[r * S:(r + 1) * S].copy()
        z = np.zeros(S, np.float32)
        p, m, v, ob = oracle.fsdp_shard_step(contribs, r, S, p, z, z.copy(), AdamWConfig(), 1)
        assert got[r][0] == p.tobytes() and got[r][1] == m.tobytes() and got[r][2] == v.tobytes()
        obs.append(ob)
    full, _ = oracle.ag_unpack(obs, lay)
    for r in range(world):
        assert got[r][3] == full.tobytes()
    # the padding position stays zero after the step
    assert np.frombuffer(got[0][3], np.uint16)[T:].tolist() == [0] * (P - T)


@pytest.mark.parametrize("workload", ["llama_7b_rank0_nd8", "llama_1b_rank0_nd8_m4",
                                      "ddp_nd8_buckets", "llama_7b_layer_ragged_nd8",
                                      "llama_7b_fsdp2_layer_nd8", "unit_9m_nd4_m4",
                                      "gpt2_small_nd8"])
def test_reference_arm_under_torchrun_prints_once(workload):
    """Launched the way the N > 1 runs are, the oracle arm runs on rank 0
    alone and prints one JSON line; the other rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", workload, "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
