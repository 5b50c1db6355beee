"""The N > 1 path on CPU, with real processes and the gloo backend: the
bench's control plane (barrier, max / sum over ranks, rank 0 alone
printing), and the step itself run across processes, which must equal, bit
for bit, the single-process emulation of N_d ranks that the library's
kernels implement:
- the sharded step on 2 ranks: each holds only its own gradient, receives
  the other's contribution to its shard through a collective, reduces in
  rank order, updates its shard and all-gathers the bf16 parameters
  ("Infra: Data Parallel", FSDP sections);
- hybrid sharding on 4 ranks with F = 2: a reduce-scatter inside each group,
  an all-reduce of the shard across the groups and an all-gather inside the
  group, over process groups of their own ("PyTorch FSDP..." section 3.3);
- the DDP step on 2 ranks: the bucketed all-reduce to a bf16 mean and the
  replicated AdamW ("4.1 数据并行详解" section 4.2);
- FSDP2 per-parameter Shard(0) on 2 ranks: chunk-cat, the reduce-scatter,
  AdamW on the padded local buffer, the all-gather copied out into the
  full tensors ("Infra: Data Parallel", FSDP2 section)."""
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


def _collect(q, procs, world, timeout=180.0):
    """Each rank's result, read before the processes are joined (a result
    larger than a pipe's buffer blocks its sender until it is read); a rank
    that dies or hangs fails the test instead of blocking it."""
    import time
    got, t0 = {}, time.monotonic()
    while len(got) < world:
        if q.empty():
            if time.monotonic() - t0 > timeout or any(p.exitcode not in (None, 0) for p in procs):
                for p in procs:
                    if p.is_alive():
                        p.kill()
                raise AssertionError(f"ranks {sorted(set(range(world)) - set(got))} gave no result")
            time.sleep(0.05)
            continue
        r, *rest = q.get()
        got[r] = rest
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return got


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
    got = _collect(q, procs, world)
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


# ------------------------------------------- hybrid sharding, four processes

def _bits32(a):
    return torch.from_numpy(np.ascontiguousarray(a).astype(np.int32))


def _hybrid_inputs(world, numels):
    import oracle
    import synth
    lay = oracle.layout(numels, 2)                  # F = 2 shards of the unit
    T, P = lay.total, lay.padded
    grads = []
    for k in range(world):
        g = np.zeros(P, np.uint16)
        g[:T] = synth.host_fill(synth.normal_stream(9, (71, k), 1e-3), 0, T, "bf16")
        grads.append(g)
    master = np.zeros(P, np.float32)
    master[:T] = synth.host_fill(synth.normal_stream(9, (72,), 0.02), 0, T, "f32")
    return lay, grads, master


def _hybrid_step(rank, world, F, port, q):
    """Rank (g, j) = g*F + j holds shard j of its replica: a reduce-scatter
    inside its group of F ranks, an all-reduce of its shard across the R
    groups, the mean over all N_d ranks, AdamW on shard j, the bf16 cast and
    the all-gather inside the group ("PyTorch FSDP..." section 3.3: full
    sharding inside groups, replication across them)."""
    _init(rank, world, port)
    import oracle
    from oracle.numerics import AdamWConfig, bf16_to_f32
    dist.init_process_group("gloo")
    R = world // F
    g_idx, j = divmod(rank, F)
    # every rank creates every group, in the same order
    intra = [dist.new_group([g * F + jj for jj in range(F)]) for g in range(R)]
    inter = [dist.new_group([g * F + jj for g in range(R)]) for jj in range(F)]
    lay, grads, master = _hybrid_inputs(world, [900, 13, 280])
    S = lay.shard
    mine = grads[rank]
    # 1. reduce-scatter inside the group: the group's gradients, summed in order j
    parts = [torch.empty(lay.padded, dtype=torch.int32) for _ in range(F)]
    dist.all_gather(parts, _bits32(mine), group=intra[g_idx])
    sl = [bf16_to_f32(p.numpy().astype(np.uint16)[j * S:(j + 1) * S]) for p in parts]
    s = sl[0].copy()
    for x in sl[1:]:
        s = s + x
    # 2. across the groups, summed in group order, then the mean over N_d
    sums = [torch.empty(S, dtype=torch.float32) for _ in range(R)]
    dist.all_gather(sums, torch.from_numpy(s), group=inter[j])
    total = sums[0].numpy().copy()
    for x in sums[1:]:
        total = total + x.numpy()
    mean = total / np.float32(world)
    p = master[j * S:(j + 1) * S].copy()
    z = np.zeros(S, np.float32)
    p, m, v = oracle.adamw(p, z, z.copy(), mean, AdamWConfig(), 1)
    ob = oracle.f32_to_bf16(p)
    # 3. all-gather of the group's bf16 shards
    shards = [torch.empty(S, dtype=torch.int32) for _ in range(F)]
    dist.all_gather(shards, _bits32(ob), group=intra[g_idx])
    full = np.concatenate([x.numpy().astype(np.uint16) for x in shards])
    q.put((rank, p.tobytes(), m.tobytes(), v.tobytes(), full.tobytes()))
    dist.destroy_process_group()


def test_hybrid_step_across_four_processes_equals_the_emulation():
    import oracle
    from oracle.numerics import AdamWConfig
    world, F = 4, 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_hybrid_step, args=(r, world, F, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = _collect(q, procs, world)
    # the one-process emulation: hybrid_shard_step over all N_d contributions
    lay, grads, master = _hybrid_inputs(world, [900, 13, 280])
    S = lay.shard
    obs = []
    for f in range(F):
        z = np.zeros(S, np.float32)
        p, m, v, ob = oracle.hybrid_shard_step(grads, F, f, S, master[f * S:(f + 1) * S].copy(),
                                               z, z.copy(), AdamWConfig(), 1)
        obs.append(ob)
        for g in range(world // F):         # every replica of shard f has the same bits
            k = g * F + f
            assert got[k][0] == p.tobytes() and got[k][1] == m.tobytes(), k
            assert got[k][2] == v.tobytes(), k
    full, _ = oracle.ag_unpack(obs, lay)
    for k in range(world):
        assert got[k][3] == full.tobytes(), k


# ----------------------------------------------- DDP buckets, two processes

def _ddp_inputs(world):
    import oracle
    import synth
    numels = [3000, 1, 4096, 17, 2500, 0, 333]
    _, _, boff = oracle.bucket_plan(numels, 2, 8192)
    total = boff[-1]
    grads = [synth.host_fill(synth.normal_stream(11, (81, k), 1e-3), 0, total, "bf16")
             for k in range(world)]
    master = synth.host_fill(synth.normal_stream(11, (82,), 0.02), 0, total, "f32")
    return boff, grads, master


def _ddp_step(rank, world, port, q):
    """Each rank all-reduces its gradient bucket by bucket (gathered, summed in
    rank order in fp32, divided by N_d, rounded to bf16: the all-reduce keeps
    the gradient's dtype), then runs the same full AdamW and cast ("4.1 数据并行详解"
    section 4.2; "Infra: Data Parallel", naive DP)."""
    _init(rank, world, port)
    import oracle
    from oracle.numerics import AdamWConfig, bf16_to_f32
    dist.init_process_group("gloo")
    boff, grads, master = _ddp_inputs(world)
    mine = grads[rank]
    avg = np.zeros(boff[-1], np.uint16)
    for a, e in zip(boff[:-1], boff[1:]):
        parts = [torch.empty(e - a, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(parts, _bits32(mine[a:e]))
        s = bf16_to_f32(parts[0].numpy().astype(np.uint16)).copy()
        for x in parts[1:]:
            s = s + bf16_to_f32(x.numpy().astype(np.uint16))
        avg[a:e] = oracle.f32_to_bf16(s / np.float32(world))
    z = np.zeros(boff[-1], np.float32)
    p, m, v = oracle.adamw(master.copy(), z, z.copy(), bf16_to_f32(avg), AdamWConfig(), 1)
    q.put((rank, avg.tobytes(), p.tobytes(), m.tobytes(), v.tobytes(),
           oracle.f32_to_bf16(p).tobytes()))
    dist.destroy_process_group()


def test_ddp_step_across_two_processes_equals_the_emulation():
    import oracle
    from oracle.numerics import AdamWConfig
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_ddp_step, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = _collect(q, procs, world)
    boff, grads, master = _ddp_inputs(world)
    z = np.zeros(boff[-1], np.float32)
    want = oracle.ddp_step(grads, boff, master.copy(), z, z.copy(), AdamWConfig(), 1)
    for r in range(world):
        assert [bytes(x) for x in got[r]] == [np.ascontiguousarray(w).tobytes() for w in want], r


# -------------------------------------------- FSDP2 Shard(0), two processes

FSDP2_SHAPES = [(7, 5), (3,), (10, 2, 2), (1, 9)]     # uneven dim 0: padding rows


def _fsdp2_inputs(world):
    import synth
    grads = [[synth.host_fill(synth.normal_stream(13, (91, k, t), 1e-3), 0, int(np.prod(s)),
                              "bf16").reshape(s) for t, s in enumerate(FSDP2_SHAPES)]
             for k in range(world)]
    masters = [synth.host_fill(synth.normal_stream(13, (92, t), 0.02), 0, int(np.prod(s)),
                               "f32").reshape(s) for t, s in enumerate(FSDP2_SHAPES)]
    return grads, masters


def _fsdp2_step(rank, world, port, q):
    """FSDP2 per-parameter Shard(0) ("Infra: Data Parallel", FSDP2 section):
    the rank's own gradients laid out rank-major with padding rows
    (chunk-cat), the reduce-scatter of its piece (gathered, summed in rank
    order), AdamW on its padded local buffer, then the all-gather of the
    local buffers copied out into the full per-parameter tensors."""
    _init(rank, world, port)
    import oracle
    from oracle.numerics import AdamWConfig
    dist.init_process_group("gloo")
    grads, masters = _fsdp2_inputs(world)
    lay = oracle.fsdp2_layout(FSDP2_SHAPES, world)
    L = lay.local
    cc = oracle.chunk_cat(grads[rank], lay)
    parts = [torch.empty(world * L, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(parts, _bits32(cc))
    contribs = [x.numpy().astype(np.uint16) for x in parts]
    p = oracle.local_buffer(masters, lay, rank)
    z = np.zeros(L, np.float32)
    p, m, v, ob = oracle.fsdp_shard_step(contribs, rank, L, p, z, z.copy(), AdamWConfig(), 1)
    locs = [torch.empty(L, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(locs, _bits32(ob))
    full = oracle.all_gather_copy_out([x.numpy().astype(np.uint16) for x in locs], lay)
    q.put((rank, p.tobytes(), m.tobytes(), v.tobytes(), b"".join(x.tobytes() for x in full)))
    dist.destroy_process_group()


def test_fsdp2_step_across_two_processes_equals_the_emulation():
    import oracle
    from oracle.numerics import AdamWConfig
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_fsdp2_step, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = _collect(q, procs, world)
    grads, masters = _fsdp2_inputs(world)
    lay = oracle.fsdp2_layout(FSDP2_SHAPES, world)
    L = lay.local
    cc = [oracle.chunk_cat(g, lay) for g in grads]
    obs = []
    for r in range(world):
        z = np.zeros(L, np.float32)
        p, m, v, ob = oracle.fsdp_shard_step(cc, r, L, oracle.local_buffer(masters, lay, r), z,
                                             z.copy(), AdamWConfig(), 1)
        assert got[r][:3] == [p.tobytes(), m.tobytes(), v.tobytes()], r
        # the padding rows of the local buffer stay zero
        for t in range(len(FSDP2_SHAPES)):
            k = lay.rows_of(r, t) * lay.row[t]
            seg = p[lay.offset[t]:lay.offset[t] + lay.chunk[t] * lay.row[t]]
            assert not seg[k:].any(), (r, t)
        obs.append(ob)
    full = oracle.all_gather_copy_out(obs, lay)
    for r in range(world):
        assert got[r][3] == b"".join(x.tobytes() for x in full), r
