"""Pins for the oracle's DDP bucket plan and bucketed all-reduce average, and
for the memory and communication ledger: a hand-worked plan, invariants
checked by brute force, the all-reduce = reduce-scatter + all-gather identity
("4.1 数据并行详解" section 5.1), a simulated ring that counts the elements it
sends, and the numbers the pages print (fixture in tests/golden)."""
import itertools
import os

import numpy as np
import pytest

import oracle
from oracle.ddp import MiB

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ bucket plan

def test_bucket_plan_hand_example():
    # params (registration order) of 4, 4, 10, 2, 2 elements, 2-byte grads, cap
    # 16 bytes = 8 elements.  Reverse order: p4(2) p3(2) p2(10) p1(4) p0(4)
    #   bucket 0: p4 p3          (4 elements; adding p2 would pass the cap)
    #   bucket 1: p2             (10 > cap: alone)
    #   bucket 2: p1 p0          (8 elements = cap, allowed)
    off, of, boff = oracle.bucket_plan([4, 4, 10, 2, 2], 2, 16)
    assert of == [2, 2, 1, 0, 0]
    assert boff == [0, 4, 14, 22]
    assert off == [18, 14, 4, 2, 0]


def _check_plan(numels, cap_elems):
    off, of, boff = oracle.bucket_plan(numels, 1, cap_elems)
    n = len(numels)
    nb = len(boff) - 1
    assert boff[0] == 0 and boff[-1] == sum(numels)
    assert all(a <= b for a, b in zip(boff, boff[1:]))
    # buckets visit the parameters in reverse registration order (zero-size
    # parameters share the offset of their neighbour)
    order = sorted(range(n), key=lambda i: (of[i], off[i], -i))
    assert order == list(reversed(range(n)))
    for k in range(nb):
        members = [i for i in range(n) if of[i] == k]
        assert members, "no empty buckets"
        size = sum(numels[i] for i in members)
        assert size == boff[k + 1] - boff[k]
        # within the cap, unless a single parameter is larger than the cap
        assert size <= cap_elems or (len(members) == 1 or
                                     sum(numels[i] > 0 for i in members) == 1)
        # greedy: the next parameter in reverse order would have passed the cap
        if k + 1 < nb:
            nxt = max(i for i in range(n) if of[i] == k + 1)
            assert size + numels[nxt] > cap_elems
    # parameters are contiguous and never split
    for i in range(n):
        assert boff[of[i]] <= off[i] and off[i] + numels[i] <= boff[of[i] + 1]


def test_bucket_plan_brute_force():
    for n in range(0, 6):
        for numels in itertools.product([0, 1, 2, 3, 5, 8], repeat=n):
            for cap in (1, 2, 4, 7, 16):
                _check_plan(list(numels), cap)


def test_default_cap_gives_a_4096_square_matrix_its_own_bucket():
    # 4096 x 4096 bf16 = 32 MiB > 25 MiB
    numels = [768, 768, 768 * 3072, 768 * 3072, 4096 * 4096]
    off, of, boff = oracle.bucket_plan(numels, 2, 25 * MiB)
    assert of[4] == 0 and boff[1] == 4096 * 4096
    assert of[0] == of[1] == of[2] == of[3] == 1


# ----------------------------------------------- all-reduce = RS + AG

@pytest.mark.parametrize("nd", [2, 3, 8])
def test_bucket_allreduce_equals_reduce_scatter_then_all_gather(nd):
    rng = np.random.default_rng(nd)
    S = 40
    P = nd * S
    grads = [oracle.f32_to_bf16((rng.standard_normal(P) * 1e-3).astype(np.float32))
             for _ in range(nd)]
    _, _, boff = oracle.bucket_plan([7, 33, 13, P - 53], 2, 60)
    ar = oracle.bucket_allreduce_avg(grads, boff)
    rs_ag = np.concatenate([oracle.f32_to_bf16(oracle.rs_avg(grads, r, S)) for r in range(nd)])
    assert np.array_equal(ar, rs_ag)


def _ring_allreduce(chunks_per_rank):
    """Simulated ring all-reduce on N ranks, each holding N chunks: N-1
    reduce-scatter steps then N-1 all-gather steps, every rank sending one
    chunk to its right neighbour per step.  Returns (result per rank, elements
    sent per rank).  Exact integer data."""
    N = len(chunks_per_rank)
    buf = [[c.copy() for c in rank] for rank in chunks_per_rank]
    sent = [0] * N
    for step in range(N - 1):              # reduce-scatter
        msgs = []
        for r in range(N):
            k = (r - step) % N
            msgs.append(((r + 1) % N, k, buf[r][k].copy()))
            sent[r] += buf[r][k].size
        for dst, k, data in msgs:
            buf[dst][k] = buf[dst][k] + data
    for step in range(N - 1):              # all-gather
        msgs = []
        for r in range(N):
            k = (r + 1 - step) % N
            msgs.append(((r + 1) % N, k, buf[r][k].copy()))
            sent[r] += buf[r][k].size
        for dst, k, data in msgs:
            buf[dst][k] = data
    return buf, sent


@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_ring_traffic_matches_comm_ledger(N):
    psi = N * 6
    rng = np.random.default_rng(N)
    data = [rng.integers(-100, 100, size=psi) for _ in range(N)]
    res, sent = _ring_allreduce([np.split(d, N) for d in data])
    total = np.sum(data, axis=0)
    for r in range(N):
        assert np.array_equal(np.concatenate(res[r]), total)
    # each rank sends 2 (N-1)/N psi elements = 2 (N-1)/N psi * 2 bytes (16-bit)
    for r in range(N):
        assert sent[r] == 2 * (N - 1) * psi // N
        assert 2 * sent[r] == pytest.approx(
            oracle.comm_bytes_per_gpu(psi, N, "all_reduce", exact=True))
        assert sent[r] // 2 * 2 == pytest.approx(
            oracle.comm_bytes_per_gpu(psi, N, "reduce_scatter", exact=True))


# ----------------------------------------------------------------- ledger

def test_memory_ledger_matches_printed_values():
    with open(os.path.join(GOLDEN, "memory_ledger.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for name, psi, nd, k, stage, value, tol in rows:
        got = oracle.state_bytes_per_gpu(float(psi), int(nd), int(stage), float(k)) / oracle.GB
        assert abs(got - float(value)) <= float(tol), name


def test_memory_ledger_closed_forms():
    psi = 7e9
    # N_d = 8: 112, 38.5, 26.25, 14 GB; N_d = 4: 112, 49, 38.5, 28 GB
    for nd, want in ((8, (112, 38.5, 26.25, 14)), (4, (112, 49, 38.5, 28))):
        got = [oracle.state_bytes_per_gpu(psi, nd, s) / oracle.GB for s in range(4)]
        assert got == pytest.approx(want, rel=1e-12)
    # N_d = 1 recovers the replicated ledger at every stage
    assert all(oracle.state_bytes_per_gpu(psi, 1, s) == 16 * psi for s in range(4))
    # ZeRO-3 scales as 1/N_d ("4.1 数据并行详解" section 7: 16 Psi / N)
    assert oracle.state_bytes_per_gpu(psi, 16, 3) == pytest.approx(16 * psi / 16)


def test_comm_ledger_matches_printed_volumes():
    """The per-GPU volumes the pages print (tests/golden/comm_volume.txt),
    in bytes at 2 bytes per element or in elements, at several N_d (the
    printed figures drop the (N_d - 1) / N_d factor, so they hold for any)."""
    with open(os.path.join(GOLDEN, "comm_volume.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 10
    psi = 7e9
    for name, kind, unit, value in rows:
        for nd in (2, 8, 512):
            got = oracle.comm_bytes_per_gpu(psi, nd, kind)
            if unit == "elements":
                got /= 2
            assert got == float(value) * psi, (name, nd)


def test_comm_ledger_closed_forms():
    psi, nd = 1e9, 8
    b = lambda kind: oracle.comm_bytes_per_gpu(psi, nd, kind)
    assert b("reduce_scatter") == b("all_gather") == 2 * psi
    assert b("all_reduce") == b("ddp") == 4 * psi
    assert b("zero1") == b("zero2") == b("ddp")          # same volume as naive DP
    assert b("zero3") == 6 * psi
    # "4.1 数据并行详解" section 8 in elements: DDP 2 Psi, FSDP 3 Psi
    assert b("ddp") / 2 == 2 * psi and b("zero3") / 2 == 3 * psi
    # section 5.3: the centralised root moves 2 (N-1) Psi elements
    assert b("centralised_root") / 2 == 2 * (nd - 1) * psi
    with pytest.raises(ValueError):
        b("broadcast")


def test_ddp_step_updates_with_the_bf16_rounded_mean():
    """The all-reduce keeps bf16, so the replicated AdamW sees the mean rounded
    to bf16, not the fp32 mean.  Two ranks with gradients 1 and 2^-8: the
    fp32 mean 0.5 + 2^-9 lies half a bf16 ulp above 0.5, so it rounds (ties
    to even) to exactly 0.5.  With beta1 = beta2 = 0, eps = 1, lr = 1, no
    decay, p = 0 at step 1: m = g, v = g^2, bc1 = bc2 = 1 and the update is
    g / (|g| + 1), so p = -(0.5 / 1.5) = -fl32(1/3) for the rounded mean,
    while the fp32 mean would give -fl32(0.501953125 / 1.501953125)."""
    from oracle.numerics import AdamWConfig
    one, tiny = 0x3F80, 0x3B80                         # bf16 bits of 1.0 and 2^-8
    assert oracle.bf16_to_f32(np.array([tiny], np.uint16))[0] == np.float32(2.0 ** -8)
    hp = AdamWConfig(lr=1.0, beta1=0.0, beta2=0.0, eps=1.0, weight_decay=0.0)
    z = np.zeros(1, np.float32)
    avg, p, m, v, pb = oracle.ddp_step([np.array([one], np.uint16), np.array([tiny], np.uint16)],
                                       [0, 1], z, z, z, hp, 1)
    assert avg[0] == 0x3F00                            # bf16 0.5
    assert m[0] == np.float32(0.5) and v[0] == np.float32(0.25)
    assert p[0] == -np.float32(1.0 / 3.0)
    assert p[0] != -np.float32(0.501953125 / 1.501953125)
