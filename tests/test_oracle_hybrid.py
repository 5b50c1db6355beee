"""Pins for the oracle's hybrid sharding (sharding factor F): the two special
cases the pages name ("PyTorch FSDP..." section 2: F = 1 is full replication,
F = N_d is full sharding), the gradient-mean identity of "4.1 数据并行详解"
section 2 on a least-squares model, exact rational means, the nested order,
and a simulated two-level ring that counts the elements it sends."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

SHAPES = [(2, 1), (2, 2), (4, 2), (6, 3), (8, 2), (8, 4), (8, 8), (8, 1), (12, 4)]


def _bf16_contribs(nd, P, seed):
    rng = np.random.default_rng(seed)
    return [oracle.f32_to_bf16((rng.standard_normal(P) * 1e-3).astype(np.float32))
            for _ in range(nd)]


@pytest.mark.parametrize("nd", [1, 2, 4, 8])
def test_full_sharding_factor_is_the_plain_reduce_scatter(nd):
    S = 37
    c = _bf16_contribs(nd, nd * S, nd)
    for r in range(nd):
        assert np.array_equal(oracle.hybrid_rs_avg(c, nd, r, S), oracle.rs_avg(c, r, S))


@pytest.mark.parametrize("nd", [1, 2, 3, 8])
def test_factor_one_is_the_replicated_all_reduce(nd):
    P = 100
    c = _bf16_contribs(nd, P, 10 + nd)
    got = oracle.hybrid_rs_avg(c, 1, 0, P)
    assert np.array_equal(got, oracle.rs_avg(c, 0, P))
    assert np.array_equal(oracle.f32_to_bf16(got), oracle.bucket_allreduce_avg(c, [0, P]))


def _mean_grad(X, y, theta):
    return X.T @ (X @ theta - y) / X.shape[0]


@pytest.mark.parametrize("nd,F", SHAPES)
def test_hybrid_mean_is_the_global_batch_gradient(nd, F):
    rng = np.random.default_rng(nd * 10 + F)
    d = 4 * F
    X = rng.standard_normal((nd * 6, d))
    y = rng.standard_normal(nd * 6)
    theta = rng.standard_normal(d)
    g = _mean_grad(X, y, theta)
    local = [_mean_grad(X[k * 6:(k + 1) * 6], y[k * 6:(k + 1) * 6], theta) for k in range(nd)]
    S = d // F
    got = np.concatenate([oracle.hybrid_rs_avg(local, F, f, S) for f in range(F)])
    assert np.allclose(got, g, rtol=0, atol=1e-12)


def _nearest_f32(q: Fraction):
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda x: (abs(Fraction(float(x)) - q),
                                     int(np.array(x, np.float32).view(np.uint32)) & 1))
    return best


@pytest.mark.parametrize("nd,F", SHAPES)
def test_hybrid_exact_rational_mean(nd, F):
    # 8-bit integers times 2^-4..2^2: every partial sum fits in 24 bits, so
    # the sums are exact and the result is the correctly rounded exact mean
    rng = np.random.default_rng(nd + 100 * F)
    S = 20
    vals = (rng.integers(-255, 256, size=(nd, F * S)) *
            np.exp2(rng.integers(-4, 3, size=(nd, F * S)))).astype(np.float32)
    contribs = [oracle.f32_to_bf16(v) for v in vals]
    for f in range(F):
        got = oracle.hybrid_rs_avg(contribs, F, f, S)
        for i in range(S):
            q = sum(Fraction(float(vals[k, f * S + i])) for k in range(nd)) / nd
            assert got[i] == _nearest_f32(q), (f, i)


def test_nested_order_differs_from_flat_order():
    # (2^24 + 1) + (1 + 1): the group sums are formed first, so the two 1s of
    # the second group survive; the flat left fold loses them
    c = [np.array([v], np.float32) for v in (2.0 ** 24, 1.0, 1.0, 1.0)]
    assert oracle.hybrid_rs_avg(c, 2, 0, 1)[0] == np.float32(4194304.5)
    assert oracle.rs_avg(c, 0, 1)[0] == np.float32(4194304.0)


def test_group_sums_are_formed_inside_each_group_of_f():
    # N_d = 4, F = 2: ranks k = g*F + j, so the groups are {0, 1} and {2, 3}
    # ("PyTorch FSDP..." section 3.3: reduce inside a group, then across).
    # By hand, with fp32 spacing 2 on [2^24, 2^25) and ties to even:
    #   groups {0,1},{2,3}: (2^24 + 1 -> 2^24) + (3 + 2) = 2^24 + 5 -> 2^24 + 4;
    #                       / 4 = 4194305
    #   groups {0,2},{1,3} (ranks grouped across instead):
    #                       (2^24 + 3 -> 2^24 + 4) + (1 + 2) = 2^24 + 7 -> 2^24 + 8;
    #                       / 4 = 4194306
    #   flat left fold:     ((2^24 + 1 -> 2^24) + 3 -> 2^24 + 4) + 2 = 2^24 + 6;
    #                       / 4 = 4194305.5
    c = [np.array([v], np.float32) for v in (2.0 ** 24, 1.0, 3.0, 2.0)]
    assert oracle.hybrid_rs_avg(c, 2, 0, 1)[0] == np.float32(4194305.0)
    assert oracle.rs_avg(c, 0, 1)[0] == np.float32(4194305.5)
    # F = 1: every rank its own group, the groups summed in rank order = flat
    assert oracle.hybrid_rs_avg(c, 1, 0, 1)[0] == np.float32(4194305.5)


def test_hybrid_rejects_a_factor_that_does_not_divide():
    c = _bf16_contribs(6, 12, 0)
    with pytest.raises(ValueError):
        oracle.hybrid_rs_avg(c, 4, 0, 3)


def _ring_rs(bufs, send):
    """Ring reduce-scatter among len(bufs) ranks, each holding len(bufs)
    chunks; returns the chunk each rank ends up owning (summed)."""
    N = len(bufs)
    for step in range(N - 1):
        msgs = []
        for r in range(N):
            k = (r - step) % N
            msgs.append(((r + 1) % N, k, bufs[r][k].copy()))
            send[r] += bufs[r][k].size
        for dst, k, data in msgs:
            bufs[dst][k] = bufs[dst][k] + data
    return [bufs[r][(r + 1) % N] for r in range(N)], [(r + 1) % N for r in range(N)]


def _ring_ag(owned, owner_chunk, N, send):
    """Ring all-gather: every rank ends with every chunk."""
    full = [[None] * N for _ in range(N)]
    for r in range(N):
        full[r][owner_chunk[r]] = owned[r]
    for step in range(N - 1):
        msgs = []
        for r in range(N):
            k = (owner_chunk[r] - step) % N
            msgs.append(((r + 1) % N, k, full[r][k]))
            send[r] += full[r][k].size
        for dst, k, data in msgs:
            full[dst][k] = data
    return full


@pytest.mark.parametrize("nd,F", [(8, 2), (8, 4), (6, 3), (4, 2), (8, 8), (8, 1)])
def test_two_level_ring_traffic_matches_the_hybrid_ledger(nd, F):
    R = nd // F
    psi = nd * F * 6
    rng = np.random.default_rng(nd * 7 + F)
    data = [rng.integers(-50, 50, size=psi) for _ in range(nd)]
    sent = [0] * nd
    S = psi // F
    # 1. reduce-scatter inside each group: rank (g, j) ends with a group sum
    #    of one shard
    shard_of_rank, group_sum = {}, {}
    for g in range(R):
        ranks = [g * F + j for j in range(F)]
        bufs = [np.split(data[k].copy(), F) for k in ranks]
        send = [0] * F
        owned, idx = _ring_rs(bufs, send) if F > 1 else ([bufs[0][0]], [0])
        for j, k in enumerate(ranks):
            shard_of_rank[k] = idx[j]
            group_sum[k] = owned[j]
            sent[k] += send[j]
    # 2. all-reduce of each shard across the R groups (ring RS + AG of the
    #    shard cut in R pieces)
    total_of_rank = {}
    for f in range(F):
        ranks = [k for k in range(nd) if shard_of_rank[k] == f]
        assert len(ranks) == R
        if R > 1:
            bufs = [np.split(group_sum[k].copy(), R) for k in ranks]
            send = [0] * R
            owned, idx = _ring_rs(bufs, send)
            full = _ring_ag(owned, idx, R, send)
            for i, k in enumerate(ranks):
                total_of_rank[k] = np.concatenate(full[i])
                sent[k] += send[i]
        else:
            total_of_rank[ranks[0]] = group_sum[ranks[0]]
    total = np.sum(data, axis=0)
    for k in range(nd):
        f = shard_of_rank[k]
        assert np.array_equal(total_of_rank[k], total[f * S:(f + 1) * S])
    # 3. all-gather of the (updated) shards inside each group
    for g in range(R):
        ranks = [g * F + j for j in range(F)]
        if F > 1:
            send = [0] * F
            full = _ring_ag([total_of_rank[k] for k in ranks], [shard_of_rank[k] for k in ranks],
                            F, send)
            for j, k in enumerate(ranks):
                assert np.array_equal(np.concatenate(full[j]), total)
                sent[k] += send[j]
    want = (oracle.hybrid_comm_bytes_per_gpu(psi, nd, F, "intra", exact=True) +
            oracle.hybrid_comm_bytes_per_gpu(psi, nd, F, "inter", exact=True))
    for k in range(nd):
        assert 2 * sent[k] == pytest.approx(want)  # 16-bit elements


def test_hybrid_ledger_special_cases():
    psi = 7e9
    # F = N_d: the ZeRO-3 ledger and the ZeRO-1/2 communication volume
    assert oracle.hybrid_state_bytes_per_gpu(psi, 8) == oracle.state_bytes_per_gpu(psi, 8, 3)
    assert (oracle.hybrid_comm_bytes_per_gpu(psi, 8, 8, "intra") +
            oracle.hybrid_comm_bytes_per_gpu(psi, 8, 8, "inter")) == oracle.comm_bytes_per_gpu(
                psi, 8, "zero1")
    # F = 1: full replication, the DDP ledger and the DDP all-reduce
    assert oracle.hybrid_state_bytes_per_gpu(psi, 1) == oracle.state_bytes_per_gpu(psi, 8, 0)
    assert oracle.hybrid_comm_bytes_per_gpu(psi, 8, 1, "intra") == 0
    assert oracle.hybrid_comm_bytes_per_gpu(psi, 8, 1, "inter") == oracle.comm_bytes_per_gpu(
        psi, 8, "all_reduce")
    # the traffic leaving a group shrinks by F: 4 Psi / F per GPU
    assert oracle.hybrid_comm_bytes_per_gpu(psi, 16, 8, "inter") == pytest.approx(4 * psi / 8)
    with pytest.raises(ValueError):
        oracle.hybrid_comm_bytes_per_gpu(psi, 8, 3, "intra")
