"""DDP bucket readiness on the host ("4.1 数据并行详解", DDP section on
buckets: a bucket is reduced once all its gradients are ready, and a
parameter that never gets a gradient leaves its bucket waiting -- the hang
find_unused_parameters exists for).  The emulated ranks are host threads;
the failure is injected on the host (a rank that never marks a parameter),
never on a GPU."""
import threading
import time

import pytest

import oracle
import sharded_optimizer_step_gb300 as ss
from sharded_optimizer_step_gb300 import _capi

NUMELS = [768, 768, 768 * 3072, 768 * 3072, 4096 * 4096] * 3 + [768 * 3072]


def _plan(cap_mib=25):
    off, bucket_of, boff = ss.ddp_bucket_plan(NUMELS, 2, cap_mib << 20)
    return bucket_of, len(boff) - 1


def _run_ranks(ready, nd, skip=None, order=None):
    """Each rank marks every parameter in reverse registration order (the
    order backward produces them), except the (rank, param) in `skip`.
    Returns the completions each thread saw."""
    seen = [[] for _ in range(nd)]
    n = len(NUMELS)

    def rank(r):
        for i in (order or list(reversed(range(n)))):
            if skip == (r, i):
                continue
            b = ready.mark(r, i)
            if b is not None:
                seen[r].append(b)
            time.sleep(0.0002)

    ts = [threading.Thread(target=rank, args=(r,)) for r in range(nd)]
    for t in ts:
        t.start()
    return ts, seen


def test_every_bucket_completes_once_when_all_ranks_mark_everything():
    bucket_of, nb = _plan()
    nd = 8
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    ts, seen = _run_ranks(ready, nd)
    # the waiter takes buckets in bucket order while ranks are still marking
    for b in range(nb):
        ready.wait(b, timeout_s=10.0)
    for t in ts:
        t.join()
    completed = sorted(b for s in seen for b in s)
    assert completed == list(range(nb))          # each bucket reported exactly once


def test_withheld_gradient_times_out_naming_rank_and_param():
    bucket_of, nb = _plan()
    nd = 4
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    victim = (2, 7)                               # rank 2 never produces param 7's gradient
    ts, _ = _run_ranks(ready, nd, skip=victim)
    for t in ts:
        t.join()
    bad = bucket_of[victim[1]]
    for b in range(nb):
        if b == bad:
            t0 = time.monotonic()
            with pytest.raises(ss.BucketNotReady) as e:
                ready.wait(b, timeout_s=0.2)
            assert 0.2 <= time.monotonic() - t0 < 5.0
            assert (e.value.bucket, e.value.rank, e.value.param) == (bad, 2, 7)
            assert "rank 2 never marked param 7" in str(e.value)
        else:
            ready.wait(b, timeout_s=1.0)          # every other bucket is complete


def test_waiter_learns_of_a_rank_that_never_joins():
    bucket_of, nb = _plan()
    nd = 3
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    # ranks 0 and 1 run; rank 2 never starts
    for r in (0, 1):
        for i in range(len(NUMELS)):
            ready.mark(r, i)
    with pytest.raises(ss.BucketNotReady) as e:
        ready.wait(0, timeout_s=0.05)
    assert e.value.rank == 2


def test_reset_starts_the_next_iteration():
    bucket_of, nb = _plan()
    nd = 2
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    for r in range(nd):
        for i in range(len(NUMELS)):
            ready.mark(r, i)
    ready.wait(0, 0.1)
    ready.reset()
    with pytest.raises(ss.BucketNotReady):
        ready.wait(0, 0.01)
    for r in range(nd):
        for i in range(len(NUMELS)):
            ready.mark(r, i)
    for b in range(nb):
        ready.wait(b, 0.1)


def test_bucket_completion_matches_the_plan():
    """A bucket completes exactly when its last (rank, parameter) mark
    arrives: marking parameters in registration order completes the buckets
    in the order of their last parameter, as the oracle's plan puts them."""
    nd = 2
    _, bucket_of, boff = oracle.bucket_plan(NUMELS, 2, 25 << 20)
    nb = len(boff) - 1
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    done = []
    for i in range(len(NUMELS)):
        for r in range(nd):
            b = ready.mark(r, i)
            if b is not None:
                done.append((i, b))
    last = {}
    for i, b in enumerate(bucket_of):
        last[b] = i
    assert sorted(done) == sorted((i, b) for b, i in last.items())


def test_invalid_uses_are_refused():
    bucket_of, nb = _plan()
    ready = ss.BucketReadiness(bucket_of, nb, 2)
    ready.mark(0, 0)
    with pytest.raises(_capi.ShardstepError):
        ready.mark(0, 0)                          # twice
    with pytest.raises(_capi.ShardstepError):
        ready.mark(2, 0)                          # no such rank
    with pytest.raises(_capi.ShardstepError):
        ready.mark(0, len(NUMELS))                # no such parameter
    with pytest.raises(_capi.ShardstepError):
        ready.wait(nb, 0.01)                      # no such bucket
    L = _capi.lib()
    assert L.ddp_ready_bytes(4, 0, 2) == -1
    assert L.ddp_ready_bytes(4, 2, 0) == -1
    assert L.ddp_ready_bytes(4, 2, 2) > 0
    import ctypes
    small = (ctypes.c_uint64 * 2)()
    bop = (ctypes.c_int32 * 4)(0, 0, 1, 1)
    assert L.ddp_ready_init(ctypes.addressof(small), 16, bop, 4, 2, 2) == _capi.ERR_CAPACITY
    big = (ctypes.c_uint64 * 64)()
    bad = (ctypes.c_int32 * 4)(0, 0, 1, 2)
    assert L.ddp_ready_init(ctypes.addressof(big), 512, bad, 4, 2, 2) == _capi.ERR_INVALID
    assert L.ddp_ready_mark(None, 0, 0, None) == _capi.ERR_INVALID
