"""DDP buckets reduced as they become ready, on the GPU: N_d rank threads
write their gradients (each on its own CUDA stream) parameter by parameter
in backward order and mark them; the caller all-reduces each bucket once
every rank has marked it.  A rank that withholds one gradient stops the
launches at that bucket with a host-side timeout -- no kernel waits for it --
and the device stays usable."""
import threading

import numpy as np
import pytest
import torch

import oracle
import sharded_optimizer_step_gb300 as ss
import synth
from tests._cmp import assert_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NUMELS = [768, 768, 768 * 3072, 768 * 3072, 1024 * 1024, 5, 768 * 3072, 4096]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    assert ss.device_status() == 0


def _stream(r, i):
    return synth.normal_stream(31, (88, r, i), 1e-3)


def _setup(nd, cap_bytes):
    off, bucket_of, boff = ss.ddp_bucket_plan(NUMELS, 2, cap_bytes)
    total = boff[-1]
    grads = [torch.full((total,), float("nan"), dtype=torch.bfloat16, device=DEV)
             for _ in range(nd)]
    return off, bucket_of, boff, total, grads


def _ranks(nd, off, grads, ready, skip=None):
    errors = []

    def rank(r):
        try:
            s = torch.cuda.Stream(device=DEV)
            with torch.cuda.stream(s):
                for i in reversed(range(len(NUMELS))):
                    if (r, i) == skip:
                        continue
                    synth.dev_fill(_stream(r, i), grads[r][off[i]:off[i] + NUMELS[i]])
                    s.synchronize()            # the gradient is in memory before it is marked
                    ready.mark(r, i)
        except Exception as e:                 # surfaced by the test below
            errors.append(e)

    ts = [threading.Thread(target=rank, args=(r,)) for r in range(nd)]
    for t in ts:
        t.start()
    return ts, errors


def _host_grads(nd, off, total):
    out = []
    for r in range(nd):
        h = np.zeros(total, np.uint16)
        for i, n in enumerate(NUMELS):
            h[off[i]:off[i] + n] = synth.host_fill(_stream(r, i), 0, n, "bf16")
        out.append(h)
    return out


@pytest.mark.parametrize("cap_mib", [1, 4])
def test_buckets_reduced_as_they_become_ready(cap_mib):
    nd = 4
    off, bucket_of, boff, total, grads = _setup(nd, cap_mib << 20)
    ready = ss.BucketReadiness(bucket_of, len(boff) - 1, nd)
    out = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    ts, errors = _ranks(nd, off, grads, ready)
    ss.ddp_allreduce_as_ready(grads, boff, out, ready, timeout_s=60.0)
    for t in ts:
        t.join()
    assert not errors
    want = oracle.bucket_allreduce_avg(_host_grads(nd, off, total), boff)
    torch.cuda.synchronize()
    assert_bits(out.view(torch.int16).cpu().numpy().view(np.uint16), want, "avg")


def test_withheld_gradient_stops_at_its_bucket_and_the_device_stays_usable():
    nd = 4
    off, bucket_of, boff, total, grads = _setup(nd, 4 << 20)
    nb = len(boff) - 1
    victim = (1, 3)
    bad = bucket_of[victim[1]]
    ready = ss.BucketReadiness(bucket_of, nb, nd)
    out = torch.full((total,), 7.0, dtype=torch.bfloat16, device=DEV)
    ts, errors = _ranks(nd, off, grads, ready, skip=victim)
    for t in ts:
        t.join()
    assert not errors
    with pytest.raises(ss.BucketNotReady) as e:
        ss.ddp_allreduce_as_ready(grads, boff, out, ready, timeout_s=0.5)
    assert (e.value.bucket, e.value.rank, e.value.param) == (bad, 1, 3)
    torch.cuda.synchronize()
    host = _host_grads(nd, off, total)
    want = oracle.bucket_allreduce_avg(host, boff)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(nb):
        a, z = boff[b], boff[b + 1]
        if b < bad:                                  # reduced before the stop
            assert_bits(got[a:z], want[a:z], f"bucket {b}")
        else:                                        # never launched
            assert (got[a:z] == np.uint16(0x40E0)).all(), b
    # the device still works: the later complete buckets reduce normally
    for b in range(bad + 1, nb):
        ready.wait(b, 1.0)
        ss.ddp_bucket_allreduce_avg(grads, boff, out, first=b, count=1)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(bad + 1, nb):
        a, z = boff[b], boff[b + 1]
        assert_bits(got[a:z], want[a:z], f"bucket {b} after the stop")
    assert ss.device_status() == 0
