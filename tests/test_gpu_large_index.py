"""GPU parity past 2^31 elements: every streaming entry point on a range
longer than a signed 32-bit index can address, so that an index or an offset
held in 32 bits anywhere on the path would show up as a wrong or missing
element.  The oracle computes sampled outputs one by one from the same
seeded inputs: the first and last elements, a band around element 2^31 (and
around byte 2^32 of the fp32 arrays), and random positions; properties that
hold at any size (the zero padding, the found-inf flag) cover the rest.
About 60 GB of device memory at most, released after each test."""
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
BIG = (1 << 31) + 13                 # elements: past the signed 32-bit range
HP = AdamWConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HPC = ss.AdamW(lr=HP.lr, beta1=HP.beta1, beta2=HP.beta2, eps=HP.eps, weight_decay=HP.weight_decay)
SEED = 31


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()
    yield
    torch.cuda.empty_cache()
    assert ss.device_status() == 0


@pytest.fixture(autouse=True)
def _release():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(params=["auto", "tma"])
def path(request):
    prev = ss.set_fused_path(request.param)
    yield request.param
    ss.set_fused_path(prev)


def _sample(n, seed=0):
    """Indices to check: both ends, bands around 2^30, 2^31 and 2^32 / 4
    (byte 2^32 of an fp32 array), and 4096 random positions."""
    rng = np.random.default_rng(seed)
    idx = set(int(i) for i in rng.integers(0, n, size=4096))
    for c in (0, 1 << 30, 1 << 31, n):
        idx.update(i for i in range(c - 64, c + 64) if 0 <= i < n)
    return np.array(sorted(idx), dtype=np.int64)


def _at(t, idx):
    return t[torch.from_numpy(idx).to(t.device)]


def _bits16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _stream(*fields, sigma=1e-3):
    return synth.normal_stream(SEED, fields, sigma)


def test_fused_step_past_2_31(path):
    nd, S = 2, BIG
    grads = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    master = torch.empty(S, dtype=torch.float32, device=DEV)
    synth.dev_fill(_stream(1, 0, sigma=0.02), master)
    m = torch.zeros(S, dtype=torch.float32, device=DEV)
    v = torch.zeros(S, dtype=torch.float32, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    idx = _sample(S)
    p = synth.host_gather(_stream(1, 0, sigma=0.02), idx, "f32")
    mh = np.zeros(idx.size, np.float32)
    vh = np.zeros(idx.size, np.float32)
    for t in (1, 2):                   # step 2 reads non-zero moments
        for q in range(nd):
            synth.dev_fill(_stream(2, t, q), grads[q])
        ss.fsdp_rs_avg_adamw_cast(grads, master, m, v, out, HPC, t)
        contribs = [synth.host_gather(_stream(2, t, q), idx, "bf16") for q in range(nd)]
        p, mh, vh, ob = oracle.fsdp_shard_step(contribs, 0, idx.size, p, mh, vh, HP, t)
    torch.cuda.synchronize()
    assert_bits(_at(master, idx).cpu().numpy(), p, "master")
    assert_bits(_at(m, idx).cpu().numpy(), mh, "m")
    assert_bits(_at(v, idx).cpu().numpy(), vh, "v")
    assert_bits(_bits16(_at(out, idx)), ob, "bf16")


def test_accumulate_past_2_31(path):
    n, M = BIG, 2
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    acc = torch.empty(n, dtype=torch.float32, device=DEV)
    idx = _sample(n, 1)
    for j in range(M):
        synth.dev_fill(_stream(3, j), g)
        ss.fsdp_grad_accumulate(g, acc, 1.0 / M, j == 0)
    want = oracle.grad_accumulate([synth.host_gather(_stream(3, j), idx, "bf16")
                                   for j in range(M)], np.float32(1.0 / M))
    torch.cuda.synchronize()
    assert_bits(_at(acc, idx).cpu().numpy(), want, "accumulator")


def test_bucket_allreduce_past_2_31(path):
    nd, n = 2, BIG
    grads = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    for q in range(nd):
        synth.dev_fill(_stream(4, q), grads[q])
    out = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    idx = _sample(n, 2)
    contribs = [synth.host_gather(_stream(4, q), idx, "bf16") for q in range(nd)]
    want = oracle.bucket_allreduce_avg(contribs, [0, idx.size])
    # one bucket over the whole range, then buckets split at 2^30 and 2^31 + 1
    for boff in ([0, n], [0, 1 << 30, (1 << 31) + 1, n]):
        out.zero_()
        ss.ddp_bucket_allreduce_avg(grads, boff, out)
        torch.cuda.synchronize()
        assert_bits(_bits16(_at(out, idx)), want, f"all-reduce {boff}")


def test_nonfinite_check_past_2_31(path):
    nd, S = 2, BIG
    grads = [torch.empty(S, dtype=torch.float16, device=DEV) for _ in range(nd)]
    for q in range(nd):
        synth.dev_fill(_stream(5, q), grads[q])
    sc = ss.GradScaler(1.0, device=DEV)
    sc.check(grads)
    torch.cuda.synchronize()
    assert int(sc.found_inf.item()) == 0
    # one inf past element 2^31 is found
    grads[1][(1 << 31) + 5] = float("inf")
    sc.check(grads)
    torch.cuda.synchronize()
    assert int(sc.found_inf.item()) == 1
    # and one in the last element
    sc.found_inf.zero_()
    grads[1][(1 << 31) + 5] = 0.0
    grads[0][S - 1] = float("nan")
    sc.check(grads)
    torch.cuda.synchronize()
    assert int(sc.found_inf.item()) == 1


def test_flat_pack_and_ag_unpack_past_2_31(path):
    """One unit of two tensors whose padded length is past 2^31 elements on
    two ranks: pack, all-gather of the two shards, views."""
    numels = [(1 << 30) + 7, (1 << 30) + 2]
    lay = oracle.layout(numels, 2)
    assert lay.padded > (1 << 31) and lay.padded - lay.total == 1
    tensors = [torch.empty(k, dtype=torch.bfloat16, device=DEV) for k in numels]
    for i, t in enumerate(tensors):
        synth.dev_fill(_stream(6, i), t)
    flat = ss.fsdp_flat_pack(tensors, 2)
    S = lay.shard
    shards = [flat[:S].clone(), flat[S:].clone()]
    del flat
    torch.cuda.empty_cache()
    full = torch.empty(2 * S, dtype=torch.bfloat16, device=DEV)
    full.fill_(1.0)
    ss.fsdp_ag_unpack(shards, full)
    views = ss.fsdp_views(full, [(k,) for k in numels], 2)
    torch.cuda.synchronize()
    assert int(_bits16(full[lay.padded - 1:])[0]) == 0          # the padding
    for i, (vw, k) in enumerate(zip(views, numels)):
        idx = _sample(k, 3 + i)
        assert_bits(_bits16(_at(vw, idx)), synth.host_gather(_stream(6, i), idx, "bf16"),
                    f"tensor {i}")


def test_fused_last_micro_batch_past_2_31(path):
    """The last micro-batch accumulated inside the fused step over 2^31 + 13
    elements: fp32 accumulators of micro-batches 0..M-2 and the last bf16
    gradient per contribution; the accumulators are read, not written."""
    nd, S, M = 2, BIG, 2
    acc = [torch.empty(S, dtype=torch.float32, device=DEV) for _ in range(nd)]
    last = [torch.empty(S, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    g = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    for q in range(nd):
        synth.dev_fill(_stream(7, q, 0), g)
        ss.fsdp_grad_accumulate(g, acc[q], 1.0 / M, True)
        synth.dev_fill(_stream(7, q, 1), last[q])
    del g
    master = torch.empty(S, dtype=torch.float32, device=DEV)
    synth.dev_fill(_stream(8, 0, sigma=0.02), master)
    m = torch.zeros(S, dtype=torch.float32, device=DEV)
    v = torch.zeros(S, dtype=torch.float32, device=DEV)
    out = torch.empty(S, dtype=torch.bfloat16, device=DEV)
    ss.fsdp_accumulate_rs_avg_adamw_cast(acc, last, 1.0 / M, master, m, v, out, HPC, 1)
    idx = _sample(S, 4)
    micro = [[synth.host_gather(_stream(7, q, j), idx, "bf16") for j in range(M)]
             for q in range(nd)]
    contribs = [oracle.grad_accumulate(micro[q], np.float32(1.0 / M)) for q in range(nd)]
    z = np.zeros(idx.size, np.float32)
    p, mh, vh, ob = oracle.fsdp_shard_step(contribs, 0, idx.size,
                                           synth.host_gather(_stream(8, 0, sigma=0.02), idx, "f32"),
                                           z, z, HP, 1)
    torch.cuda.synchronize()
    assert_bits(_at(master, idx).cpu().numpy(), p, "master")
    assert_bits(_at(m, idx).cpu().numpy(), mh, "m")
    assert_bits(_at(v, idx).cpu().numpy(), vh, "v")
    assert_bits(_bits16(_at(out, idx)), ob, "bf16")
    for q in range(nd):
        assert_bits(_at(acc[q], idx).cpu().numpy(),
                    oracle.grad_accumulate(micro[q][:1], np.float32(1.0 / M)), f"accumulator {q}")


def test_fused_ddp_step_past_2_31(path):
    nd, n = 2, BIG
    grads = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    for q in range(nd):
        synth.dev_fill(_stream(9, q), grads[q])
    master = torch.empty(n, dtype=torch.float32, device=DEV)
    synth.dev_fill(_stream(10, 0, sigma=0.02), master)
    m = torch.zeros(n, dtype=torch.float32, device=DEV)
    v = torch.zeros(n, dtype=torch.float32, device=DEV)
    pb = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    mean = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    # buckets split at 2^30 and 2^31 + 1, all in one call (one launch)
    ss.ddp_bucket_allreduce_avg_adamw_cast(grads, [0, 1 << 30, (1 << 31) + 1, n], master, m, v,
                                           pb, HPC, 1, mean_out=mean)
    idx = _sample(n, 5)
    contribs = [synth.host_gather(_stream(9, q), idx, "bf16") for q in range(nd)]
    z = np.zeros(idx.size, np.float32)
    avg, p, mh, vh, ob = oracle.ddp_step(contribs, [0, idx.size],
                                         synth.host_gather(_stream(10, 0, sigma=0.02), idx, "f32"),
                                         z, z, HP, 1)
    torch.cuda.synchronize()
    assert_bits(_bits16(_at(mean, idx)), avg, "mean")
    assert_bits(_at(master, idx).cpu().numpy(), p, "master")
    assert_bits(_at(m, idx).cpu().numpy(), mh, "m")
    assert_bits(_at(v, idx).cpu().numpy(), vh, "v")
    assert_bits(_bits16(_at(pb, idx)), ob, "params")

