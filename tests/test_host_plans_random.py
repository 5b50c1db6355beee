"""The host-side planners of the C ABI against the oracle on random inputs,
with element counts up to 2^40 and N_d up to 64 where the oracle's planner
is arithmetic (the FlatParameter layout, the FSDP2 layout, the DDP bucket
plan), and on random small units for the checkpoint reshard plan, whose
oracle walks every element; the memory and communication ledgers, plain and
hybrid, on random Psi up to 2^44.  CPU only."""
import pytest

import oracle
import sharded_optimizer_step_gb300 as ss
from oracle import checkpoint as ock
from sharded_optimizer_step_gb300 import checkpoint as ck

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings, example = hyp.given, hyp.settings, hyp.example

BIG = 1 << 40
ND = st.integers(min_value=1, max_value=ss.MAX_ND)
# element counts from empty through small to very large
NUMEL = st.one_of(st.integers(0, 8), st.integers(0, 1 << 20), st.integers(0, BIG))


@pytest.fixture(scope="module", autouse=True)
def built():
    ss.build()


@settings(max_examples=300, deadline=None)
@given(numels=st.lists(NUMEL, max_size=8), nd=ND)
@example(numels=[BIG, BIG - 1, 3, 0, (1 << 31) + 13], nd=ss.MAX_ND)
@example(numels=[(1 << 31) - 1, 1, 1], nd=63)
def test_flat_layout(numels, nd):
    a = ss.fsdp_layout(numels, nd)
    b = oracle.layout(numels, nd)
    assert (a.total, a.padded, a.shard) == (b.total, b.padded, b.shard)
    assert a.offsets == b.offsets
    assert a.lo == b.lo and a.hi == b.hi


@settings(max_examples=300, deadline=None)
@given(shapes=st.lists(st.one_of(st.tuples(st.integers(1, 1 << 24)),
                                 st.tuples(st.integers(1, 1 << 20), st.integers(0, 1 << 16)),
                                 st.tuples(st.integers(0, 64), st.integers(1, 64),
                                           st.integers(1, 64))),
                       min_size=1, max_size=6),
       nd=ND)
@example(shapes=[(11008, 4096), (4096,), ((1 << 24) - 1, 1 << 16)], nd=ss.MAX_ND)
def test_fsdp2_layout(shapes, nd):
    a = ss.fsdp2_layout(shapes, nd)
    b = oracle.fsdp2_layout(shapes, nd)
    assert (a.chunk, a.offset, a.local) == (b.chunk, b.offset, b.local)


@settings(max_examples=300, deadline=None)
@given(numels=st.lists(NUMEL, max_size=10), es=st.sampled_from([1, 2, 4]),
       cap=st.one_of(st.integers(1, 1 << 12), st.integers(1, 1 << 40)))
@example(numels=[BIG, 1, 0, 25 << 20, (25 << 20) + 1], es=2, cap=25 << 20)
def test_ddp_bucket_plan(numels, es, cap):
    assert ss.ddp_bucket_plan(numels, es, cap) == tuple(
        list(x) for x in oracle.bucket_plan(numels, es, cap))


@settings(max_examples=300, deadline=None)
@given(total=st.integers(0, 200_000), old_nd=ND, new_nd=ND, data=st.data())
def test_reshard_plan(total, old_nd, new_nd, data):
    rank = data.draw(st.integers(0, new_nd - 1))
    assert ck.plan(total, old_nd, new_nd, rank) == ock.plan(total, old_nd, new_nd, rank)


PSI = st.one_of(st.integers(1, 1 << 20), st.integers(1, 1 << 44)).map(float)


@settings(max_examples=300, deadline=None)
@given(psi=PSI, nd=ND, stage=st.integers(0, 3),
       kind=st.sampled_from(["reduce_scatter", "all_gather", "all_reduce", "zero1", "zero2",
                             "zero3"]),
       exact=st.booleans())
def test_memory_and_communication_ledger(psi, nd, stage, kind, exact):
    assert ss.state_bytes(psi, nd, stage) == pytest.approx(
        oracle.state_bytes_per_gpu(psi, nd, stage), rel=1e-15)
    assert ss.comm_bytes(psi, nd, kind, exact) == pytest.approx(
        oracle.comm_bytes_per_gpu(psi, nd, kind, exact), rel=1e-15)


@settings(max_examples=300, deadline=None)
@given(psi=PSI, groups=st.integers(1, 16), F=st.integers(1, 16),
       kind=st.sampled_from(["intra", "inter"]), exact=st.booleans())
def test_hybrid_ledger(psi, groups, F, kind, exact):
    nd = groups * F
    if nd > ss.MAX_ND:
        return
    assert ss.hybrid_state_bytes(psi, F) == pytest.approx(
        oracle.hybrid_state_bytes_per_gpu(psi, F), rel=1e-15)
    assert ss.hybrid_comm_bytes(psi, nd, F, kind, exact) == pytest.approx(
        oracle.hybrid_comm_bytes_per_gpu(psi, nd, F, kind, exact), rel=1e-15, abs=0)
