"""The host-side planners of the C ABI against the oracle on random inputs,
with element counts up to 2^40 and N_d up to 64 where the oracle's planner
is arithmetic (the FlatParameter layout, the FSDP2 layout, the DDP bucket
plan), and on random small units for the checkpoint reshard plan, whose
oracle walks every element.  CPU only."""
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
