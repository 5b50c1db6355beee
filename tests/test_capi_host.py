"""CPU checks of the C ABI: the library loads, exports every symbol the
header declares, and its host-only entry points (layout, views, bucket plan,
ledger, argument validation) agree with the oracle.  No call here reaches the
GPU: validation rejects the arguments before any launch."""
import ctypes
import itertools
import os
import random
import re

import numpy as np
import pytest

import oracle
import sharded_optimizer_step_gb300 as ss
from sharded_optimizer_step_gb300 import _capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    ss.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "shardstep.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(_capi.lib_path())
    for n in names:
        assert hasattr(lib, n), n
    # and the binding declares exactly these
    assert sorted(_capi.SIGNATURES) == names


def _layout_matches(numels, nd):
    a = ss.fsdp_layout(numels, nd)
    b = oracle.layout(numels, nd)
    assert (a.total, a.padded, a.shard) == (b.total, b.padded, b.shard)
    assert a.offsets == b.offsets
    assert a.lo == b.lo and a.hi == b.hi


def test_layout_matches_oracle_brute_force():
    for K in range(0, 4):
        for numels in itertools.product(range(0, 6), repeat=K):
            for nd in range(1, 6):
                _layout_matches(list(numels), nd)


def test_layout_matches_oracle_on_model_units():
    gpt2_block = [768 * 2304, 2304, 768 * 768, 768, 768 * 3072, 3072, 3072 * 768, 768,
                  768, 768, 768, 768]
    llama_layer = [2048 * 2048] * 4 + [2048 * 8192] * 2 + [8192 * 2048] + [2048, 2048]
    for unit, nd in ((gpt2_block, 8), (llama_layer, 8), ([1024 * 1024, 1024 * 4096, 4096 * 1024], 4),
                     ([5, 7, 11, 3], 6), ([1], 64)):
        _layout_matches(unit, nd)


def test_worked_example_views_through_the_abi():
    # three (4,2) tensors on two ranks: pieces (count) per rank
    shapes = [(4, 2)] * 3
    numels = [8, 8, 8]
    base = 0x10000
    for r, want in ((0, [8, 4, 0]), (1, [0, 4, 8])):
        ptrs = (_capi.c_vp * 3)()
        counts = (_capi.c_i64 * 3)()
        _capi.check("fsdp_views", _capi.lib().fsdp_views(
            _capi.i64_array(numels), 3, 2, r, ctypes.c_void_p(base), 2, ptrs, counts))
        assert list(counts) == want
        lay = oracle.layout(numels, 2)
        for t in range(3):
            assert (ptrs[t] or 0) == base + 2 * lay.lo[r][t]
    ptrs = (_capi.c_vp * 3)()
    counts = (_capi.c_i64 * 3)()
    _capi.check("fsdp_views", _capi.lib().fsdp_views(
        _capi.i64_array(numels), 3, 2, -1, ctypes.c_void_p(base), 2, ptrs, counts))
    assert [p - base for p in ptrs] == [0, 16, 32] and list(counts) == [8, 8, 8]
    del shapes


def test_bucket_plan_matches_oracle():
    rng = random.Random(3)
    for _ in range(300):
        n = rng.randrange(0, 12)
        numels = [rng.choice([0, 1, 3, 768, 2048, 5000]) for _ in range(n)]
        es = rng.choice([1, 2, 4])
        cap = rng.choice([1, 100, 4096, 10000, 1 << 20])
        assert ss.ddp_bucket_plan(numels, es, cap) == tuple(
            list(x) for x in oracle.bucket_plan(numels, es, cap))


def test_bucket_plan_sweep_workload():
    unit = [768, 768, 768 * 3072, 768 * 3072, 4096 * 4096]
    numels = unit * 16 + [768 * 3072] * 3
    assert sum(numels) == 351_035_392
    for mib in (1, 4, 25, 64, 256):
        got = ss.ddp_bucket_plan(numels, 2, mib << 20)
        want = oracle.bucket_plan(numels, 2, mib << 20)
        assert got == tuple(list(x) for x in want)
        assert got[2][-1] == sum(numels)


def test_ledger_matches_oracle():
    for psi in (7e9, 1.2e9, 351e6):
        for nd in (1, 2, 4, 8, 16):
            for stage in range(4):
                assert ss.state_bytes(psi, nd, stage) == pytest.approx(
                    oracle.state_bytes_per_gpu(psi, nd, stage), rel=1e-15)
            for kind in ("reduce_scatter", "all_gather", "all_reduce", "zero1", "zero2", "zero3"):
                for exact in (False, True):
                    assert ss.comm_bytes(psi, nd, kind, exact) == pytest.approx(
                        oracle.comm_bytes_per_gpu(psi, nd, kind, exact), rel=1e-15)
    with pytest.raises(ValueError):
        ss.state_bytes(1e9, 8, 4)


def _fused(slices, nd, S, master, m, v, out, dtype=_capi.DTYPE_BF16, step=1):
    hp = _capi.AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01, step)
    return _capi.lib().fsdp_rs_avg_adamw_cast(_capi.ptr_array(slices), dtype, nd, S,
                                              ctypes.c_void_p(master), ctypes.c_void_p(m),
                                              ctypes.c_void_p(v), ctypes.c_void_p(out),
                                              ctypes.byref(hp), None)


def test_fused_step_rejects_bad_arguments_before_launch():
    L = _capi.lib()
    S = 1024
    A = 1 << 40  # fake device addresses, never dereferenced: validation fails first
    g = [A + k * (1 << 20) for k in range(8)]
    st = [A + (1 << 30) + k * (1 << 20) for k in range(4)]
    assert _fused(g, 0, S, *st) == _capi.ERR_INVALID
    assert _fused(g * 9, 65, S, *st) == _capi.ERR_CAPACITY
    assert _fused(g, 8, S, *st, step=0) == _capi.ERR_INVALID
    assert _fused(g, 8, S, *st, dtype=7) == _capi.ERR_INVALID
    assert _fused(g, 8, -1, *st) == _capi.ERR_INVALID
    assert _fused(g[:7] + [0], 8, S, *st) == _capi.ERR_INVALID          # NULL slice
    assert _fused(g, 8, S, st[0], st[0] + 8, st[2], st[3]) == _capi.ERR_INVALID  # m overlaps master
    assert _fused(g[:7] + [st[3]], 8, S, *st) == _capi.ERR_INVALID      # grad overlaps output
    assert _fused(g, 8, S, st[0] + 2, st[1], st[2], st[3]) == _capi.ERR_INVALID  # misaligned fp32
    assert "misaligned" in L.shardstep_last_error().decode()
    assert _fused(g, 8, 0, *st) == _capi.OK                             # nothing to do


def test_accumulate_step_rejects_bad_arguments_before_launch():
    L = _capi.lib()
    S = 1024
    A = 1 << 40  # fake device addresses, never dereferenced: validation fails first
    acc = [A + k * (1 << 20) for k in range(8)]
    last = [A + (1 << 28) + k * (1 << 20) for k in range(8)]
    st = [A + (1 << 30) + k * (1 << 20) for k in range(4)]

    def call(acc, last, nd, S, *state, step=1):
        hp = ss.AdamW().at_step(step)
        return L.fsdp_accumulate_rs_avg_adamw_cast(
            _capi.ptr_array(acc), _capi.ptr_array(last), nd, nd, S, ctypes.c_float(0.25),
            *[ctypes.c_void_p(a) for a in state], ctypes.byref(hp), None)

    assert call(acc, last, 0, S, *st) == _capi.ERR_INVALID
    assert call(acc * 9, last * 9, 65, S, *st) == _capi.ERR_CAPACITY
    assert call(acc, last, 8, S, *st, step=0) == _capi.ERR_INVALID
    assert call(acc, last, 8, -1, *st) == _capi.ERR_INVALID
    assert call(acc[:7] + [0], last, 8, S, *st) == _capi.ERR_INVALID       # NULL accumulator
    assert call(acc, last[:7] + [0], 8, S, *st) == _capi.ERR_INVALID       # NULL last slice
    assert call(acc, last[:7] + [st[3]], 8, S, *st) == _capi.ERR_INVALID   # input overlaps out
    assert "overlaps" in L.shardstep_last_error().decode()
    assert call(acc[:7] + [st[1]], last, 8, S, *st) == _capi.ERR_INVALID   # acc overlaps m
    assert call(acc, last, 8, S, st[0], st[0] + 8, st[2], st[3]) == _capi.ERR_INVALID
    assert call(acc[:7] + [acc[7] + 2], last, 8, S, *st) == _capi.ERR_INVALID  # misaligned fp32
    assert call(acc, last, 8, 0, *st) == _capi.OK                           # nothing to do
    sp = [ctypes.c_void_p(a) for a in st]
    assert L.fsdp_state_accumulate_rs_avg_adamw_cast(
        _capi.ptr_array(acc), _capi.ptr_array(last), 8, 8, S, ctypes.c_float(0.25), *sp, None,
        None) == _capi.ERR_INVALID
    assert "state is NULL" in L.shardstep_last_error().decode()
    assert L.fsdp_state_accumulate_rs_avg_adamw_cast(
        _capi.ptr_array(acc), _capi.ptr_array(last), 8, 8, S, ctypes.c_float(0.25), *sp,
        ctypes.c_void_p(A + 4), None) == _capi.ERR_INVALID
    assert "misaligned" in L.shardstep_last_error().decode()
    hp = ss.AdamW().at_step(1)
    assert L.fsdp_accumulate_rs_avg_adamw_cast(
        _capi.ptr_array(acc), _capi.ptr_array(last), 8, 3, S, ctypes.c_float(0.25), *sp,
        ctypes.byref(hp), None) == _capi.ERR_INVALID       # 3 does not divide 8
    assert "sharding factor" in L.shardstep_last_error().decode()


def test_other_entry_points_reject_bad_arguments():
    L = _capi.lib()
    A = 1 << 40
    assert L.fsdp_ag_unpack(_capi.ptr_array([A, A + 3000]), 2, 1024, ctypes.c_void_p(A + 2048),
                            None) == _capi.ERR_INVALID    # shard overlaps full
    assert L.fsdp_ag_unpack(_capi.ptr_array([A]), 0, 16, ctypes.c_void_p(A), None) == \
        _capi.ERR_INVALID
    assert L.fsdp_grad_accumulate(ctypes.c_void_p(A), ctypes.c_void_p(A + 8), 64,
                                  ctypes.c_float(0.25), 1, None) == _capi.ERR_INVALID
    assert L.fsdp_flat_pack(_capi.ptr_array([A]), _capi.i64_array([16]), 1, 2, 9,
                            ctypes.c_void_p(A + 4096), None) == _capi.ERR_INVALID
    assert L.fsdp_flat_pack(_capi.ptr_array([A]), _capi.i64_array([16]), 1, 2,
                            _capi.DTYPE_BF16, ctypes.c_void_p(A + 8), None) == _capi.ERR_INVALID
    boff = _capi.i64_array([0, 10, 5])
    assert L.ddp_bucket_allreduce_avg(_capi.ptr_array([A, A + 4096]), 2, boff, 0, 2,
                                      ctypes.c_void_p(A + 8192), None) == _capi.ERR_INVALID
    assert L.ddp_bucket_plan(_capi.i64_array([1]), 1, 2, 0, (_capi.c_i64 * 1)(),
                             (_capi.c_i32 * 1)(), (_capi.c_i64 * 2)(),
                             ctypes.byref(_capi.c_i32())) == _capi.ERR_INVALID
    with pytest.raises(ss.ShardstepError):
        ss.fsdp_layout([3, -1], 2)


def test_empty_calls_return_ok_with_null_data_pointers():
    """A call with no element to process returns OK once its scalar
    arguments are valid, whatever its data pointers (here NULL); with an
    element to process, a NULL output is rejected.  None of these calls
    reaches a launch."""
    L = _capi.lib()
    hp = ss.AdamW().at_step(1)
    nul = ctypes.c_void_p(None)
    nulls = _capi.ptr_array([0, 0, 0])
    assert L.fsdp_rs_avg_adamw_cast(nulls, _capi.DTYPE_BF16, 3, 0, nul, nul, nul, nul,
                                    ctypes.byref(hp), None) == _capi.OK
    assert L.fsdp_ag_unpack(None, 3, 0, nul, None) == _capi.OK
    assert L.fsdp_grad_accumulate(nul, nul, 0, ctypes.c_float(0.5), 1, None) == _capi.OK
    assert L.fsdp_flat_pack(nulls, _capi.i64_array([0, 0]), 2, 4, _capi.DTYPE_F32, nul,
                            None) == _capi.OK
    empty = _capi.i64_array([0, 7, 7, 7])
    assert L.ddp_bucket_allreduce_avg(nulls, 3, empty, 1, 2, nul, None) == _capi.OK
    assert L.ddp_bucket_allreduce_avg(nulls, 3, empty, 0, 0, nul, None) == _capi.OK
    assert L.ddp_bucket_allreduce_avg_adamw_cast(nulls, 3, empty, 1, 2, nul, nul, nul, nul, nul,
                                                 ctypes.byref(hp), None) == _capi.OK
    # an element to process: the NULL output is rejected
    assert L.ddp_bucket_allreduce_avg(nulls, 3, empty, 0, 1, nul, None) == _capi.ERR_INVALID
    assert L.fsdp_rs_avg_adamw_cast(nulls, _capi.DTYPE_BF16, 3, 5, nul, nul, nul, nul,
                                    ctypes.byref(hp), None) == _capi.ERR_INVALID
    # the scalar arguments are still checked on an empty call
    assert L.fsdp_rs_avg_adamw_cast(nulls, _capi.DTYPE_BF16, 0, 0, nul, nul, nul, nul,
                                    ctypes.byref(hp), None) == _capi.ERR_INVALID
    assert L.fsdp_rs_avg_adamw_cast(nulls, _capi.DTYPE_BF16, 3, 0, nul, nul, nul, nul,
                                    None, None) == _capi.ERR_INVALID
    assert L.fsdp_grad_unscale_check(nulls, _capi.DTYPE_F16, 3, 3, 0, nul, nul,
                                     None) == _capi.ERR_INVALID     # no scaler words


def test_comm_counter_reads_and_resets():
    """The counter of emulated inter-rank bytes: read, reset, and no count
    for calls with nothing to process (they reach no collective)."""
    L = _capi.lib()
    ss.comm_counter(reset=True)
    assert ss.comm_counter() == 0.0
    hp = ss.AdamW().at_step(1)
    nul = ctypes.c_void_p(None)
    assert L.fsdp_rs_avg_adamw_cast(_capi.ptr_array([0, 0]), _capi.DTYPE_BF16, 2, 0, nul, nul,
                                    nul, nul, ctypes.byref(hp), None) == _capi.OK
    assert L.fsdp_ag_unpack(None, 8, 0, nul, None) == _capi.OK
    assert L.ddp_bucket_allreduce_avg(_capi.ptr_array([0, 0]), 2, _capi.i64_array([0, 0]), 0, 1,
                                      nul, None) == _capi.OK
    # a rejected call counts nothing either
    assert L.fsdp_ag_unpack(None, 8, 16, nul, None) == _capi.ERR_INVALID
    assert ss.comm_counter(reset=True) == 0.0


@pytest.mark.parametrize("nd,F", [(4, 4), (8, 8), (4, 2), (8, 1)])
def test_rank_state_bytes_are_the_ledger_terms(nd, F):
    """The per-rank state the optimizer allocates is the ZeRO ledger's terms
    ("Infra: Data Parallel", ZeRO figure; "4.1 数据并行详解" section 7), with Psi
    the padded parameter count: k Psi / F of fp32 master + m + v (k = 12) and
    2 Psi / F of bf16 parameters; the reduced gradient shard (2 Psi / F) lives
    only in the fused kernel's registers; the N_d contributions to the shard
    that the emulated reduce-scatter reads add up to one full gradient, 2 Psi,
    under full sharding (F = N_d)."""
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    from synth import workloads as W
    opt = RankShardOptimizer(W.unit_9m().units + [[(1000, 3), (7,)]], nd, 0, ss.AdamW(),
                             device="cpu", shard_group=F)
    psi = F * opt.shard_total
    nbytes = lambda ts: sum(t.numel() * t.element_size() for t in ts)
    optimizer = nbytes([opt.master, opt.m, opt.v])
    params = nbytes([opt.params])
    assert optimizer == 12 * psi / F and params == 2 * psi / F
    assert ss.hybrid_state_bytes(psi, F) == optimizer + params + params   # + the gradient shard
    if F == nd:
        assert ss.state_bytes(psi, nd, 3) == optimizer + 2 * params
    # N_d contributions of the rank's S = Psi / F positions: one full
    # gradient (2 Psi) under full sharding, R = N_d / F of them under hybrid
    assert nbytes(opt.grad_in) == nd * 2 * psi / F
    if F == nd:
        assert nbytes(opt.grad_in) == 2 * psi


def test_hybrid_ledger_matches_oracle():
    for psi in (7e9, 351e6):
        for nd, F in ((8, 1), (8, 2), (8, 4), (8, 8), (16, 8), (6, 3)):
            assert ss.hybrid_state_bytes(psi, F) == pytest.approx(
                oracle.hybrid_state_bytes_per_gpu(psi, F), rel=1e-15)
            for kind in ("intra", "inter"):
                for exact in (False, True):
                    assert ss.hybrid_comm_bytes(psi, nd, F, kind, exact) == pytest.approx(
                        oracle.hybrid_comm_bytes_per_gpu(psi, nd, F, kind, exact), rel=1e-15,
                        abs=0)
    with pytest.raises(ValueError):
        ss.hybrid_comm_bytes(1e9, 8, 3, "intra")


def test_hybrid_step_rejects_a_factor_that_does_not_divide():
    L = _capi.lib()
    A = 1 << 40
    g = [A + k * (1 << 20) for k in range(8)]
    st = [A + (1 << 30) + k * (1 << 20) for k in range(4)]
    hp = _capi.AdamWHP(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    for F in (0, 3, 5, 16, -2):
        rc = L.fsdp_hybrid_rs_avg_adamw_cast(_capi.ptr_array(g), _capi.DTYPE_BF16, 8, F, 1024,
                                             *[ctypes.c_void_p(x) for x in st], ctypes.byref(hp),
                                             None)
        assert rc == _capi.ERR_INVALID, F


def test_fsdp2_layout_matches_oracle():
    dims = [(0,), (1,), (3,), (5,), (2, 3), (7, 1), (4, 2), (5, 2, 2), (11008, 4096), (4096,)]
    for n in range(1, 4):
        for shapes in itertools.product(dims, repeat=n):
            for nd in (1, 2, 3, 8):
                a = ss.fsdp2_layout(list(shapes), nd)
                b = oracle.fsdp2_layout(list(shapes), nd)
                assert (a.chunk, a.offset, a.local) == (b.chunk, b.offset, b.local)


def test_fsdp2_local_views_of_the_page_examples():
    L = _capi.lib()
    base = 0x20000
    for shapes, nd, want_rows in (([(4, 2)] * 3, 2, [2, 2, 2]), ([(8, 4)], 4, [2])):
        d0 = [s[0] for s in shapes]
        row = [int(np.prod(s[1:])) for s in shapes]
        n = len(shapes)
        for r in range(nd):
            ptrs = (_capi.c_vp * n)()
            rows = (_capi.c_i64 * n)()
            _capi.check("fsdp2_local_views", L.fsdp2_local_views(
                _capi.i64_array(d0), _capi.i64_array(row), n, nd, r, ctypes.c_void_p(base), 2,
                ptrs, rows))
            assert list(rows) == want_rows
            lay = oracle.fsdp2_layout(shapes, nd)
            assert [p - base for p in ptrs] == [2 * o for o in lay.offset]


def test_fsdp2_entry_points_reject_bad_arguments():
    L = _capi.lib()
    A = 1 << 40
    d0, row = _capi.i64_array([8, 3]), _capi.i64_array([4, 1])
    local = _capi.c_i64()
    assert L.fsdp2_layout(d0, row, 2, 0, None, None, ctypes.byref(local)) == _capi.ERR_INVALID
    assert L.fsdp2_layout(_capi.i64_array([-1]), row, 1, 2, None, None,
                          ctypes.byref(local)) == _capi.ERR_INVALID
    # gradient overlapping the output buffer
    assert L.fsdp2_chunk_cat(_capi.ptr_array([A, A + 4096]), d0, row, 2, 2, _capi.DTYPE_BF16,
                             ctypes.c_void_p(A + 16), None) == _capi.ERR_INVALID
    assert L.fsdp2_chunk_cat(_capi.ptr_array([A, A + 4096]), d0, row, 2, 2, 5,
                             ctypes.c_void_p(A + 1 << 20), None) == _capi.ERR_INVALID
    # parameter overlapping a local buffer
    assert L.fsdp2_all_gather_copy_out(_capi.ptr_array([A, A + 4096]), d0, row, 2, 2,
                                       _capi.DTYPE_BF16, _capi.ptr_array([A + 32, A + 8192]),
                                       None) == _capi.ERR_INVALID


def test_last_kernel_is_empty_until_a_launch():
    """A call that validation rejects launches nothing and names no kernel."""
    import threading
    seen = []

    def body():
        seen.append(ss.last_kernel())
        L = _capi.lib()
        rc = L.fsdp_grad_accumulate(None, None, 16, ctypes.c_float(1.0), 1, None)
        seen.append((rc, ss.last_kernel()))

    t = threading.Thread(target=body)
    t.start()
    t.join()
    assert seen[0] == ""
    assert seen[1][0] < 0 and seen[1][1] == ""


class _AdamWState(ctypes.Structure):
    """shardstep_adamw_state_t as the header declares it."""
    _fields_ = [("step", ctypes.c_int64), ("beta1_pow", ctypes.c_double),
                ("beta2_pow", ctypes.c_double), ("scalars", ctypes.c_float * 8)]


def test_adamw_state_layout_and_validation():
    assert ctypes.sizeof(_AdamWState) == _capi.ADAMW_STATE_BYTES == 56
    assert _AdamWState.scalars.offset == 24
    L = _capi.lib()
    hp = ss.AdamW().at_step(1)
    # rejected before any launch: no state, no hp, a misaligned state, a negative step
    assert L.shardstep_adamw_state_init(None, ctypes.byref(hp), 0, None) < 0
    assert "NULL" in L.shardstep_last_error().decode()
    assert L.shardstep_adamw_state_init(ctypes.c_void_p(4096), None, 0, None) < 0
    assert L.shardstep_adamw_state_init(ctypes.c_void_p(4100), ctypes.byref(hp), 0, None) < 0
    assert "misaligned" in L.shardstep_last_error().decode()
    assert L.shardstep_adamw_state_init(ctypes.c_void_p(4096), ctypes.byref(hp), -1, None) < 0
    assert L.shardstep_adamw_state_advance(None, ctypes.byref(hp), None, None) < 0
    assert L.shardstep_adamw_state_advance(ctypes.c_void_p(4100), ctypes.byref(hp), None,
                                           None) < 0
    assert L.shardstep_adamw_state_advance(ctypes.c_void_p(4096), ctypes.byref(hp),
                                           ctypes.c_void_p(4098), None) < 0
    assert "skip misaligned" in L.shardstep_last_error().decode()
    ptrs = _capi.ptr_array([4096])
    assert L.fsdp_state_rs_avg_adamw_cast(ptrs, 0, 1, 1, 16, None, None, None, None, None,
                                          None) < 0
    assert "state is NULL" in L.shardstep_last_error().decode()
    assert L.fsdp_state_rs_avg_adamw_cast(ptrs, 0, 4, 3, 16, None, None, None, None,
                                          ctypes.c_void_p(4096), None) < 0


def test_shard_pieces_place_every_element_like_the_oracle_pack():
    """fsdp_shard_pieces against the oracle's FlatParameter, by element
    tracking: the piece of tensor t in rank r's shard holds exactly tensor t's
    elements tensor_lo.., the pieces of a shard do not overlap, and what no
    piece covers is the zero padding."""
    rnd = random.Random(3)
    for _ in range(300):
        nd = rnd.randint(1, 7)
        numels = [rnd.randint(0, 12) for _ in range(rnd.randint(0, 5))]
        tensors = [(t + 1) * 1000.0 + np.arange(n, dtype=np.float64) for t, n in enumerate(numels)]
        flat, lay = oracle.flat_pack(tensors, nd) if numels else (np.zeros(0), oracle.layout([], nd))
        for r in range(nd):
            shard = flat[r * lay.shard:(r + 1) * lay.shard]
            covered = np.zeros(lay.shard, bool)
            pieces = ss.fsdp_shard_pieces(numels, nd, r)
            assert len(pieces) == len(numels)
            for t, (slo, tlo, cnt) in enumerate(pieces):
                if cnt == 0:
                    assert (slo, tlo) == (0, 0)
                    continue
                assert np.array_equal(shard[slo:slo + cnt], tensors[t][tlo:tlo + cnt])
                assert not covered[slo:slo + cnt].any()
                covered[slo:slo + cnt] = True
            assert not shard[~covered].any()
            assert covered.sum() == max(0, min(lay.total, (r + 1) * lay.shard) - r * lay.shard)


def test_shard_pieces_of_the_worked_example_and_bad_arguments():
    # [P1] FSDP1 figure: three (4,2) weights on two ranks; rank 0 holds W1 and
    # W2's first 4 elements, rank 1 the rest of W2 and all of W3
    assert ss.fsdp_shard_pieces([8, 8, 8], 2, 0) == [(0, 0, 8), (8, 0, 4), (0, 0, 0)]
    assert ss.fsdp_shard_pieces([8, 8, 8], 2, 1) == [(0, 0, 0), (0, 4, 4), (4, 0, 8)]
    for nd, rank in ((2, 2), (2, -1), (0, 0)):
        with pytest.raises(ss.ShardstepError):
            ss.fsdp_shard_pieces([8, 8, 8], nd, rank)


def test_new_entry_points_reject_bad_arguments_before_launch():
    """The fused DDP step, the watchdog limit and the division self-check
    validate everything on the host; nothing here reaches the GPU."""
    L = _capi.lib()
    A = 1 << 40
    n = 4096
    boff = _capi.i64_array([0, n])
    grads = _capi.ptr_array([A, A + 2 * n])
    master, m, v = (ctypes.c_void_p(A + (1 << 20) * k) for k in (1, 2, 3))
    params = ctypes.c_void_p(A + (1 << 20) * 4)
    hp = ss.AdamW().at_step(1)
    call = L.ddp_bucket_allreduce_avg_adamw_cast
    # params is gradient 1
    assert call(grads, 2, boff, 0, 1, None, master, m, v, ctypes.c_void_p(A + 2 * n),
                ctypes.byref(hp), None) == _capi.ERR_INVALID
    # m is v
    assert call(grads, 2, boff, 0, 1, None, master, v, v, params, ctypes.byref(hp),
                None) == _capi.ERR_INVALID
    # the mean is the parameters
    assert call(grads, 2, boff, 0, 1, params, master, m, v, params, ctypes.byref(hp),
                None) == _capi.ERR_INVALID
    # decreasing bucket offsets, a null gradient, too many ranks, step 0
    assert call(grads, 2, _capi.i64_array([0, n, 5]), 0, 2, None, master, m, v, params,
                ctypes.byref(hp), None) == _capi.ERR_INVALID
    assert call(_capi.ptr_array([A, 0]), 2, boff, 0, 1, None, master, m, v, params,
                ctypes.byref(hp), None) == _capi.ERR_INVALID
    assert call(grads, _capi.MAX_ND + 1, boff, 0, 1, None, master, m, v, params,
                ctypes.byref(hp), None) == _capi.ERR_CAPACITY
    hp0 = ss.AdamW().at_step(0)
    assert call(grads, 2, boff, 0, 1, None, master, m, v, params, ctypes.byref(hp0),
                None) == _capi.ERR_INVALID
    # an empty range is accepted and launches nothing
    assert call(grads, 2, _capi.i64_array([0, 0]), 0, 1, None, master, m, v, params,
                ctypes.byref(hp), None) == _capi.OK
    assert L.shardstep_set_tma_wait_ns(-5) == _capi.ERR_INVALID
    check = L.shardstep_check_mean_division
    for nd in (0, _capi.MAX_ND + 1):
        assert check(nd, ctypes.c_void_p(A), ctypes.c_void_p(A + 8), None) == _capi.ERR_INVALID
    assert check(3, None, ctypes.c_void_p(A + 8), None) == _capi.ERR_INVALID
    assert check(3, ctypes.c_void_p(A + 4), ctypes.c_void_p(A + 8), None) == _capi.ERR_INVALID
    assert b"misaligned" in L.shardstep_last_error()


def test_every_profiled_kernel_matches_its_counters():
    """bench.py reports roofline.traffic only while the source of the kernel
    a profile's DRAM counters were taken on is unchanged (a hash of its code
    without comments); every line with a profile must still have its
    counters, so a kernel change without a new capture is caught here."""
    import bench
    stale = [w for w in bench.PROFILES if bench.profiled_traffic(w) is None]
    assert not stale, f"profiles whose kernel source changed since the capture: {stale}"
