"""The degenerate cases of the method, on the GPU against the oracle.

"Infra: Data Parallel", FSDP1 section: a FlatParameter is the unit's tensors
concatenated and split into N_d equal shards, so a shard may cut a tensor,
hold only padding, or hold nothing of a tensor (the empty view of
use_orig_params).  These tests drive every entry point with the sizes where
that happens: an empty shard (S = 0), zero-size tensors between others, a
unit smaller than N_d (ranks holding only padding), a unit of zero-size
tensors only, N_d = 1, single-element shards, empty buckets among the DDP
buckets.  An empty call launches nothing and writes nothing; every other
result equals the oracle's bit for bit."""
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
HP = AdamWConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HPC = ss.AdamW(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    yield
    assert ss.device_status() == 0


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _bf16_dev(h):
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).to(DEV).view(torch.bfloat16)


def _f32_dev(h):
    return torch.from_numpy(np.ascontiguousarray(h, dtype=np.float32)).to(DEV)


# ------------------------------------------------------- empty calls

def test_empty_calls_launch_nothing():
    """S = 0 (or n = 0, or no buckets) is a valid call at every entry point:
    it returns without a launch, and the scaler's words stay as they were."""
    e16 = torch.empty(0, dtype=torch.bfloat16, device=DEV)
    f16 = torch.empty(0, dtype=torch.float16, device=DEV)
    e32 = torch.empty(0, dtype=torch.float32, device=DEV)
    st = ss.AdamWState(HPC, 1, device=DEV)
    sc = ss.GradScaler(init_scale=1024.0, device=DEV)
    torch.cuda.synchronize()
    before = ss.launch_count()
    for nd in (1, 3, 8):
        g = [e16] * nd
        ss.fsdp_rs_avg_adamw_cast(g, e32, e32, e32, e16, HPC, 1)
        ss.fsdp_rs_avg_adamw_cast([e32] * nd, e32, e32, e32, e16, HPC, 1)
        ss.fsdp_hybrid_rs_avg_adamw_cast(g, 1, e32, e32, e32, e16, HPC, 1)
        ss.fsdp_state_rs_avg_adamw_cast(g, e32, e32, e32, e16, st)
        ss.fsdp_accumulate_rs_avg_adamw_cast([e32] * nd, g, 0.25, e32, e32, e32, e16, HPC, 1)
        ss.fsdp_state_accumulate_rs_avg_adamw_cast([e32] * nd, g, 0.25, e32, e32, e32, e16, st)
        sc.check([f16] * nd)
        sc.step([f16] * nd, e32, e32, e32, e16, HPC, 1)
        sc.step_state([f16] * nd, e32, e32, e32, e16, st)
        ss.fsdp_ag_unpack([e16] * nd, e16)
        ss.ddp_bucket_allreduce_avg(g, [0], e16)
        ss.ddp_bucket_allreduce_avg(g, [0, 0, 0], e16)
        ss.ddp_bucket_allreduce_avg_adamw_cast(g, [0, 0], e32, e32, e32, e16, HPC, 1)
        ss.fsdp_flat_pack([e32, e32], nd, flat=e32)
    ss.fsdp_grad_accumulate(e16, e32, 0.5, True)
    torch.cuda.synchronize()
    assert ss.launch_count() == before
    assert int(sc.found_inf.item()) == 0 and float(sc.scale.item()) == 1024.0
    assert st.step() == 1


# ------------------------------------------- degenerate FlatParameters

UNITS = [
    ("zero_size_between", [(0,), (1,), (0,), (3,), (2, 2), (0,)], 8),   # T = 8, S = 1
    ("smaller_than_nd", [(3,)], 8),                                     # ranks 3..7: padding only
    ("one_element", [(1,)], 4),
    ("ragged_three_ranks", [(5,), (0,), (7,)], 3),                     # T = 12, S = 4
    ("nd_one", [(2, 3), (0,), (5,)], 1),
    ("a_rank_holds_nothing_of_a_tensor", [(6,), (1,), (9,)], 4),        # T = 16, S = 4
]


@pytest.mark.parametrize("name,shapes,nd", UNITS, ids=[u[0] for u in UNITS])
def test_degenerate_unit_through_the_whole_step(name, shapes, nd):
    """Pack the master and every rank's gradients, each rank's fused step
    (even ranks write their bf16 output into their slot of the full buffer,
    odd ranks into a buffer of their own that the all-gather copies), the
    all-gather and the views, two steps; the sharded and full views against
    the oracle's."""
    numels = [int(np.prod(s)) for s in shapes]
    seed = sum(numels) * 31 + nd
    mh = [synth.host_fill(synth.normal_stream(seed, (1, t), 0.02), 0, n, "f32").reshape(s)
          for t, (n, s) in enumerate(zip(numels, shapes))]
    gh = [[synth.host_fill(synth.normal_stream(seed, (2, q, t), 1e-3), 0, n, "bf16").reshape(s)
           for t, (n, s) in enumerate(zip(numels, shapes))] for q in range(nd)]
    want_master, lay = oracle.flat_pack(mh, nd)
    want_g = [oracle.flat_pack(g, nd)[0] for g in gh]
    S, P = lay.shard, lay.padded

    glay = ss.fsdp_layout(numels, nd)
    assert (glay.total, glay.padded, glay.shard) == (lay.total, lay.padded, lay.shard)
    master = ss.fsdp_flat_pack([_f32_dev(x) for x in mh], nd)
    grads = [ss.fsdp_flat_pack([_bf16_dev(x) for x in g], nd) for g in gh]
    torch.cuda.synchronize()
    assert_bits(master.cpu().numpy(), want_master, "packed master")
    for q in range(nd):
        assert_bits(_u16(grads[q]), want_g[q], f"packed gradient {q}")

    m = torch.zeros(P, device=DEV)
    v = torch.zeros(P, device=DEV)
    full = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    p_h = want_master.copy()
    m_h = np.zeros(P, np.float32)
    v_h = np.zeros(P, np.float32)
    own = [full[r * S:(r + 1) * S] if r % 2 == 0
           else torch.empty(S, dtype=torch.bfloat16, device=DEV) for r in range(nd)]
    for t in (1, 2):
        outs = []
        for r in range(nd):
            sl = slice(r * S, (r + 1) * S)
            ss.fsdp_rs_avg_adamw_cast([g[sl] for g in grads], master[sl], m[sl], v[sl], own[r],
                                      HPC, t)
            p1, m1, v1, o1 = oracle.fsdp_shard_step(want_g, r, S, p_h[sl], m_h[sl], v_h[sl], HP, t)
            p_h[sl], m_h[sl], v_h[sl] = p1, m1, v1
            outs.append(o1)
        ss.fsdp_ag_unpack(own, full)
        want_full, want_views = oracle.ag_unpack(outs, lay, shapes)
        torch.cuda.synchronize()
        assert_bits(master.cpu().numpy(), p_h, f"step {t} master")
        assert_bits(m.cpu().numpy(), m_h, f"step {t} m")
        assert_bits(v.cpu().numpy(), v_h, f"step {t} v")
        assert_bits(_u16(full), want_full, f"step {t} gathered")
        assert not want_full[lay.total:].any()          # the padding stays zero
        for k, (gv, wv) in enumerate(zip(ss.fsdp_views(full, shapes, nd), want_views)):
            assert tuple(gv.shape) == tuple(shapes[k])
            assert_bits(_u16(gv).reshape(-1), np.asarray(wv).reshape(-1), f"view {k}")
        for r in range(nd):
            sh = master[r * S:(r + 1) * S]
            for k, (gv, wv) in enumerate(zip(ss.fsdp_views(sh, shapes, nd, r),
                                             oracle.sharded_views(p_h[r * S:(r + 1) * S], lay, r))):
                assert gv.numel() == wv.size, (r, k)
                assert_bits(gv.cpu().numpy(), wv, f"rank {r} view {k}")


def test_unit_of_zero_size_tensors_only():
    """T = 0: no padding either (P = 0); the views are empty and every call
    on the unit is empty."""
    shapes = [(0,), (0, 4), (3, 0)]
    numels = [0, 0, 0]
    for nd in (1, 2, 8):
        lay = ss.fsdp_layout(numels, nd)
        olay = oracle.layout(numels, nd)
        assert (lay.total, lay.padded, lay.shard) == (olay.total, olay.padded, olay.shard) == (0, 0, 0)
        flat = ss.fsdp_flat_pack([torch.empty(s, dtype=torch.bfloat16, device=DEV)
                                  for s in shapes], nd)
        assert flat.numel() == 0
        views = ss.fsdp_views(flat, shapes, nd)
        assert [tuple(x.shape) for x in views] == shapes
        for r in range(nd):
            assert all(x.numel() == 0 for x in ss.fsdp_views(flat, shapes, nd, r))


# ----------------------------------------------------------- DDP

def test_empty_buckets_among_buckets():
    """Bucket offsets with empty buckets (equal neighbours) at the start, in
    the middle and at the end: the empty ones are skipped, the others equal
    the oracle, for the all-reduce alone and fused with AdamW."""
    nd = 3
    boff = [0, 0, 7, 7, 7, 4103, 4104, 4104]
    total = boff[-1]
    gh = [synth.host_fill(synth.normal_stream(44, (q,), 1e-3), 0, total, "bf16") for q in range(nd)]
    grads = [_bf16_dev(h) for h in gh]
    out = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    before = ss.launch_count()
    ss.ddp_bucket_allreduce_avg(grads, boff, out)
    torch.cuda.synchronize()
    assert ss.launch_count() - before == 3            # the non-empty buckets only
    want = oracle.bucket_allreduce_avg(gh, boff)
    assert_bits(_u16(out), want, "bucket mean")
    p0 = synth.host_fill(synth.normal_stream(44, (9,), 0.02), 0, total, "f32")
    pd, md, vd = _f32_dev(p0), torch.zeros(total, device=DEV), torch.zeros(total, device=DEV)
    params = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    mean = torch.empty(total, dtype=torch.bfloat16, device=DEV)
    ss.ddp_bucket_allreduce_avg_adamw_cast(grads, boff, pd, md, vd, params, HPC, 1, mean_out=mean)
    z = np.zeros(total, np.float32)
    avg, p1, m1, v1, o1 = oracle.ddp_step(gh, boff, p0, z, z, HP, 1)
    torch.cuda.synchronize()
    for name, got, w in (("mean", _u16(mean), avg), ("master", pd.cpu().numpy(), p1),
                         ("m", md.cpu().numpy(), m1), ("v", vd.cpu().numpy(), v1),
                         ("params", _u16(params), o1)):
        assert_bits(got, w, name)

