"""GPU round trips of the sharded checkpoint: live RankShardOptimizer state
(after real fused steps) saved by every rank of one layout and loaded under
other rank counts and sharding factors equals the oracle's resharding of the
saved state, bit for bit, and training continues from it."""
import numpy as np
import pytest
import torch

import sharded_optimizer_step_gb300 as ss
import synth
from oracle import checkpoint as ock
from sharded_optimizer_step_gb300 import checkpoint as ck
from sharded_optimizer_step_gb300.engine import RankShardOptimizer
from synth import workloads as W
from tests._views import gpu_fill_rank

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ss.build()
    synth.build_dev()


def _opts(w, nd, F=0):
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    return [RankShardOptimizer(w.units, nd, r, hp, device=DEV, shard_group=F)
            for r in range(F or nd)]


def _train(w, opts, steps):
    for o in opts:
        gpu_fill_rank(o, o.master, w.master_stream)
    for t in range(1, steps + 1):
        for o in opts:
            for q in range(o.nd):
                gpu_fill_rank(o, o.grad_in[q], lambda u, k, q=q: w.grad_stream(t, q, 0, u, k))
            o.step()
    torch.cuda.synchronize()


def _host_state(opts):
    """Per unit, per kind: the saved ranks' shards as numpy arrays."""
    out = []
    for u in range(len(opts[0].layouts)):
        kinds = []
        for name in ("master", "m", "v"):
            kinds.append([getattr(o, name)[o.starts[u]:o.starts[u] + o.layouts[u].shard]
                          .cpu().numpy() for o in opts])
        out.append(kinds)
    return out


@pytest.mark.parametrize("new_nd,new_F", [(4, 0), (16, 0), (8, 0), (16, 4), (3, 0)])
def test_save_under_8_ranks_load_under_another_layout(tmp_path, new_nd, new_F):
    w = W.gpt2_small()
    old = _opts(w, 8)
    _train(w, old, 2)
    saved = _host_state(old)
    ck.save(str(tmp_path), old)
    ck.verify(str(tmp_path))
    new = _opts(w, new_nd, new_F)
    ck.load(str(tmp_path), new)
    for o in new:
        assert o.t == 2
        for u, lay in enumerate(o.layouts):
            for k, name in enumerate(("master", "m", "v")):
                want = ock.reshard(saved[u][k], lay.total, o.F, o.rank)
                got = getattr(o, name)[o.starts[u]:o.starts[u] + lay.shard].cpu().numpy()
                assert got.tobytes() == want.tobytes(), (o.rank, u, name)
    # training continues from the restored state
    for o in new:
        for q in range(o.nd):
            o.grad_in[q].normal_(0, 1e-3)
        o.step()
    torch.cuda.synchronize()
    assert all(o.t == 3 and torch.isfinite(o.master).all() for o in new)


def test_hybrid_group_checkpoint_round_trip(tmp_path):
    w = W.gpt2_small()
    old = _opts(w, 16, 8)          # one group of 8 shards (the other group is a replica)
    _train(w, old, 1)
    saved = _host_state(old)
    ck.save(str(tmp_path), old)
    new = _opts(w, 16, 8)
    ck.load(str(tmp_path), new)
    for o, s in zip(new, range(8)):
        for u in range(len(o.layouts)):
            got = o.master[o.starts[u]:o.starts[u] + o.layouts[u].shard].cpu().numpy()
            assert got.tobytes() == saved[u][0][s].tobytes()


def test_reload_through_used_staging_restores_padding(tmp_path):
    """Save and load reuse each optimizer's pinned staging: a load after a
    save of other values must still give zeros at the padding positions of
    the new layout (N_d = 5 pads every GPT-2 unit)."""
    w = W.gpt2_small()
    old = _opts(w, 8)
    _train(w, old, 1)
    saved = _host_state(old)
    a, b = tmp_path / "a", tmp_path / "b"
    ck.save(str(a), old)
    new = _opts(w, 5)
    assert any(lay.padded > lay.total for lay in new[0].layouts)
    for o in new:
        for buf in (o.master, o.m, o.v):
            buf.uniform_(1.0, 2.0)       # padding positions included
    ck.save(str(b), new)                 # staging now holds these values
    ck.load(str(a), new)
    for o in new:
        for u, lay in enumerate(o.layouts):
            for k, name in enumerate(("master", "m", "v")):
                want = ock.reshard(saved[u][k], lay.total, o.F, o.rank)
                got = getattr(o, name)[o.starts[u]:o.starts[u] + lay.shard].cpu().numpy()
                assert got.tobytes() == want.tobytes(), (o.rank, u, name)
    for o in new:
        ck.release_staging(o)


def test_device_step_state_is_saved_and_restored(tmp_path):
    """Steps taken on the device step state (the host count does not move)
    are saved with the device count; a load into optimizers that also keep
    their count on the device restores it there, and the next replayed-style
    step continues with the bits of uninterrupted training."""
    w = W.gpt2_small_nd7()
    w.units = w.units[:2]
    nd = 4
    a = _opts(w, nd)
    for o in a:
        gpu_fill_rank(o, o.master, w.master_stream)
        for q in range(nd):
            gpu_fill_rank(o, o.grad_in[q], lambda u, k, q=q: w.grad_stream(1, q, 0, u, k))
        o.device_step_state()
    for _ in range(3):
        for o in a:
            o.step_on_device()
    torch.cuda.synchronize()
    assert all(o.t == 0 and o.state.step() == 3 for o in a)
    ck.save(str(tmp_path / "ck"), a)
    assert ck.info(str(tmp_path / "ck"))[1] == 3
    b = _opts(w, nd)
    for o in b:
        o.device_step_state()              # at step 0, until the load
        for q in range(nd):
            o.grad_in[q].copy_(a[o.rank].grad_in[q])
    ck.load(str(tmp_path / "ck"), b)
    assert all(o.t == 3 and o.state.step() == 3 for o in b)
    for o, p in zip(a, b):
        o.step_on_device()
        p.step_on_device()
    torch.cuda.synchronize()
    for o, p in zip(a, b):
        for name in ("master", "m", "v", "params"):
            x, y = getattr(o, name), getattr(p, name)
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), name
        assert o.state.step() == p.state.step() == 4
