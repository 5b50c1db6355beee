"""Pins for the oracle's checkpoint resharding: what "Infra: Data Parallel"
(section on checkpoints) fixes -- a load at the same rank count restores the
saved shards, and a load at another rank count gives each new rank its slice
of the same state -- checked by element tracking and by composition."""
import itertools

import numpy as np

import oracle
from oracle import checkpoint as ock


def _saved(total, nd, seed=0):
    flat, lay = oracle.flat_pack([np.arange(1, total + 1, dtype=np.float32)], nd)
    return [oracle.shard_of(flat, lay, r) for r in range(nd)], flat


def test_same_rank_count_restores_every_shard():
    for total, nd in ((24, 2), (25, 4), (7, 8), (1000, 3)):
        shards, _ = _saved(total, nd)
        for r in range(nd):
            assert np.array_equal(ock.reshard(shards, total, nd, r), shards[r])


def test_other_rank_counts_slice_the_same_state():
    for total in (1, 7, 24, 25, 97):
        for old_nd, new_nd in itertools.product((1, 2, 3, 4, 8), repeat=2):
            shards, _ = _saved(total, old_nd)
            new = [ock.reshard(shards, total, new_nd, r) for r in range(new_nd)]
            # element tracking: element k of the unit (value k + 1) is at its
            # FlatParameter position under the new layout, padding is zero
            lay = oracle.layout([total], new_nd)
            cat = np.concatenate(new)
            assert cat.size == lay.padded
            assert np.array_equal(cat[:total], np.arange(1, total + 1, dtype=np.float32))
            assert not cat[total:].any()


def test_resharding_composes():
    total = 1001
    shards, _ = _saved(total, 8)
    via4 = [ock.reshard(shards, total, 4, r) for r in range(4)]
    back = [ock.reshard(via4, total, 8, r) for r in range(8)]
    for a, b in zip(back, shards):
        assert np.array_equal(a, b)


def test_plan_pieces_rebuild_the_new_shard():
    for total in (1, 5, 24, 97, 256):
        for old_nd, new_nd in itertools.product((1, 2, 3, 5, 8), repeat=2):
            shards, _ = _saved(total, old_nd)
            S_new = -(-total // new_nd)
            for r in range(new_nd):
                out = np.zeros(S_new, np.float32)
                for q, off, k, n in ock.plan(total, old_nd, new_nd, r):
                    out[k:k + n] = shards[q][off:off + n]
                assert np.array_equal(out, ock.reshard(shards, total, new_nd, r))
