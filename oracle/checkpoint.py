"""Sharded checkpoint resharding.  TEST INFRASTRUCTURE.

"Infra: Data Parallel", section "Checkpoint：让各张卡保存自己的分片": with the
model state spread over the GPUs, each rank saves the shards it owns plus the
metadata needed to restore them; loading reads according to the target
model's sharding layout, so the GPU count may differ between saving and
loading; optimizer state is saved with the weights.

Plain definition of a load at a different N_d: every unit's flat state is
the concatenation of the saved ranks' shards cut to the unit's T elements;
the new rank's shard is that flat state zero-padded to the new multiple of
N_d and sliced as in the FlatParameter layout.
"""
from __future__ import annotations

import numpy as np


def unit_flat(old_shards, total: int):
    """One unit's flat state from the saved ranks' shards (rank order)."""
    return np.concatenate([np.asarray(s).reshape(-1) for s in old_shards])[:total]


def reshard(old_shards, total: int, new_nd: int, new_rank: int):
    """Rank ``new_rank``'s shard of one unit under ``new_nd`` ranks."""
    flat = unit_flat(old_shards, total)
    padded = -(-total // new_nd) * new_nd
    S = padded // new_nd
    full = np.zeros(padded, dtype=flat.dtype)
    full[:total] = flat
    return full[new_rank * S:(new_rank + 1) * S]


def plan(total: int, old_nd: int, new_nd: int, new_rank: int):
    """Pieces (old_rank, old_offset, new_offset, count) that fill rank
    ``new_rank``'s new shard of a unit from the saved shards, in new-offset
    order; positions past the unit's total are padding (zero) and in no
    piece.  Brute force: walk the new shard element by element."""
    S_old = -(-total // old_nd)
    S_new = -(-total // new_nd)
    pieces = []
    for k in range(S_new):
        g = new_rank * S_new + k
        if g >= total:
            break
        q, off = divmod(g, S_old)
        if pieces and pieces[-1][0] == q and pieces[-1][1] + pieces[-1][3] == off:
            pieces[-1][3] += 1
        else:
            pieces.append([q, off, k, 1])
    return [tuple(p) for p in pieces]
