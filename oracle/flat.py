"""FlatParameter layout, pack, shards, views and all-gather.  TEST INFRASTRUCTURE.

Follows "Infra: Data Parallel", section "Fully Sharded Data Parallel (FSDP)",
sub-section "FSDP1：先打包，再切分" and its figure "FSDP1：先拼成
FlatParameter，再切给两个 rank": the tensors of one FSDP unit are flattened,
concatenated in registration order into one 1-D FlatParameter and split
evenly across the N_d ranks, so a shard may cut a tensor; with
use_orig_params the original tensors become views into the flat buffer and,
in the sharded state, a view holds only the rank's piece of the tensor, or
nothing at all.  "PyTorch FSDP..." section 3.1 gives the same per-unit
flatten + shard + all-gather cycle.

The figure leaves padding out; the padded length is the smallest multiple of
N_d not below the total, with zeros at the tail (the only reading that keeps
the shards equal).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Layout:
    numels: list            # n_t, registration order
    nd: int                 # N_d
    total: int              # T = sum n_t
    padded: int             # P = ceil(T / N_d) * N_d
    shard: int              # S = P / N_d
    offsets: list           # off_t = sum of n_u for u < t
    lo: list = field(default_factory=list)   # lo[r][t], shard coordinates
    hi: list = field(default_factory=list)   # hi[r][t]; empty piece when lo == hi


def layout(numels, nd: int) -> Layout:
    """Offsets of each tensor in the FlatParameter and, per rank r and tensor t,
    the piece [lo, hi) of shard r (shard coordinates) that holds tensor t.

    Shard r covers flat[r*S, (r+1)*S).  The piece is the intersection of that
    range with [off_t, off_t + n_t), written in shard coordinates and clamped
    to [0, S]; when the two do not meet it is empty (lo == hi), the "empty
    tensor" view of the use_orig_params paragraph.
    """
    if nd < 1:
        raise ValueError("nd must be >= 1")
    numels = [int(n) for n in numels]
    if any(n < 0 for n in numels):
        raise ValueError("negative numel")
    total = sum(numels)
    padded = -(-total // nd) * nd
    shard = padded // nd
    offsets, acc = [], 0
    for n in numels:
        offsets.append(acc)
        acc += n
    lo, hi = [], []
    for r in range(nd):
        base = r * shard
        lo.append([min(max(off - base, 0), shard) for off in offsets])
        hi.append([min(max(off + n - base, 0), shard) for off, n in zip(offsets, numels)])
    return Layout(numels, nd, total, padded, shard, offsets, lo, hi)


def flat_pack(tensors, nd: int):
    """Concatenate the row-major flattened tensors (all of one dtype: uint16 for
    bf16 bits, or float32) and zero-pad to P.  Returns (flat, layout)."""
    arrs = [np.ascontiguousarray(t).reshape(-1) for t in tensors]
    dtypes = {a.dtype for a in arrs}
    if len(dtypes) > 1:
        raise ValueError("one dtype per unit")
    dtype = dtypes.pop() if dtypes else np.uint16
    lay = layout([a.size for a in arrs], nd)
    flat = np.zeros(lay.padded, dtype=dtype)
    for a, off in zip(arrs, lay.offsets):
        flat[off:off + a.size] = a
    return flat, lay


def shard_of(flat, lay: Layout, r: int):
    """Rank r's flat shard: flat[r*S, (r+1)*S)."""
    return flat[r * lay.shard:(r + 1) * lay.shard]


def sharded_views(shard, lay: Layout, r: int):
    """use_orig_params views of rank r's shard: 1-D piece of each tensor held
    by the rank (possibly empty)."""
    return [shard[lo:hi] for lo, hi in zip(lay.lo[r], lay.hi[r])]


def ag_unpack(shards, lay: Layout, shapes=None):
    """All-gather: full[q*S + i] = shards[q][i] for every rank q, then one view
    per tensor, full[off_t, off_t + n_t) reshaped to the tensor's shape; the
    padding is in no view."""
    if len(shards) != lay.nd or any(s.size != lay.shard for s in shards):
        raise ValueError("need N_d shards of S elements")
    full = np.concatenate([np.asarray(s).reshape(-1) for s in shards]) if shards else np.zeros(0)
    return full, unpack_views(full, lay, shapes)


def unpack_views(full, lay: Layout, shapes=None):
    views = []
    for t, (off, n) in enumerate(zip(lay.offsets, lay.numels)):
        v = full[off:off + n]
        if shapes is not None:
            v = v.reshape(shapes[t])
        views.append(v)
    return views


def element_source(lay: Layout, flat_idx):
    """Where FlatParameter element f comes from: tensor t = the one whose range
    [off_t, off_t + n_t) holds f, at row-major index k = f - off_t; t = -1
    (and k = 0) for the zero padding [T, P).  The inverse of flat_pack,
    element by element."""
    flat_idx = np.asarray(flat_idx, dtype=np.int64)
    t = np.full(flat_idx.size, -1, dtype=np.int64)
    k = np.zeros(flat_idx.size, dtype=np.int64)
    for ti, (off, n) in enumerate(zip(lay.offsets, lay.numels)):
        sel = (flat_idx >= off) & (flat_idx < off + n)
        t[sel] = ti
        k[sel] = flat_idx[sel] - off
    return t, k


def rank_view_sources(layouts, r: int, idx):
    """A rank that keeps its shard of every unit back to back (unit order):
    for position i of that concatenation, the unit u, and the tensor t and
    row-major index k it comes from (t = -1 in a unit's padding).  Unit u's
    part is shard_of(flat_u, r), i.e. flat_u[r*S_u + j] for j < S_u."""
    idx = np.asarray(idx, dtype=np.int64)
    u_out = np.full(idx.size, -1, dtype=np.int64)
    t_out = np.full(idx.size, -1, dtype=np.int64)
    k_out = np.zeros(idx.size, dtype=np.int64)
    start = 0
    for u, lay in enumerate(layouts):
        sel = np.nonzero((idx >= start) & (idx < start + lay.shard))[0]
        if sel.size:
            t, k = element_source(lay, r * lay.shard + (idx[sel] - start))
            u_out[sel] = u
            t_out[sel] = t
            k_out[sel] = k
        start += lay.shard
    if (u_out < 0).any():
        raise IndexError("position past the rank's shards")
    return u_out, t_out, k_out

