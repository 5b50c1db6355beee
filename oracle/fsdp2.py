"""FSDP2 per-parameter sharding along dim 0.  TEST INFRASTRUCTURE.

"Infra: Data Parallel", section "FSDP2：分别记录每个参数的分片" and its figure
("FSDP2：每个参数分别沿 dim 0 切给两个 rank"): every parameter of a
fully_shard group is a DTensor split along dim 0 -- a (4,2) weight on two
ranks is (2,2) locally, rank 0 holding the first two rows; an (8,4) weight on
four ranks is (2,4) locally while its global shape stays (8,4).  The group's
parameters are still communicated together: one all-gather and one
reduce-scatter per group.

Readings where the pages are silent:
  * uneven dim 0: c = ceil(d0 / N_d) rows per rank; rank r holds rows
    [r*c, min((r+1)*c, d0)), possibly none (torch.chunk semantics);
  * the group's communication buffers are rank-major: rank r's piece is the
    concatenation, in registration order, of its rows of every parameter,
    each padded with zero rows to c rows, so every rank's piece has the same
    length L = sum_t c_t * row_t (row_t = product of the trailing dims);
  * the optimizer state of a rank is that padded local buffer (padding rows
    stay zero: their gradient and master are zero).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class Fsdp2Layout:
    shapes: list
    nd: int
    dim0: list        # d0_t
    row: list         # elements per dim-0 row of t
    chunk: list       # c_t = ceil(d0_t / nd) rows per rank
    offset: list      # element offset of t inside a rank's local buffer
    local: int        # L, elements of a rank's local buffer

    def rows_of(self, r: int, t: int) -> int:
        """Rows of parameter t held by rank r."""
        c, d0 = self.chunk[t], self.dim0[t]
        return max(0, min(c, d0 - r * c))


def fsdp2_layout(shapes, nd: int) -> Fsdp2Layout:
    if nd < 1:
        raise ValueError("nd must be >= 1")
    dim0, row, chunk, offset = [], [], [], []
    pos = 0
    for s in shapes:
        s = tuple(int(d) for d in s)
        if len(s) == 0:
            raise ValueError("scalar parameters have no dim 0")
        d0 = s[0]
        rw = 1
        for d in s[1:]:
            rw *= d
        c = -(-d0 // nd)
        dim0.append(d0)
        row.append(rw)
        chunk.append(c)
        offset.append(pos)
        pos += c * rw
    return Fsdp2Layout([tuple(s) for s in shapes], nd, dim0, row, chunk, offset, pos)


def local_shards(tensors, lay: Fsdp2Layout, r: int):
    """DTensor.to_local() of rank r: its rows of every parameter, local shape
    (rows, trailing dims...)."""
    out = []
    for t, x in enumerate(tensors):
        x = np.asarray(x).reshape(lay.shapes[t])
        c = lay.chunk[t]
        out.append(x[r * c:r * c + lay.rows_of(r, t)])
    return out


def chunk_cat(tensors, lay: Fsdp2Layout):
    """One rank's reduce-scatter input: its full per-parameter gradients laid
    out rank-major, nd pieces of L elements, piece r = rank r's rows of every
    parameter, each zero-padded to c_t rows."""
    dtype = np.asarray(tensors[0]).dtype if tensors else np.float32
    out = np.zeros(lay.nd * lay.local, dtype=dtype)
    for r in range(lay.nd):
        for t, x in enumerate(tensors):
            flat = np.asarray(x).reshape(-1)
            n = lay.rows_of(r, t) * lay.row[t]
            src = r * lay.chunk[t] * lay.row[t]
            dst = r * lay.local + lay.offset[t]
            out[dst:dst + n] = flat[src:src + n]
    return out


def local_buffer(tensors, lay: Fsdp2Layout, r: int):
    """Rank r's padded local buffer of the group (its piece of chunk_cat)."""
    return chunk_cat(tensors, lay)[r * lay.local:(r + 1) * lay.local]


def all_gather_copy_out(local_buffers, lay: Fsdp2Layout):
    """All-gather of the ranks' local buffers followed by the copy into full
    per-parameter tensors of the global shapes (padding rows dropped)."""
    if len(local_buffers) != lay.nd:
        raise ValueError("need one local buffer per rank")
    dtype = np.asarray(local_buffers[0]).dtype
    outs = []
    for t, shape in enumerate(lay.shapes):
        full = np.zeros(lay.dim0[t] * lay.row[t], dtype=dtype)
        for r in range(lay.nd):
            n = lay.rows_of(r, t) * lay.row[t]
            dst = r * lay.chunk[t] * lay.row[t]
            full[dst:dst + n] = np.asarray(local_buffers[r])[lay.offset[t]:lay.offset[t] + n]
        outs.append(full.reshape(shape))
    return outs
