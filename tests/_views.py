"""Inputs of a rank's buffers, built by the two independent layouts.

A rank keeps its shard of every unit back to back.  On the GPU side the
positions of each tensor's piece in those buffers come from the library
(``RankShardOptimizer.rank_pieces``, i.e. ``fsdp_shard_pieces``); on the
oracle side each sampled position is traced back to its tensor element with
the oracle's own layout (``oracle.rank_view_sources``).  ``synth`` only turns
(tensor, element index) into a value."""
import oracle
import synth


def gpu_fill_rank(opt, buf, stream_of):
    """buf (a rank buffer of ``opt``) receives, at every piece the library
    places there, the piece's elements of ``stream_of(unit, tensor)``; the
    units' padding is left as it is (zero in a fresh buffer)."""
    synth.dev_fill_pieces(buf, opt.rank_pieces(), stream_of)


def oracle_layouts(w):
    return [oracle.layout(w.unit_numels(u), w.F) for u in range(len(w.units))]


def oracle_rank_values(w, r, idx, stream_of, dtype):
    """The values at positions idx of rank r's buffer, from the oracle's
    layout (zero in padding)."""
    u, t, k = oracle.rank_view_sources(oracle_layouts(w), r, idx)
    return synth.host_gather_sources(u, t, k, stream_of, dtype)


def oracle_rank_total(w):
    return sum(lay.shard for lay in oracle_layouts(w))
