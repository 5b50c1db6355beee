"""Sharded checkpoints of RankShardOptimizer state.

Each rank writes the shards it owns -- fp32 master weights and both AdamW
moments of every unit -- to a file of its own, with the step count and every
unit's element count; a load under another rank count (or sharding factor)
reads, for each unit, only the pieces of the saved shards that make up the
new rank's shard.  File format, checksums and the reshard plan are native
(libshardstep: shardstep_ckpt_*, fsdp_reshard_plan); this module stages the
device state through pinned host memory.

Under hybrid sharding the F shards of one group are saved (the other groups
hold identical replicas); a load into any sharding factor works the same way.
"""
from __future__ import annotations

import ctypes
import os
import threading
import weakref
from concurrent.futures import ThreadPoolExecutor

from . import _capi

KIND_MASTER, KIND_M, KIND_V = 0, 1, 2
_KINDS = (KIND_MASTER, KIND_M, KIND_V)

# pinned host staging per optimizer, kept for its next save or load: pinning
# ~12 bytes per shard element costs more than the copies and the file IO
_STAGING = weakref.WeakKeyDictionary()
_STAGING_LOCK = threading.Lock()


def _staging(opt):
    import torch
    with _STAGING_LOCK:
        bufs = _STAGING.get(opt)
    if bufs is None or bufs[0].numel() != opt.shard_total:
        bufs = [torch.empty(opt.shard_total, dtype=torch.float32, pin_memory=True)
                for _ in _KINDS]
        with _STAGING_LOCK:
            _STAGING[opt] = bufs
    return bufs


def release_staging(opt) -> None:
    """Drop ``opt``'s pinned staging buffers (they are reused by every later
    save and load of the same optimizer until then)."""
    with _STAGING_LOCK:
        _STAGING.pop(opt, None)


def rank_file(directory: str, rank: int) -> str:
    return os.path.join(directory, f"rank{rank:05d}.shst")


def _states(opt):
    return (opt.master, opt.m, opt.v)


def _step_count(opt) -> int:
    """The optimizer's step count: the device step state's when it has one
    (``step_on_device`` advances that one only; reading it synchronises),
    else the host count."""
    state = getattr(opt, "state", None)
    return state.step() if state is not None else opt.t


def save_rank(directory: str, opt) -> str:
    """Write ``opt``'s shard state and step count to ``directory`` (rank =
    opt.rank of opt.F shards).  Synchronises with the device."""
    import torch
    os.makedirs(directory, exist_ok=True)
    host = _staging(opt)
    for buf, h in zip(_states(opt), host):
        h.copy_(buf, non_blocking=True)
    torch.cuda.synchronize(opt.master.device)
    n_units = len(opt.layouts)
    secs = (_capi.CkptSection * max(1, 3 * n_units))()
    k = 0
    for u, lay in enumerate(opt.layouts):
        for kind, h in zip(_KINDS, host):
            secs[k] = _capi.CkptSection(u, kind, lay.shard * 4, h.data_ptr() + opt.starts[u] * 4)
            k += 1
    path = rank_file(directory, opt.rank)
    _capi.check("shardstep_ckpt_save_rank", _capi.lib().shardstep_ckpt_save_rank(
        path.encode(), opt.F, opt.rank, _step_count(opt),
        _capi.i64_array([l.total for l in opt.layouts]),
        n_units, secs, k))
    return path


def save(directory: str, opts, threads: int = 8):
    """Write every rank of a checkpoint (one optimizer per rank of one shard
    group), ranks in parallel."""
    with ThreadPoolExecutor(max(1, min(threads, len(opts)))) as ex:
        return list(ex.map(lambda o: save_rank(directory, o), opts))


def info(directory: str, rank: int = 0):
    """(nd, step, unit totals) of a saved checkpoint."""
    inf = _capi.CkptInfo()
    path = rank_file(directory, rank).encode()
    L = _capi.lib()
    _capi.check("shardstep_ckpt_info", L.shardstep_ckpt_info(path, ctypes.byref(inf), None, 0))
    totals = (_capi.c_i64 * max(1, inf.n_units))()
    _capi.check("shardstep_ckpt_info", L.shardstep_ckpt_info(path, ctypes.byref(inf), totals,
                                                             inf.n_units))
    return inf.nd, inf.step, list(totals[:inf.n_units])


def verify(directory: str) -> None:
    """Check every section checksum of every rank file (raises on a mismatch)."""
    nd, _, _ = info(directory)
    for r in range(nd):
        _capi.check("shardstep_ckpt_verify",
                    _capi.lib().shardstep_ckpt_verify(rank_file(directory, r).encode()))


def plan(total: int, old_nd: int, new_nd: int, new_rank: int):
    """Reshard pieces (old_rank, old_offset, new_offset, count) of one unit."""
    cap = old_nd + 2
    pieces = (_capi.CkptPiece * cap)()
    n = _capi.c_i32(0)
    _capi.check("fsdp_reshard_plan", _capi.lib().fsdp_reshard_plan(
        total, old_nd, new_nd, new_rank, pieces, cap, ctypes.byref(n)))
    return [(p.old_rank, p.old_offset, p.new_offset, p.count) for p in pieces[:n.value]]


_READ_PIECE = 16 << 20   # bytes per read task, so that the pool stays balanced


def _read_tasks(directory: str, opt, old_nd: int):
    """The reads that fill ``opt``'s pinned staging from the saved rank
    files: (path, unit, kind, byte offset in the section, bytes, destination
    address), at most _READ_PIECE bytes each.  Zeroes the padding positions
    of the new layout (no piece covers them) on the way."""
    host = _staging(opt)
    tasks = []
    for u, lay in enumerate(opt.layouts):
        covered = max(0, min(lay.shard, lay.total - opt.rank * lay.shard))
        for h in host:
            h[opt.starts[u] + covered:opt.starts[u] + lay.shard].zero_()
        for q, off, new_off, count in plan(lay.total, old_nd, opt.F, opt.rank):
            path = rank_file(directory, q).encode()
            for kind, h in zip(_KINDS, host):
                dst = h.data_ptr() + (opt.starts[u] + new_off) * 4
                for b0 in range(0, count * 4, _READ_PIECE):
                    n = min(_READ_PIECE, count * 4 - b0)
                    tasks.append((path, u, kind, off * 4 + b0, n, dst + b0))
    return tasks


def _run_read(task) -> None:
    path, u, kind, off, n, dst = task
    _capi.check("shardstep_ckpt_read", _capi.lib().shardstep_ckpt_read(
        path, u, kind, off, n, ctypes.c_void_p(dst)))


def _finish_load(opt, step: int) -> None:
    """Staging -> device (queued; the caller synchronises), and the step
    count (host and device)."""
    for buf, h in zip(_states(opt), _staging(opt)):
        buf.copy_(h, non_blocking=True)
    opt.t = step
    state = getattr(opt, "state", None)
    if state is not None:                 # the device step state continues from here too
        state.init(step)


def _check_units(opt, totals) -> None:
    if totals != [l.total for l in opt.layouts]:
        raise ValueError("checkpoint units do not match the optimizer's units")


def load_rank(directory: str, opt) -> None:
    """Fill ``opt``'s master / m / v and step count (the host count, and the
    device step state's when it has one) from a checkpoint saved under any
    rank count; padding positions of the new layout are zero."""
    old_nd, step, totals = info(directory)
    _check_units(opt, totals)
    import torch
    for t in _read_tasks(directory, opt, old_nd):
        _run_read(t)
    _finish_load(opt, step)
    torch.cuda.synchronize(opt.master.device)


def load(directory: str, opts, threads: int | None = None) -> None:
    """Load every optimizer (one per rank of the new layout): every rank's
    reads from the saved files go to one pool of ``threads`` workers (default:
    the host's cores; the native reads release the interpreter lock), then
    each rank's state is copied to its device."""
    old_nd, step, totals = info(directory)
    for o in opts:
        _check_units(o, totals)
    tasks = [t for o in opts for t in _read_tasks(directory, o, old_nd)]
    workers = max(1, threads or os.cpu_count() or 1)
    import torch
    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(_run_read, tasks))
    for o in opts:
        _finish_load(o, step)
    for dev in {o.master.device for o in opts}:
        torch.cuda.synchronize(dev)
