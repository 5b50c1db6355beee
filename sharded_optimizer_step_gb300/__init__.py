"""sharded_optimizer_step_gb300 -- the data-parallel hot path of a ZeRO / FSDP
sharded optimizer step over a FlatParameter, as hand-written sm_103a CUDA
kernels behind the C ABI of include/shardstep.h.

This module is argument marshalling only: every step of the path runs in
libshardstep.so.  PyTorch supplies device memory and streams.  Each function
enqueues work on torch's current CUDA stream (or ``stream=``) and returns
without synchronising.

N_d data-parallel ranks are emulated as N_d buffers in one GPU's memory.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from . import _capi
from ._capi import ShardstepError, AdamWHP, MAX_ND
from .build import build

__all__ = [
    "build", "ShardstepError", "AdamW", "Layout", "fsdp_layout", "fsdp_flat_pack", "fsdp_views",
    "fsdp_grad_accumulate", "fsdp_rs_avg_adamw_cast", "fsdp_ag_unpack", "ddp_bucket_plan",
    "ddp_bucket_allreduce_avg", "state_bytes", "comm_bytes", "comm_counter", "launch_count",
    "last_kernel",
    "MAX_ND",
    "set_fused_path", "device_status", "fsdp_hybrid_rs_avg_adamw_cast", "hybrid_state_bytes",
    "hybrid_comm_bytes", "Fsdp2Layout", "fsdp2_layout", "fsdp2_local_views", "fsdp2_chunk_cat",
    "fsdp2_all_gather_copy_out", "AdamWState", "fsdp_state_rs_avg_adamw_cast",
    "fsdp_accumulate_rs_avg_adamw_cast", "fsdp_state_accumulate_rs_avg_adamw_cast",
    "ddp_bucket_allreduce_avg_adamw_cast", "set_tma_wait_ns", "check_mean_division",
    "fsdp_shard_pieces", "fsdp2_rs_avg_adamw_cast", "Fsdp2Step",
]


@dataclass
class AdamW:
    """AdamW hyper-parameters (decoupled weight decay, bias-corrected moments)."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01

    def at_step(self, step: int) -> AdamWHP:
        return AdamWHP(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, int(step))


@dataclass
class Layout:
    numels: list
    nd: int
    total: int
    padded: int
    shard: int
    offsets: list
    lo: list   # lo[r][t]
    hi: list   # hi[r][t]


def _stream(stream, device=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return _capi.DTYPE_BF16
    if t.dtype == torch.float32:
        return _capi.DTYPE_F32
    if t.dtype == torch.float16:
        return _capi.DTYPE_F16
    raise TypeError(f"unsupported dtype {t.dtype} (bf16, fp16 or fp32)")


def _group(shard_group, nd):
    """The sharding factor passed to the C ABI: None means full sharding
    (F = N_d); any other value goes through as given, so that the library
    rejects 0, negative factors and factors that do not divide N_d."""
    return nd if shard_group is None else int(shard_group)


def _need_cuda(*tensors):
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("expected CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("expected contiguous tensors")


# ---------------------------------------------------------------- layout

def fsdp_layout(numels, nd: int) -> Layout:
    """FlatParameter layout of one FSDP unit (host only)."""
    L = _capi.lib()
    n = len(numels)
    info = _capi.LayoutInfo()
    off = (_capi.c_i64 * max(1, n))()
    lo = (_capi.c_i64 * max(1, n * max(nd, 1)))()
    hi = (_capi.c_i64 * max(1, n * max(nd, 1)))()
    _capi.check("fsdp_layout", L.fsdp_layout(_capi.i64_array(numels), n, nd, ctypes.byref(info),
                                             off, lo, hi))
    return Layout(list(int(x) for x in numels), nd, info.total, info.padded, info.shard,
                  list(off[:n]), [list(lo[r * n:(r + 1) * n]) for r in range(nd)],
                  [list(hi[r * n:(r + 1) * n]) for r in range(nd)])


def fsdp_shard_pieces(numels, nd: int, rank: int):
    """Per tensor of a unit, the piece that rank ``rank`` holds: a list of
    (position in the rank's shard, first element within the tensor, length)
    (length 0: the rank holds nothing of that tensor).  Host only."""
    L = _capi.lib()
    n = len(numels)
    slo = (_capi.c_i64 * max(1, n))()
    tlo = (_capi.c_i64 * max(1, n))()
    cnt = (_capi.c_i64 * max(1, n))()
    _capi.check("fsdp_shard_pieces", L.fsdp_shard_pieces(_capi.i64_array(numels), n, nd, rank,
                                                         slo, tlo, cnt))
    return [(int(slo[t]), int(tlo[t]), int(cnt[t])) for t in range(n)]


def fsdp_flat_pack(tensors, nd: int, flat=None, stream=None):
    """Flatten + concatenate + zero-pad one unit's tensors (all bf16 or all
    fp32) into ``flat`` (allocated with torch if None).  Returns flat."""
    import torch
    if not tensors:
        raise ValueError("empty unit")
    dt = tensors[0].dtype
    if any(t.dtype != dt for t in tensors):
        raise TypeError("one dtype per unit")
    _need_cuda(*tensors)
    numels = [t.numel() for t in tensors]
    lay = fsdp_layout(numels, nd)
    if flat is None:
        flat = torch.empty(lay.padded, dtype=dt, device=tensors[0].device)
    _need_cuda(flat)
    if flat.dtype != dt or flat.numel() != lay.padded:
        raise ValueError(f"flat must be {dt} with {lay.padded} elements")
    L = _capi.lib()
    _capi.check("fsdp_flat_pack", L.fsdp_flat_pack(
        _capi.ptr_array([t.data_ptr() for t in tensors]), _capi.i64_array(numels), len(tensors),
        nd, _dtype_code(flat), ctypes.c_void_p(flat.data_ptr()), _stream(stream, flat.device)))
    return flat


def fsdp_views(buf, shapes, nd: int, rank: int = -1):
    """Per-tensor views into ``buf``: the full flat buffer (rank < 0, views
    reshaped to ``shapes``) or rank ``rank``'s shard (1-D pieces, possibly
    empty), as use_orig_params exposes them."""
    L = _capi.lib()
    numels = []
    for s in shapes:
        n = 1
        for d in s:
            n *= int(d)
        numels.append(n)
    n = len(numels)
    ptrs = (_capi.c_vp * max(1, n))()
    counts = (_capi.c_i64 * max(1, n))()
    es = buf.element_size()
    _capi.check("fsdp_views", L.fsdp_views(_capi.i64_array(numels), n, nd, rank,
                                           ctypes.c_void_p(buf.data_ptr()), es, ptrs, counts))
    views = []
    base = buf.data_ptr()
    for t in range(n):
        off = ((ptrs[t] or 0) - base) // es
        v = buf[off:off + counts[t]]
        views.append(v.view(tuple(shapes[t])) if rank < 0 else v)
    return views


# ---------------------------------------------------------- accumulation

def fsdp_grad_accumulate(g, acc, scale: float, first: bool, stream=None):
    """acc = g*scale (first) or acc + g*scale; g bf16, acc fp32, same numel."""
    import torch
    _need_cuda(g, acc)
    if g.dtype != torch.bfloat16 or acc.dtype != torch.float32 or g.numel() != acc.numel():
        raise ValueError("g must be bf16 and acc fp32 with the same numel")
    _capi.check("fsdp_grad_accumulate", _capi.lib().fsdp_grad_accumulate(
        ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(acc.data_ptr()), g.numel(),
        ctypes.c_float(scale), int(bool(first)), _stream(stream, g.device)))


# --------------------------------------------------------- the fused step

def fsdp_rs_avg_adamw_cast(grad_slices, master, m, v, out_bf16, hp: AdamW, step: int,
                           stream=None):
    """Reduce-scatter average of the N_d gradient slices, AdamW on the fp32
    shard (in place) and the bf16 cast into ``out_bf16``, in one kernel pass.
    ``grad_slices[q]`` is rank q's contribution to this shard (S elements,
    all bf16 or all fp32)."""
    _fused(grad_slices, master, m, v, out_bf16, hp, step, stream, None)


def fsdp_accumulate_rs_avg_adamw_cast(acc_slices, last_slices, scale: float, master, m, v,
                                      out_bf16, hp: AdamW, step: int,
                                      shard_group: int | None = None, stream=None):
    """The last micro-batch accumulated and the shard stepped in one pass:
    rank q's contribution is ``acc_slices[q] + last_slices[q] * scale`` (fp32
    accumulators of micro-batches 0..M-2, bf16 gradients of the last one,
    ``scale`` = 1/M), then the step of ``fsdp_rs_avg_adamw_cast`` (of the
    hybrid step with ``shard_group`` = F).  The accumulators are read, not
    written."""
    S = _accum_args(acc_slices, last_slices, master, m, v, out_bf16)
    hpc = hp.at_step(step)
    _capi.check("fsdp_accumulate_rs_avg_adamw_cast",
                _capi.lib().fsdp_accumulate_rs_avg_adamw_cast(
                    *_accum_ptrs(acc_slices, last_slices, shard_group, S, scale, master, m, v,
                                 out_bf16),
                    ctypes.byref(hpc), _stream(stream, master.device)))


def fsdp_state_accumulate_rs_avg_adamw_cast(acc_slices, last_slices, scale: float, master, m,
                                            v, out_bf16, state: AdamWState,
                                            shard_group: int | None = None, stream=None):
    """``fsdp_accumulate_rs_avg_adamw_cast`` with the AdamW scalars read on the
    device from ``state`` (at a step >= 1): CUDA-graph capturable."""
    S = _accum_args(acc_slices, last_slices, master, m, v, out_bf16)
    _need_cuda(state.buf)
    _capi.check("fsdp_state_accumulate_rs_avg_adamw_cast",
                _capi.lib().fsdp_state_accumulate_rs_avg_adamw_cast(
                    *_accum_ptrs(acc_slices, last_slices, shard_group, S, scale, master, m, v,
                                 out_bf16),
                    ctypes.c_void_p(state.buf.data_ptr()), _stream(stream, master.device)))


def _accum_ptrs(acc_slices, last_slices, shard_group, S, scale, master, m, v, out_bf16):
    nd = len(acc_slices)
    return (_capi.ptr_array([a.data_ptr() for a in acc_slices]),
            _capi.ptr_array([g.data_ptr() for g in last_slices]), nd,
            _group(shard_group, nd), S,
            ctypes.c_float(scale), ctypes.c_void_p(master.data_ptr()),
            ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(out_bf16.data_ptr()))


def _accum_args(acc_slices, last_slices, master, m, v, out_bf16):
    import torch
    if not acc_slices or len(acc_slices) != len(last_slices):
        raise ValueError("need as many accumulator slices as last-micro-batch slices (>= 1)")
    _need_cuda(*acc_slices, *last_slices, master, m, v, out_bf16)
    S = master.numel()
    for a, g in zip(acc_slices, last_slices):
        if a.dtype != torch.float32 or g.dtype != torch.bfloat16 or a.numel() != S \
                or g.numel() != S:
            raise ValueError("accumulator slices fp32, last slices bf16, S elements each")
    for t in (master, m, v):
        if t.dtype != torch.float32 or t.numel() != S:
            raise ValueError("master / m / v must be fp32 with S elements")
    if out_bf16.dtype != torch.bfloat16 or out_bf16.numel() != S:
        raise ValueError("out_bf16 must be bf16 with S elements")
    return S


def fsdp_hybrid_rs_avg_adamw_cast(grad_slices, shard_group: int, master, m, v, out_bf16,
                                  hp: AdamW, step: int, stream=None):
    """Hybrid sharding with sharding factor F = ``shard_group``: the N_d
    contributions (rank order k = g*F + j) are summed inside each group of F,
    then across the groups, averaged over N_d, and the shard is updated and
    cast as in ``fsdp_rs_avg_adamw_cast``."""
    _fused(grad_slices, master, m, v, out_bf16, hp, step, stream, int(shard_group))


def _fused(grad_slices, master, m, v, out_bf16, hp, step, stream, shard_group):
    import torch
    if not grad_slices:
        raise ValueError("need at least one gradient slice")
    _need_cuda(*grad_slices, master, m, v, out_bf16)
    S = master.numel()
    gd = grad_slices[0].dtype
    for g in grad_slices:
        if g.dtype != gd or g.numel() != S:
            raise ValueError("gradient slices must share dtype and have S elements")
    for t in (m, v):
        if t.dtype != torch.float32 or t.numel() != S:
            raise ValueError("master / m / v must be fp32 with S elements")
    if master.dtype != torch.float32 or out_bf16.dtype != torch.bfloat16 or out_bf16.numel() != S:
        raise ValueError("master fp32 and out bf16 with S elements")
    hpc = hp.at_step(step)
    ptrs = _capi.ptr_array([g.data_ptr() for g in grad_slices])
    state = (ctypes.c_void_p(master.data_ptr()), ctypes.c_void_p(m.data_ptr()),
             ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out_bf16.data_ptr()))
    if shard_group is None:
        _capi.check("fsdp_rs_avg_adamw_cast", _capi.lib().fsdp_rs_avg_adamw_cast(
            ptrs, _dtype_code(grad_slices[0]), len(grad_slices), S, *state, ctypes.byref(hpc),
            _stream(stream, master.device)))
    else:
        _capi.check("fsdp_hybrid_rs_avg_adamw_cast", _capi.lib().fsdp_hybrid_rs_avg_adamw_cast(
            ptrs, _dtype_code(grad_slices[0]), len(grad_slices), shard_group, S, *state,
            ctypes.byref(hpc), _stream(stream, master.device)))


class AdamWState:
    """The AdamW step count and its fp32 scalars in device memory
    (``shardstep_adamw_state_t``), so that a step needs no host work:
    ``advance`` then ``fsdp_state_rs_avg_adamw_cast`` (and the all-gather)
    can be captured in a CUDA graph once and replayed every iteration.
    The hyper-parameters are passed by value at each ``advance``; a captured
    graph replays the ones it was captured with."""

    def __init__(self, hp: AdamW, step: int = 0, device="cuda", stream=None):
        import torch
        self.hp = hp
        # 56 bytes, 8-byte aligned
        self.buf = torch.zeros(_capi.ADAMW_STATE_BYTES // 8, dtype=torch.float64, device=device)
        self.init(step, stream)

    def init(self, step: int, stream=None):
        """Set the state to step ``step`` (>= 0; scalars too from step 1)."""
        _capi.check("shardstep_adamw_state_init", _capi.lib().shardstep_adamw_state_init(
            ctypes.c_void_p(self.buf.data_ptr()), ctypes.byref(self.hp.at_step(1)), int(step),
            _stream(stream, self.buf.device)))

    def advance(self, skip=None, stream=None):
        """Step t -> t + 1 on the device; with ``skip`` (a device int32 word,
        e.g. a GradScaler's ``found_inf``) non-zero when it runs, no change."""
        if skip is not None:
            _need_cuda(skip)
        _capi.check("shardstep_adamw_state_advance", _capi.lib().shardstep_adamw_state_advance(
            ctypes.c_void_p(self.buf.data_ptr()), ctypes.byref(self.hp.at_step(1)),
            ctypes.c_void_p(skip.data_ptr() if skip is not None else None),
            _stream(stream, self.buf.device)))

    def step(self) -> int:
        """The current step count (reads the device; synchronises)."""
        import torch
        return int(self.buf[:1].view(torch.int64).item())


def fsdp_state_rs_avg_adamw_cast(grad_slices, master, m, v, out_bf16, state: AdamWState,
                                 shard_group: int | None = None, stream=None):
    """The fused step (hybrid with ``shard_group`` = F) with the AdamW scalars
    read on the device from ``state``, which must be at a step >= 1."""
    import torch
    if not grad_slices:
        raise ValueError("need at least one gradient slice")
    _need_cuda(*grad_slices, master, m, v, out_bf16, state.buf)
    S = master.numel()
    for g in grad_slices:
        if g.dtype != grad_slices[0].dtype or g.numel() != S:
            raise ValueError("gradient slices must share dtype and have S elements")
    for t in (master, m, v):
        if t.dtype != torch.float32 or t.numel() != S:
            raise ValueError("master / m / v must be fp32 with S elements")
    if out_bf16.dtype != torch.bfloat16 or out_bf16.numel() != S:
        raise ValueError("out must be bf16 with S elements")
    _capi.check("fsdp_state_rs_avg_adamw_cast", _capi.lib().fsdp_state_rs_avg_adamw_cast(
        _capi.ptr_array([g.data_ptr() for g in grad_slices]), _dtype_code(grad_slices[0]),
        len(grad_slices), _group(shard_group, len(grad_slices)), S,
        ctypes.c_void_p(master.data_ptr()),
        ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out_bf16.data_ptr()), ctypes.c_void_p(state.buf.data_ptr()),
        _stream(stream, master.device)))


# -------------------------------------------------------- gradient scaler

class GradScaler:
    """Sharded dynamic loss scaling over the emulated ranks (fp16 gradients):
    device words for the scale, the growth tracker and the found-inf flag,
    and the three C-ABI calls of one step.  Nothing synchronises with the
    host; read ``scale`` / ``found_inf`` when needed."""

    def __init__(self, init_scale: float = 65536.0, growth_factor: float = 2.0,
                 backoff_factor: float = 0.5, growth_interval: int = 2000, device="cuda"):
        import torch
        self.scale = torch.tensor([init_scale], dtype=torch.float32, device=device)
        self.tracker = torch.zeros(1, dtype=torch.int32, device=device)
        self.found_inf = torch.zeros(1, dtype=torch.int32, device=device)
        self.growth_factor, self.backoff_factor = growth_factor, backoff_factor
        self.growth_interval = growth_interval

    def check(self, grad_slices, shard_group: int | None = None, stream=None):
        """OR this shard's non-finite flag (of the mean times 1/scale) into
        ``found_inf``."""
        _need_cuda(*grad_slices)
        S = grad_slices[0].numel()
        nd = len(grad_slices)
        _capi.check("fsdp_grad_unscale_check", _capi.lib().fsdp_grad_unscale_check(
            _capi.ptr_array([g.data_ptr() for g in grad_slices]), _dtype_code(grad_slices[0]),
            nd, _group(shard_group, nd), S, ctypes.c_void_p(self.scale.data_ptr()),
            ctypes.c_void_p(self.found_inf.data_ptr()), _stream(stream, grad_slices[0].device)))

    def step(self, grad_slices, master, m, v, out_bf16, hp: AdamW, step: int,
             shard_group: int | None = None, stream=None):
        """The fused update on the unscaled gradient, skipped on the device
        when any rank's check found inf/NaN."""
        _need_cuda(*grad_slices, master, m, v, out_bf16)
        S = master.numel()
        nd = len(grad_slices)
        hpc = hp.at_step(step)
        _capi.check("fsdp_scaled_rs_avg_adamw_cast", _capi.lib().fsdp_scaled_rs_avg_adamw_cast(
            _capi.ptr_array([g.data_ptr() for g in grad_slices]), _dtype_code(grad_slices[0]),
            nd, _group(shard_group, nd), S, ctypes.c_void_p(master.data_ptr()),
            ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(out_bf16.data_ptr()), ctypes.byref(hpc),
            ctypes.c_void_p(self.scale.data_ptr()), ctypes.c_void_p(self.found_inf.data_ptr()),
            _stream(stream, master.device)))

    def step_state(self, grad_slices, master, m, v, out_bf16, state, shard_group: int | None = None,
                   stream=None):
        """``step`` with the AdamW scalars read on the device from ``state``
        (an ``AdamWState``): with ``check`` before it, ``state.advance(
        skip=self.found_inf)`` and ``update`` after, a loss-scaled step made
        of device words only, which a CUDA graph can capture."""
        _need_cuda(*grad_slices, master, m, v, out_bf16, state.buf)
        S = master.numel()
        nd = len(grad_slices)
        _capi.check("fsdp_state_scaled_rs_avg_adamw_cast",
                    _capi.lib().fsdp_state_scaled_rs_avg_adamw_cast(
                        _capi.ptr_array([g.data_ptr() for g in grad_slices]),
                        _dtype_code(grad_slices[0]), nd, _group(shard_group, nd), S,
                        ctypes.c_void_p(master.data_ptr()), ctypes.c_void_p(m.data_ptr()),
                        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out_bf16.data_ptr()),
                        ctypes.c_void_p(state.buf.data_ptr()),
                        ctypes.c_void_p(self.scale.data_ptr()),
                        ctypes.c_void_p(self.found_inf.data_ptr()),
                        _stream(stream, master.device)))

    def update(self, stream=None):
        """Back off or grow the scale and reset ``found_inf``."""
        _capi.check("fsdp_grad_scaler_update", _capi.lib().fsdp_grad_scaler_update(
            ctypes.c_void_p(self.scale.data_ptr()), ctypes.c_void_p(self.tracker.data_ptr()),
            ctypes.c_void_p(self.found_inf.data_ptr()), ctypes.c_float(self.growth_factor),
            ctypes.c_float(self.backoff_factor), self.growth_interval,
            _stream(stream, self.scale.device)))


# ------------------------------------------------------------- all-gather

def fsdp_ag_unpack(shards, full, stream=None):
    """full[q*S:(q+1)*S] = shards[q] for every rank q (bf16).  A shard that
    already is its slot of ``full`` is not copied."""
    import torch
    _need_cuda(*shards, full)
    nd = len(shards)
    S = shards[0].numel()
    if any(s.numel() != S or s.dtype != torch.bfloat16 for s in shards):
        raise ValueError("shards must be bf16 with equal numel")
    if full.dtype != torch.bfloat16 or full.numel() != nd * S:
        raise ValueError("full must be bf16 with nd*S elements")
    _capi.check("fsdp_ag_unpack", _capi.lib().fsdp_ag_unpack(
        _capi.ptr_array([s.data_ptr() for s in shards]), nd, S, ctypes.c_void_p(full.data_ptr()),
        _stream(stream, full.device)))
    return full


# ----------------------------------------------------------------- FSDP2

def _dims(shapes):
    d0, row = [], []
    for s in shapes:
        s = tuple(int(d) for d in s)
        if not s:
            raise ValueError("scalar parameters have no dim 0")
        r = 1
        for d in s[1:]:
            r *= d
        d0.append(s[0])
        row.append(r)
    return d0, row


@dataclass
class Fsdp2Layout:
    shapes: list
    nd: int
    chunk: list     # rows per rank of each parameter
    offset: list    # element offset of each parameter in a rank's local buffer
    local: int      # elements of a rank's local buffer


def fsdp2_layout(shapes, nd: int) -> Fsdp2Layout:
    """Per-parameter dim-0 sharding of one group (host only)."""
    d0, row = _dims(shapes)
    n = len(shapes)
    chunk = (_capi.c_i64 * max(1, n))()
    off = (_capi.c_i64 * max(1, n))()
    local = _capi.c_i64(0)
    _capi.check("fsdp2_layout", _capi.lib().fsdp2_layout(
        _capi.i64_array(d0), _capi.i64_array(row), n, nd, chunk, off, ctypes.byref(local)))
    return Fsdp2Layout([tuple(s) for s in shapes], nd, list(chunk[:n]), list(off[:n]),
                       local.value)


def fsdp2_local_views(buf, shapes, nd: int, rank: int):
    """Rank ``rank``'s local tensors (rows, trailing dims) inside its local
    buffer, as DTensor.to_local() shows them."""
    d0, row = _dims(shapes)
    n = len(shapes)
    ptrs = (_capi.c_vp * max(1, n))()
    rows = (_capi.c_i64 * max(1, n))()
    es = buf.element_size()
    _capi.check("fsdp2_local_views", _capi.lib().fsdp2_local_views(
        _capi.i64_array(d0), _capi.i64_array(row), n, nd, rank, ctypes.c_void_p(buf.data_ptr()),
        es, ptrs, rows))
    out = []
    for t, s in enumerate(shapes):
        off = ((ptrs[t] or buf.data_ptr()) - buf.data_ptr()) // es
        k = rows[t] * row[t]
        out.append(buf[off:off + k].view((rows[t],) + tuple(s[1:])))
    return out


def fsdp2_chunk_cat(grads, nd: int, out=None, stream=None):
    """One rank's reduce-scatter input of a group: nd rank pieces of the
    local length, each rank's rows of every gradient zero-padded."""
    import torch
    _need_cuda(*grads)
    shapes = [tuple(g.shape) for g in grads]
    lay = fsdp2_layout(shapes, nd)
    if out is None:
        out = torch.empty(nd * lay.local, dtype=grads[0].dtype, device=grads[0].device)
    _need_cuda(out)
    if out.numel() != nd * lay.local or any(g.dtype != out.dtype for g in grads):
        raise ValueError("out must have nd * local elements of the gradients' dtype")
    d0, row = _dims(shapes)
    _capi.check("fsdp2_chunk_cat", _capi.lib().fsdp2_chunk_cat(
        _capi.ptr_array([g.data_ptr() for g in grads]), _capi.i64_array(d0), _capi.i64_array(row),
        len(grads), nd, _dtype_code(out), ctypes.c_void_p(out.data_ptr()),
        _stream(stream, out.device)))
    return out


def fsdp2_rs_avg_adamw_cast(rank_grads, rank: int, master, m, v, out_bf16, hp: AdamW, step: int,
                            stream=None):
    """Rank ``rank``'s FSDP2 step read straight from every rank's full
    per-parameter gradients (``rank_grads[q][t]``: rank q's gradient of
    parameter t, global shape): the bits of ``fsdp2_chunk_cat`` of each
    rank's gradients followed by ``fsdp_rs_avg_adamw_cast`` on the rank's
    pieces, without the chunk-cat copy.  ``master`` / ``m`` / ``v`` /
    ``out_bf16`` are the rank's padded local buffers.  For repeated steps
    over the same gradient buffers, ``Fsdp2Step`` checks them once."""
    Fsdp2Step(rank_grads)(rank, master, m, v, out_bf16, hp, step, stream)


class Fsdp2Step:
    """``fsdp2_rs_avg_adamw_cast`` over one group's gradient buffers, checked
    once: the ranks' per-parameter gradient tensors (``rank_grads[q][t]``)
    are validated and their device pointers, shapes and the local length
    taken when the object is made, and it keeps the tensors alive.  Each
    call then checks only that no gradient's storage has moved and the
    rank's four local buffers before the C call (which checks every pointer
    again), so a step of many small parameters costs little host time."""

    def __init__(self, rank_grads):
        import torch
        self.nd = len(rank_grads)
        if self.nd == 0:
            raise ValueError("need at least one rank")
        self.shapes = [tuple(g.shape) for g in rank_grads[0]]
        dt = rank_grads[0][0].dtype if self.shapes else torch.bfloat16
        for gs in rank_grads:
            _need_cuda(*gs)
            if [tuple(g.shape) for g in gs] != self.shapes or any(g.dtype != dt for g in gs):
                raise ValueError("every rank's gradients must have the same shapes and dtype")
        self._keep = [g for gs in rank_grads for g in gs]
        self._addrs = [g.data_ptr() for g in self._keep]
        self.local = fsdp2_layout(self.shapes, self.nd).local
        d0, row = _dims(self.shapes)
        self._d0, self._row = _capi.i64_array(d0), _capi.i64_array(row)
        self._ptrs = _capi.ptr_array(self._addrs)
        self._code = _dtype_code(rank_grads[0][0]) if self.shapes else _capi.DTYPE_BF16

    def _check(self, master, m, v, out_bf16):
        import torch
        L = self.local
        for t in (master, m, v):
            if not t.is_cuda or t.dtype != torch.float32 or t.numel() != L or not t.is_contiguous():
                raise ValueError(f"master / m / v must be contiguous CUDA fp32 with {L} elements")
        if (not out_bf16.is_cuda or out_bf16.dtype != torch.bfloat16 or out_bf16.numel() != L
                or not out_bf16.is_contiguous()):
            raise ValueError(f"out must be contiguous CUDA bf16 with {L} elements")
        # a gradient whose storage moved (an in-place resize) would leave a
        # stale pointer in the table
        if any(g.data_ptr() != a for g, a in zip(self._keep, self._addrs)):
            raise ValueError("a gradient buffer moved since this Fsdp2Step was made")

    def __call__(self, rank: int, master, m, v, out_bf16, hp: AdamW, step: int, stream=None):
        """Rank ``rank``'s step at step count ``step`` (host scalars)."""
        self._check(master, m, v, out_bf16)
        hpc = hp.at_step(step)
        _capi.check("fsdp2_rs_avg_adamw_cast", _capi.lib().fsdp2_rs_avg_adamw_cast(
            self._ptrs, self._code, self._d0, self._row, len(self.shapes), self.nd, int(rank),
            ctypes.c_void_p(master.data_ptr()), ctypes.c_void_p(m.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out_bf16.data_ptr()),
            ctypes.byref(hpc), _stream(stream, master.device)))

    def step_state(self, rank: int, master, m, v, out_bf16, state: AdamWState, stream=None):
        """Rank ``rank``'s step with the AdamW scalars read on the device from
        ``state`` (an ``AdamWState`` at a step >= 1): with ``state.advance()``
        before the ranks' calls, a step a CUDA graph can capture."""
        self._check(master, m, v, out_bf16)
        _need_cuda(state.buf)
        _capi.check("fsdp2_state_rs_avg_adamw_cast", _capi.lib().fsdp2_state_rs_avg_adamw_cast(
            self._ptrs, self._code, self._d0, self._row, len(self.shapes), self.nd, int(rank),
            ctypes.c_void_p(master.data_ptr()), ctypes.c_void_p(m.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out_bf16.data_ptr()),
            ctypes.c_void_p(state.buf.data_ptr()), _stream(stream, master.device)))


def fsdp2_all_gather_copy_out(local_bufs, params, stream=None):
    """All-gather the ranks' local buffers straight into the full
    per-parameter tensors ``params`` (global shapes)."""
    _need_cuda(*local_bufs, *params)
    shapes = [tuple(p.shape) for p in params]
    nd = len(local_bufs)
    lay = fsdp2_layout(shapes, nd)
    if any(b.numel() != lay.local or b.dtype != params[0].dtype for b in local_bufs):
        raise ValueError("local buffers must have the local length and the params' dtype")
    d0, row = _dims(shapes)
    _capi.check("fsdp2_all_gather_copy_out", _capi.lib().fsdp2_all_gather_copy_out(
        _capi.ptr_array([b.data_ptr() for b in local_bufs]), _capi.i64_array(d0),
        _capi.i64_array(row), len(params), nd, _dtype_code(params[0]),
        _capi.ptr_array([p.data_ptr() for p in params]), _stream(stream, params[0].device)))
    return params


# ----------------------------------------------------------- DDP buckets

def ddp_bucket_plan(numels, elem_size: int, cap_bytes: int):
    """Greedy reverse-order buckets.  Returns (param_offset, bucket_of_param,
    bucket_offsets) as lists; bucket_offsets has n_buckets + 1 entries."""
    L = _capi.lib()
    n = len(numels)
    off = (_capi.c_i64 * max(1, n))()
    of = (_capi.c_i32 * max(1, n))()
    boff = (_capi.c_i64 * (n + 1))()
    nb = _capi.c_i32(0)
    _capi.check("ddp_bucket_plan", L.ddp_bucket_plan(_capi.i64_array(numels), n, elem_size,
                                                     cap_bytes, off, of, boff, ctypes.byref(nb)))
    return list(off[:n]), list(of[:n]), list(boff[:nb.value + 1])


def ddp_bucket_allreduce_avg(rank_grads, bucket_offsets, out, first: int = 0,
                             count: int | None = None, stream=None):
    """Bucket-by-bucket all-reduce average of the ranks' bf16 gradients into
    ``out`` (one kernel launch per non-empty bucket)."""
    import torch
    _need_cuda(*rank_grads, out)
    if any(g.dtype != torch.bfloat16 for g in rank_grads) or out.dtype != torch.bfloat16:
        raise ValueError("bf16 gradients")
    nb = len(bucket_offsets) - 1
    if count is None:
        count = nb - first
    if first < 0 or count < 0 or first + count > nb:
        raise ValueError("bucket range out of bounds")
    total = bucket_offsets[first + count] if nb >= 0 else 0
    if out.numel() < total or any(g.numel() < total for g in rank_grads):
        raise ValueError("buffers shorter than the bucketed range")
    _capi.check("ddp_bucket_allreduce_avg", _capi.lib().ddp_bucket_allreduce_avg(
        _capi.ptr_array([g.data_ptr() for g in rank_grads]), len(rank_grads),
        _capi.i64_array(bucket_offsets), first, count, ctypes.c_void_p(out.data_ptr()),
        _stream(stream, out.device)))
    return out


def ddp_bucket_allreduce_avg_adamw_cast(rank_grads, bucket_offsets, master, m, v, params,
                                        hp: AdamW, step: int, mean_out=None, first: int = 0,
                                        count: int | None = None, stream=None):
    """The bucket all-reduce average of buckets first..first+count-1 fused with
    the replicated AdamW + bf16 cast of the same elements (one launch): the
    bits of ``ddp_bucket_allreduce_avg`` followed by the fused step at
    N_d = 1 on its output.  ``mean_out`` (optional) receives the bf16 mean."""
    import torch
    _need_cuda(*rank_grads, master, m, v, params, mean_out)
    if any(g.dtype != torch.bfloat16 for g in rank_grads) or params.dtype != torch.bfloat16:
        raise ValueError("bf16 gradients and parameters")
    if any(t.dtype != torch.float32 for t in (master, m, v)):
        raise ValueError("master / m / v must be fp32")
    if mean_out is not None and mean_out.dtype != torch.bfloat16:
        raise ValueError("mean_out must be bf16")
    nb = len(bucket_offsets) - 1
    if count is None:
        count = nb - first
    if first < 0 or count < 0 or first + count > nb:
        raise ValueError("bucket range out of bounds")
    total = bucket_offsets[first + count] if nb >= 0 else 0
    bufs = [*rank_grads, master, m, v, params] + ([mean_out] if mean_out is not None else [])
    if any(t.numel() < total for t in bufs):
        raise ValueError("buffers shorter than the bucketed range")
    hpc = hp.at_step(step)
    _capi.check("ddp_bucket_allreduce_avg_adamw_cast",
                _capi.lib().ddp_bucket_allreduce_avg_adamw_cast(
                    _capi.ptr_array([g.data_ptr() for g in rank_grads]), len(rank_grads),
                    _capi.i64_array(bucket_offsets), first, count,
                    ctypes.c_void_p(mean_out.data_ptr() if mean_out is not None else None),
                    ctypes.c_void_p(master.data_ptr()), ctypes.c_void_p(m.data_ptr()),
                    ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(params.data_ptr()),
                    ctypes.byref(hpc), _stream(stream, master.device)))


class BucketNotReady(TimeoutError):
    """A bucket's wait ran out: `rank` never marked `param` ready."""

    def __init__(self, msg, bucket, rank, param):
        super().__init__(msg)
        self.bucket, self.rank, self.param = bucket, rank, param


class BucketReadiness:
    """Host-side readiness of the DDP buckets across N_d emulated ranks
    (libshardstep's ddp_ready_*): ranks -- host threads -- mark parameters
    whose gradients they have; a bucket's all-reduce is launched only after
    ``wait`` saw every rank's every parameter of it.  Marks and waits release
    the interpreter lock, so rank threads run while a caller waits."""

    def __init__(self, bucket_of_param, n_buckets: int, nd: int):
        L = _capi.lib()
        n = int(L.ddp_ready_bytes(len(bucket_of_param), n_buckets, nd))
        if n < 0:
            raise ValueError("bad parameter / bucket / rank counts")
        self._buf = (ctypes.c_uint64 * ((n + 7) // 8))()     # 8-byte aligned host memory
        self._ptr = ctypes.c_void_p(ctypes.addressof(self._buf))
        self.n_buckets, self.nd = n_buckets, nd
        bop = (_capi.c_i32 * max(1, len(bucket_of_param)))(*[int(b) for b in bucket_of_param])
        _capi.check("ddp_ready_init", L.ddp_ready_init(self._ptr, n, bop, len(bucket_of_param),
                                                       n_buckets, nd))

    def mark(self, rank: int, param: int):
        """Rank `rank` has param's gradient in device memory; returns the
        bucket this completed on every rank, or None.  Mark only once the
        gradient's writes have completed (e.g. after synchronising the
        stream that produced it): the bucket's all-reduce may be launched on
        another stream as soon as the mark completes the bucket."""
        done = _capi.c_i32(-1)
        _capi.check("ddp_ready_mark", _capi.lib().ddp_ready_mark(self._ptr, rank, param,
                                                                 ctypes.byref(done)))
        return done.value if done.value >= 0 else None

    def wait(self, bucket: int, timeout_s: float) -> None:
        """Return once the bucket is ready; raise BucketNotReady after
        timeout_s seconds, naming a (rank, parameter) that never arrived."""
        mr, mp = _capi.c_i32(-1), _capi.c_i32(-1)
        L = _capi.lib()
        rc = L.ddp_ready_wait(self._ptr, bucket, int(timeout_s * 1e6), ctypes.byref(mr),
                              ctypes.byref(mp))
        if rc == _capi.ERR_TIMEOUT:
            raise BucketNotReady(L.shardstep_last_error().decode(), bucket, mr.value, mp.value)
        _capi.check("ddp_ready_wait", rc)

    def reset(self) -> None:
        _capi.check("ddp_ready_reset", _capi.lib().ddp_ready_reset(self._ptr))


def ddp_allreduce_as_ready(rank_grads, bucket_offsets, out, ready: BucketReadiness,
                           timeout_s: float = 10.0, stream=None):
    """Bucket by bucket, in bucket order: wait on the host until every rank
    marked the bucket's gradients, then launch its all-reduce average.  A
    bucket that never fills raises BucketNotReady before anything is launched
    for it (the buckets before it are already reduced)."""
    for b in range(len(bucket_offsets) - 1):
        ready.wait(b, timeout_s)
        ddp_bucket_allreduce_avg(rank_grads, bucket_offsets, out, first=b, count=1,
                                 stream=stream)
    return out


# ---------------------------------------------------------------- ledger

def state_bytes(psi: float, nd: int, stage: int, k: float = 12.0) -> float:
    r = _capi.lib().shardstep_state_bytes(psi, nd, stage, k)
    if r < 0:
        raise ValueError("bad stage or nd")
    return r


def comm_bytes(psi: float, nd: int, kind: str, exact: bool = False) -> float:
    r = _capi.lib().shardstep_comm_bytes(psi, nd, _capi.COMM_KINDS[kind], int(exact))
    if r < 0:
        raise ValueError("bad kind or nd")
    return r


def set_fused_path(path: str) -> str:
    """Which kernels the streaming calls (fused steps, accumulation, bucket
    all-reduce, non-finite check) may use: "auto" (TMA-staged where it
    measured faster and the arguments allow), "register" (register-staged
    only) or "tma" (TMA-staged whenever the arguments allow).  Returns
    the previous setting."""
    codes = {"auto": _capi.PATH_AUTO, "register": _capi.PATH_REGISTER, "tma": _capi.PATH_TMA}
    names = {v: k for k, v in codes.items()}
    prev = _capi.lib().shardstep_set_fused_path(codes[path])
    if prev < 0:
        _capi.check("shardstep_set_fused_path", prev)
    return names[prev]


def set_tma_stages(stages: int) -> int:
    """Shared-memory stages of each TMA-staged launch (0: about 128 KB of
    tiles in flight per SM; else 2..16, limited to what fits).  Tuning only;
    returns the previous setting."""
    prev = _capi.lib().shardstep_set_tma_stages(int(stages))
    if prev < 0:
        _capi.check("shardstep_set_tma_stages", prev)
    return prev


def set_dependent_launch(enable: bool) -> bool:
    """Whether kernels are launched as programmatic dependents of the kernel
    before them in the stream (default True): each call's first kernel
    waits for its predecessor before touching memory (only the launch
    latency overlaps), later buckets / copies of one call overlap the
    previous one's drain.  Results do not depend on it; returns the previous
    setting."""
    return bool(_capi.lib().shardstep_set_dependent_launch(int(bool(enable))))


def device_status(clear: bool = False) -> int:
    """Watchdog bits of the current device (0: no TMA-staged wait ran out)."""
    st = ctypes.c_uint32(0)
    _capi.check("shardstep_device_status",
                _capi.lib().shardstep_device_status(ctypes.byref(st), int(bool(clear))))
    return st.value


def set_tma_wait_ns(ns: int) -> int:
    """How long a TMA-staged kernel's waits for a tile or a free stage may
    last (ns; 0 = the default of about two seconds).  A test control: a wait
    that runs out sets a bit of ``device_status``.  Returns the previous
    limit."""
    prev = _capi.lib().shardstep_set_tma_wait_ns(int(ns))
    if prev < 0:
        _capi.check("shardstep_set_tma_wait_ns", int(prev))
    return int(prev)


def check_mean_division(nd: int, device=None, stream=None):
    """Runs the library's division by N_d and IEEE fp32 division on all 2^32
    fp32 bit patterns on the GPU.  Returns (mismatches, smallest differing
    pattern or None); synchronises the stream."""
    import torch
    dev = torch.device(device) if device is not None else torch.device("cuda")
    count = torch.zeros(1, dtype=torch.int64, device=dev)
    first = torch.full((1,), -1, dtype=torch.int32, device=dev)
    _capi.check("shardstep_check_mean_division", _capi.lib().shardstep_check_mean_division(
        int(nd), ctypes.c_void_p(count.data_ptr()), ctypes.c_void_p(first.data_ptr()),
        _stream(stream, dev)))
    n = int(count.item())
    f = int(first.item()) & 0xFFFFFFFF
    return n, (f if n else None)


def hybrid_state_bytes(psi: float, shard_group: int, k: float = 12.0) -> float:
    r = _capi.lib().shardstep_hybrid_state_bytes(psi, shard_group, k)
    if r < 0:
        raise ValueError("bad sharding factor")
    return r


def hybrid_comm_bytes(psi: float, nd: int, shard_group: int, kind: str,
                      exact: bool = False) -> float:
    code = {"intra": 0, "inter": 1}[kind]
    r = _capi.lib().shardstep_hybrid_comm_bytes(psi, nd, shard_group, code, int(exact))
    if r < 0:
        raise ValueError("the sharding factor must divide N_d")
    return r


def comm_counter(reset: bool = False) -> float:
    """Bytes the emulated collectives of the calls so far would send between
    ranks as rings (``shardstep_comm_counter``); ``reset`` zeroes it after
    reading."""
    return float(_capi.lib().shardstep_comm_counter(int(bool(reset))))


def launch_count() -> int:
    """Kernels libshardstep has launched in this process."""
    return int(_capi.lib().shardstep_launch_count())


def last_kernel() -> str:
    """Name of the kernel this thread's last streaming call launched (fused
    step, accumulation, non-finite check, bucket all-reduce); "" before the
    first."""
    return _capi.lib().shardstep_last_kernel().decode()
