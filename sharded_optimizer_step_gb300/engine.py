"""One rank's sharded optimizer over a model's FSDP units.

The rank keeps its shard of every unit back to back in one buffer per state
(fp32 master, m, v and the bf16 parameter shard), so one fused launch updates
the whole rank.  The N_d incoming gradient contributions (the reduce-scatter
inputs: rank q's flat gradient, restricted to this rank's slices) are the
buffers ``grad_in[q]`` laid out the same way, which the caller fills between
steps.  ``gather_unit`` all-gathers one unit's bf16 shards into its full flat
buffer and returns the per-tensor views.

Buffers are allocated with torch once, at construction; ``step`` and
``gather_unit`` allocate nothing.
"""
from __future__ import annotations

import torch

from . import (AdamW, AdamWState, Fsdp2Step, fsdp2_all_gather_copy_out, fsdp2_layout,
               fsdp2_local_views, fsdp_accumulate_rs_avg_adamw_cast, fsdp_ag_unpack,
               fsdp_hybrid_rs_avg_adamw_cast, fsdp_layout, fsdp_rs_avg_adamw_cast,
               fsdp_shard_pieces,
               fsdp_state_accumulate_rs_avg_adamw_cast, fsdp_state_rs_avg_adamw_cast,
               fsdp_views)


def _numel(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n


class RankShardOptimizer:
    def __init__(self, unit_shapes, nd: int, rank: int, hp: AdamW, device="cuda",
                 grad_dtype=torch.bfloat16, shard_group: int = 0):
        """``shard_group`` = F enables hybrid sharding: units are split into F
        shards, ``rank`` is the shard index 0..F-1 inside the rank's group,
        and the N_d contributions come in rank order k = g*F + j."""
        self.F = shard_group or nd
        if nd % self.F != 0:
            raise ValueError("the sharding factor must divide N_d")
        if not 0 <= rank < self.F:
            raise ValueError("rank out of range")
        self.unit_shapes = [list(u) for u in unit_shapes]
        self.nd, self.rank, self.hp = nd, rank, hp
        self.layouts = [fsdp_layout([_numel(s) for s in u], self.F) for u in self.unit_shapes]
        self.starts = []
        pos = 0
        for lay in self.layouts:
            self.starts.append(pos)
            pos += lay.shard
        self.shard_total = pos
        dev = torch.device(device)
        self.master = torch.zeros(pos, dtype=torch.float32, device=dev)
        self.m = torch.zeros(pos, dtype=torch.float32, device=dev)
        self.v = torch.zeros(pos, dtype=torch.float32, device=dev)
        self.params = torch.zeros(pos, dtype=torch.bfloat16, device=dev)
        self.grad_in = [torch.zeros(pos, dtype=grad_dtype, device=dev) for _ in range(nd)]
        self.t = 0
        self.state = None                 # the device step state, once made

    def _next_host_step(self):
        """Advance the count for a host-scalar step.  When the count is also
        kept on the device (``device_step_state``), the device count is the
        current one (reading it synchronises) and the device state moves to
        the new count too, so the two forms of step can be mixed."""
        if self.state is not None:
            self.t = self.state.step()
        self.t += 1
        if self.state is not None:
            self.state.init(self.t)

    def unit_slice(self, buf, u):
        """This rank's piece of unit u inside a rank-shard buffer."""
        return buf[self.starts[u]:self.starts[u] + self.layouts[u].shard]

    def rank_pieces(self):
        """Where each original tensor's piece sits in this rank's buffers:
        a list of (unit, tensor, position in the rank buffer, first element
        within the tensor, length), one entry per piece the rank holds (the
        library's FlatParameter layout).  Positions not covered are the
        units' padding."""
        out = []
        for u, shapes in enumerate(self.unit_shapes):
            pieces = fsdp_shard_pieces([_numel(s) for s in shapes], self.F, self.rank)
            for t, (pos, tpos, cnt) in enumerate(pieces):
                if cnt:
                    out.append((u, t, self.starts[u] + pos, tpos, cnt))
        return out

    def step(self, stream=None):
        """Reduce-scatter average + AdamW + bf16 cast over the whole rank shard
        (one launch)."""
        self._next_host_step()
        self._update(self.grad_in, self.master, self.m, self.v, self.params, stream)

    def _update(self, grads, master, m, v, params, stream):
        if self.F == self.nd:
            fsdp_rs_avg_adamw_cast(grads, master, m, v, params, self.hp, self.t, stream=stream)
        else:
            fsdp_hybrid_rs_avg_adamw_cast(grads, self.F, master, m, v, params, self.hp, self.t,
                                          stream=stream)

    def step_with_last_micro_batch(self, last, scale: float, stream=None):
        """The step of ``step`` where ``grad_in`` holds fp32 accumulators of
        micro-batches 0..M-2 and ``last[q]`` is contribution q's bf16
        gradient of the last micro-batch (laid out like ``grad_in[q]``):
        the last accumulation (``scale`` = 1/M) runs inside the fused launch
        and ``grad_in`` is left as it was."""
        self._next_host_step()
        fsdp_accumulate_rs_avg_adamw_cast(self.grad_in, last, scale, self.master, self.m, self.v,
                                          self.params, self.hp, self.t, shard_group=self.F,
                                          stream=stream)

    def begin_step(self):
        """Advance the step count for an update issued piece by piece with
        ``update_range`` (e.g. overlapped with the arrival of the gradients)."""
        self._next_host_step()

    def update_range(self, a: int, b: int, stream=None):
        """The fused update of shard positions [a, b) at the current step count."""
        sl = slice(a, b)
        self._update([g[sl] for g in self.grad_in], self.master[sl], self.m[sl], self.v[sl],
                     self.params[sl], stream)

    def device_step_state(self) -> AdamWState:
        """Moves the step count to the device (an ``AdamWState`` at the
        current count) for ``step_on_device``; returns it."""
        self.state = AdamWState(self.hp, self.t, device=self.master.device)
        return self.state

    def step_on_device(self, stream=None):
        """The step of ``step`` with the count advanced and the AdamW scalars
        derived on the device: the same launches every call, so it can be
        captured in a CUDA graph.  Needs ``device_step_state`` first; the
        host count ``t`` is not advanced."""
        self.state.advance(stream=stream)
        fsdp_state_rs_avg_adamw_cast(self.grad_in, self.master, self.m, self.v, self.params,
                                     self.state, shard_group=self.F, stream=stream)

    def step_with_last_micro_batch_on_device(self, last, scale: float, stream=None):
        """``step_with_last_micro_batch`` with the count advanced and the AdamW
        scalars derived on the device (see ``step_on_device``): capturable in
        a CUDA graph together with the accumulate launches.  Needs
        ``device_step_state`` first."""
        self.state.advance(stream=stream)
        fsdp_state_accumulate_rs_avg_adamw_cast(self.grad_in, last, scale, self.master, self.m,
                                                self.v, self.params, self.state,
                                                shard_group=self.F, stream=stream)

    def gather_unit(self, u, peer_shards, full, stream=None):
        """All-gather unit u inside the rank's shard group: ``peer_shards[q]``
        is shard q's bf16 piece (q < F; this rank's own entry is ignored and
        taken from ``params``); ``full`` is the unit's flat bf16 buffer of P
        elements.  Returns the tensor views."""
        shards = list(peer_shards)
        shards[self.rank] = self.unit_slice(self.params, u)
        fsdp_ag_unpack(shards, full, stream=stream)
        return fsdp_views(full, self.unit_shapes[u], self.F)


class Fsdp2RankOptimizer:
    """One rank's optimizer over an FSDP2 group (per-parameter Shard(0)): the
    rank's padded local buffers -- fp32 master, m, v and the bf16 parameter
    rows, ``local`` elements laid out as fsdp2_layout gives -- and the step
    read straight from every rank's per-parameter gradients (``Fsdp2Step``,
    no chunk-cat copy).  ``rank_grads[q][t]`` is rank q's gradient of
    parameter t (global shape), kept and checked once.  ``gather`` copies the
    ranks' bf16 rows out into the full parameters; ``local_views`` are the
    rank's DTensor.to_local() views of a local buffer."""

    def __init__(self, rank_grads, rank: int, hp: AdamW, device="cuda"):
        self._step = Fsdp2Step(rank_grads)
        self.nd, self.rank, self.hp = self._step.nd, rank, hp
        if not 0 <= rank < self.nd:
            raise ValueError("rank out of range")
        self.shapes = self._step.shapes
        self.layout = fsdp2_layout(self.shapes, self.nd)
        L = self._step.local
        dev = torch.device(device)
        self.master = torch.zeros(L, dtype=torch.float32, device=dev)
        self.m = torch.zeros(L, dtype=torch.float32, device=dev)
        self.v = torch.zeros(L, dtype=torch.float32, device=dev)
        self.params = torch.zeros(L, dtype=torch.bfloat16, device=dev)
        self.t = 0
        self.state = None                 # the device step state, once made

    def local_views(self, buf):
        """The rank's rows of every parameter inside ``buf`` (one of its local
        buffers), shaped (rows, trailing dims)."""
        return fsdp2_local_views(buf, self.shapes, self.nd, self.rank)

    def step(self, stream=None):
        """The rank's step with host scalars (the count advanced on the host;
        with a device step state, from and into the device count)."""
        if self.state is not None:
            self.t = self.state.step()
        self.t += 1
        if self.state is not None:
            self.state.init(self.t)
        self._step(self.rank, self.master, self.m, self.v, self.params, self.hp, self.t,
                   stream=stream)

    def device_step_state(self) -> AdamWState:
        """Moves the step count to the device for ``step_on_device``."""
        self.state = AdamWState(self.hp, self.t, device=self.master.device)
        return self.state

    def step_on_device(self, stream=None):
        """The count advanced and the AdamW scalars derived on the device: the
        same launches every call, so a CUDA graph can capture it."""
        self.state.advance(stream=stream)
        self._step.step_state(self.rank, self.master, self.m, self.v, self.params, self.state,
                              stream=stream)

    def gather(self, peer_params, params, stream=None):
        """All-gather: ``peer_params[q]`` is rank q's bf16 local buffer (this
        rank's own entry is ignored and taken from ``params`` of this
        optimizer); ``params`` are the full parameter tensors (global shapes)
        written in place."""
        bufs = list(peer_params)
        bufs[self.rank] = self.params
        fsdp2_all_gather_copy_out(bufs, params, stream=stream)
        return params
