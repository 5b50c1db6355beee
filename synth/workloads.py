"""Synthetic workloads: model-shaped FSDP units and the seeded streams their
inputs come from.  Shapes only -- no weights, no data set.

Each workload is a list of FSDP units (one FlatParameter each), the number of
emulated data-parallel ranks N_d, micro-batches M and optimizer steps.  The
inputs are:
  * rank q's micro-batch j gradient of unit u at step t: bf16, approximately
    N(0, grad_sigma), optionally with a fraction of elements scaled x100,
    element index = position in the unit's flat (padded) buffer;
  * the fp32 master weights of unit u: approximately N(0, master_sigma);
  * moments start at zero.
Padding positions (past the unit's last tensor) are zero in every input.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import KIND_GRAD, KIND_MASTER, KIND_SHARD_BF16, normal_stream


@dataclass
class Workload:
    name: str
    cfg_id: int
    units: list                     # per unit: list of tensor shapes (tuples)
    nd: int
    micro: int = 1
    steps: int = 1
    grad_sigma: float = 1e-3
    master_sigma: float = 0.02
    outlier_p: float = 0.0
    outlier_scale: float = 100.0
    seed: int = 0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    shard_group: int = 0            # hybrid sharding factor F (0: F = nd, full sharding)
    extra: dict = field(default_factory=dict)

    @property
    def F(self):
        return self.shard_group or self.nd

    def unit_numels(self, u):
        out = []
        for s in self.units[u]:
            n = 1
            for d in s:
                n *= int(d)
            out.append(n)
        return out

    def unit_total(self, u):
        return sum(self.unit_numels(u))

    def unit_padded(self, u):
        T = self.unit_total(u)
        return -(-T // self.F) * self.F

    def unit_shard(self, u):
        return self.unit_padded(u) // self.F

    @property
    def psi(self):
        return sum(self.unit_total(u) for u in range(len(self.units)))

    # ---------------------------------------------------------- streams
    def grad_stream(self, step: int, rank: int, micro: int, unit: int):
        return normal_stream(self.seed, (self.cfg_id, KIND_GRAD, step, rank, micro, unit),
                             self.grad_sigma, self.outlier_p, self.outlier_scale)

    def master_stream(self, unit: int):
        return normal_stream(self.seed, (self.cfg_id, KIND_MASTER, 0, 0, 0, unit),
                             self.master_sigma)

    def peer_shard_stream(self, step: int, rank: int, unit: int):
        """bf16 parameter shard of another rank, for the all-gather input."""
        return normal_stream(self.seed, (self.cfg_id, KIND_SHARD_BF16, step, rank, 0, unit),
                             self.master_sigma)


def _llama_layer(h, ffn):
    return [(h, h)] * 4 + [(ffn, h), (ffn, h), (h, ffn), (h,), (h,)]


def unit_9m() -> Workload:
    """One unit of (1024,1024), (1024,4096), (4096,1024), N_d = 4, M = 4."""
    return Workload("unit_9m_nd4_m4", 1, [[(1024, 1024), (1024, 4096), (4096, 1024)]], nd=4,
                    micro=4, steps=1)


def gpt2_small() -> Workload:
    """GPT-2 small shape: 12 block units (qkv, proj, fc, proj with biases and
    two LayerNorms) and one embedding unit (wte, wpe, ln_f; tied head)."""
    h, f, v, ctx = 768, 3072, 50257, 1024
    block = [(h, 3 * h), (3 * h,), (h, h), (h,), (h, f), (f,), (f, h), (h,), (h,), (h,), (h,), (h,)]
    units = [list(block) for _ in range(12)] + [[(v, h), (ctx, h), (h,), (h,)]]
    return Workload("gpt2_small_nd8", 2, units, nd=8, micro=1, steps=10)


def llama_1b() -> Workload:
    """Llama-style 1B: 16 layer units (hidden 2048, SwiGLU ffn 8192, two
    RMSNorm vectors) and an embedding unit (embedding, untied head, final
    norm); 1% of gradient elements are x100 outliers."""
    h, f, v = 2048, 8192, 32000
    units = [_llama_layer(h, f) for _ in range(16)] + [[(v, h), (v, h), (h,)]]
    return Workload("llama_1b_nd8_m4", 3, units, nd=8, micro=4, steps=10, outlier_p=0.01)


def llama_7b_rank_view() -> Workload:
    """Llama-style 7B (hidden 4096, ffn 11008, vocab 32000): 32 layer units and
    an embedding unit; one rank's view, i.e. its shard of every unit, with
    the 8 ranks' gradient contributions.  The all-gather input is one layer
    unit (202,383,360 parameters)."""
    h, f, v = 4096, 11008, 32000
    units = [_llama_layer(h, f) for _ in range(32)] + [[(v, h), (v, h), (h,)]]
    return Workload("llama_7b_rank0_nd8", 4, units, nd=8, micro=1, steps=5,
                    extra={"rank": 0, "ag_unit": 0})


def llama_7b_hybrid_view() -> Workload:
    """Hybrid sharding of the Llama-style 7B model: N_d = 16 ranks in 2 groups
    of F = 8 (sharded inside a group, replicated across the two); one rank's
    view, i.e. its shard f = 0 of every unit and the 16 ranks' gradient
    contributions to it."""
    h, f, v = 4096, 11008, 32000
    units = [_llama_layer(h, f) for _ in range(32)] + [[(v, h), (v, h), (h,)]]
    return Workload("llama_7b_hybrid_nd16_f8_rank0", 6, units, nd=16, micro=1, steps=5,
                    shard_group=8, extra={"rank": 0, "ag_unit": 0})


def ddp_sweep() -> Workload:
    """Replicated DDP bucketing: 16 x [768, 768, (768,3072), (768,3072),
    (4096,4096)] + 3 x (768,3072), bf16 gradients, N_d = 8, bucket caps of 1,
    4, 25, 64 and 256 MiB in reverse order, then full AdamW."""
    unit = [(768,), (768,), (768, 3072), (768, 3072), (4096, 4096)]
    params = unit * 16 + [(768, 3072)] * 3
    return Workload("ddp_sweep_nd8", 5, [params], nd=8, micro=1, steps=1,
                    extra={"caps_mib": [1, 4, 25, 64, 256]})


ALL = {w().name: w for w in (unit_9m, gpt2_small, llama_1b, llama_7b_rank_view,
                               llama_7b_hybrid_view, ddp_sweep)}


# ------------------------------------------------- one rank's shard of all units
# A rank keeps its shard of every unit back to back: shard index i of the
# rank's concatenated shard belongs to unit u at local position i - start_u,
# which is element r*S_u + (i - start_u) of that unit's flat buffer (r is the
# shard index: the rank itself under full sharding, its position in the group
# under hybrid sharding).

def rank_shard_index(w: Workload):
    """[(unit, start in the rank's concatenated shard, S_u)] and the total."""
    out, pos = [], 0
    for u in range(len(w.units)):
        s = w.unit_shard(u)
        out.append((u, pos, s))
        pos += s
    return out, pos


def _split_by_unit(w: Workload, idx):
    import numpy as np
    parts, total = rank_shard_index(w)
    idx = np.asarray(idx, dtype=np.int64)
    for u, start, s in parts:
        sel = np.nonzero((idx >= start) & (idx < start + s))[0]
        if sel.size:
            yield u, sel, idx[sel] - start


def host_gather_rank_grad(w: Workload, step: int, rank: int, q: int, micro: int, idx, dtype="bf16"):
    """Rank q's gradient at positions idx of rank `rank`'s concatenated shard
    (zero on padding)."""
    import numpy as np
    from . import host_gather
    out = np.zeros(len(idx), dtype=np.uint16 if dtype == "bf16" else np.float32)
    for u, sel, local in _split_by_unit(w, idx):
        flat = rank * w.unit_shard(u) + local
        vals = host_gather(w.grad_stream(step, q, micro, u), flat, dtype)
        vals[flat >= w.unit_total(u)] = 0
        out[sel] = vals
    return out


def host_gather_rank_master(w: Workload, rank: int, idx):
    import numpy as np
    from . import host_gather
    out = np.zeros(len(idx), dtype=np.float32)
    for u, sel, local in _split_by_unit(w, idx):
        flat = rank * w.unit_shard(u) + local
        vals = host_gather(w.master_stream(u), flat, "f32")
        vals[flat >= w.unit_total(u)] = 0
        out[sel] = vals
    return out


def dev_fill_rank_grad(w: Workload, step: int, rank: int, q: int, micro: int, buf) -> None:
    """Fill a CUDA bf16 tensor holding rank q's contribution to rank `rank`'s
    concatenated shard (zero on padding)."""
    from . import dev_fill
    parts, total = rank_shard_index(w)
    assert buf.numel() == total
    for u, start, s in parts:
        seg = buf[start:start + s]
        dev_fill(w.grad_stream(step, q, micro, u), seg, rank * s)
        T = w.unit_total(u)
        if (rank + 1) * s > T:
            seg[max(0, T - rank * s):].zero_()


def dev_fill_rank_master(w: Workload, rank: int, buf) -> None:
    from . import dev_fill
    parts, total = rank_shard_index(w)
    assert buf.numel() == total
    for u, start, s in parts:
        seg = buf[start:start + s]
        dev_fill(w.master_stream(u), seg, rank * s)
        T = w.unit_total(u)
        if (rank + 1) * s > T:
            seg[max(0, T - rank * s):].zero_()
