"""Synthetic workloads: model-shaped FSDP units and the seeded streams their
inputs come from.  Shapes only -- no weights, no data set.

Each workload is a list of FSDP units (one FlatParameter each) given as the
shapes of their tensors, the number of emulated data-parallel ranks N_d,
micro-batches M and optimizer steps.  Every input value is addressed by the
tensor it belongs to and its row-major index within that tensor:
  * rank q's micro-batch j gradient of tensor t of unit u at step t_s: bf16,
    approximately N(0, grad_sigma), optionally with a fraction of elements
    scaled x100;
  * the fp32 master weights of tensor t of unit u: approximately
    N(0, master_sigma);
  * moments start at zero.
Where an element sits in a FlatParameter, a shard or a rank's buffer (and
the zero padding) is the business of the layout -- the library's on the GPU
side, the oracle's on the CPU side -- never of this module.
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

    @property
    def psi(self):
        return sum(sum(self.unit_numels(u)) for u in range(len(self.units)))

    # ---------------------------------------------------------- streams
    def grad_stream(self, step: int, rank: int, micro: int, unit: int, tensor: int):
        return normal_stream(self.seed, (self.cfg_id, KIND_GRAD, step, rank, micro, unit, tensor),
                             self.grad_sigma, self.outlier_p, self.outlier_scale)

    def master_stream(self, unit: int, tensor: int):
        return normal_stream(self.seed, (self.cfg_id, KIND_MASTER, 0, 0, 0, unit, tensor),
                             self.master_sigma)

    def peer_shard_stream(self, step: int, rank: int, unit: int):
        """bf16 parameter shard of another rank (a flat buffer of the shard's
        length), for the all-gather input."""
        return normal_stream(self.seed, (self.cfg_id, KIND_SHARD_BF16, step, rank, 0, unit),
                             self.master_sigma)


def _llama_layer(h, ffn):
    return [(h, h)] * 4 + [(ffn, h), (ffn, h), (h, ffn), (h,), (h,)]


def _gpt2_units():
    h, f, v, ctx = 768, 3072, 50257, 1024
    block = [(h, 3 * h), (3 * h,), (h, h), (h,), (h, f), (f,), (f, h), (h,), (h,), (h,), (h,), (h,)]
    return [list(block) for _ in range(12)] + [[(v, h), (ctx, h), (h,), (h,)]]


def unit_9m() -> Workload:
    """One unit of (1024,1024), (1024,4096), (4096,1024), N_d = 4, M = 4."""
    return Workload("unit_9m_nd4_m4", 1, [[(1024, 1024), (1024, 4096), (4096, 1024)]], nd=4,
                    micro=4, steps=1)


def gpt2_small() -> Workload:
    """GPT-2 small shape: 12 block units (qkv, proj, fc, proj with biases and
    two LayerNorms) and one embedding unit (wte, wpe, ln_f; tied head)."""
    return Workload("gpt2_small_nd8", 2, _gpt2_units(), nd=8, micro=1, steps=10)


def gpt2_small_nd7() -> Workload:
    """The GPT-2 small units over N_d = 7 ranks: every unit's length is not a
    multiple of 7 (blocks of 7,087,872 elements, embedding unit of
    39,385,344), so every unit carries padding."""
    return Workload("gpt2_small_nd7", 7, _gpt2_units(), nd=7, micro=1, steps=3)


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


ALL = {w().name: w for w in (unit_9m, gpt2_small, gpt2_small_nd7, llama_1b, llama_7b_rank_view,
                               llama_7b_hybrid_view, ddp_sweep)}
