"""Per-GPU model-state memory and communication volume.  TEST INFRASTRUCTURE.

Memory: "Infra: Data Parallel", ZeRO figure ("ZeRO：从复制模型状态到逐步分片"),
per-GPU model-state bytes with 16-bit parameters and gradients and k bytes of
optimizer state per parameter:
    baseline  2Ψ + 2Ψ + kΨ
    ZeRO-1    2Ψ + 2Ψ + kΨ/N_d
    ZeRO-2    2Ψ + (2Ψ + kΨ)/N_d
    ZeRO-3    (2Ψ + 2Ψ + kΨ)/N_d
"4.1 数据并行详解" section 7 prints the same ledger (k = 12) with ~112, ~26 and
~14 GB for Ψ = 7e9, N = 8.

Communication ("Infra: Data Parallel", ZeRO section): per GPU, 16-bit
elements, ring model, the (N_d-1)/N_d factor dropped unless ``exact``:
reduce-scatter or all-gather of the whole model ~2Ψ bytes, all-reduce ~4Ψ;
naive DP 4Ψ, ZeRO-1 and ZeRO-2 4Ψ, ZeRO-3 6Ψ.  "4.1 数据并行详解" sections 5
and 8 count elements instead: ring all-reduce 2Ψ(N-1)/N, FSDP 3Ψ, and the
centralised reduce 2(N-1)Ψ at the root.
"""
from __future__ import annotations

GB = 1e9  # "4.1 数据并行详解" section 4.3: 16 x 7e9 bytes is "about 112 GB"


def state_bytes_per_gpu(psi: float, nd: int, stage: int, k: float = 12.0) -> float:
    """Model-state bytes per GPU for ZeRO stage 0 (replicated), 1, 2 or 3."""
    if stage == 0:
        return 2 * psi + 2 * psi + k * psi
    if stage == 1:
        return 2 * psi + 2 * psi + k * psi / nd
    if stage == 2:
        return 2 * psi + (2 * psi + k * psi) / nd
    if stage == 3:
        return (2 * psi + 2 * psi + k * psi) / nd
    raise ValueError("stage must be 0..3")


def comm_bytes_per_gpu(psi: float, nd: int, kind: str, exact: bool = False) -> float:
    """Bytes sent per GPU for one pass of ``kind`` over a model of psi 16-bit
    elements.  kinds: reduce_scatter, all_gather, all_reduce, ddp, zero1,
    zero2, zero3, centralised_root."""
    f = (nd - 1) / nd if exact else 1.0
    one = 2 * psi * f  # one reduce-scatter or all-gather of every element
    table = {
        "reduce_scatter": one,
        "all_gather": one,
        "all_reduce": 2 * one,
        "ddp": 2 * one,
        "zero1": one + one,
        "zero2": one + one,
        "zero3": one + one + one,
        "centralised_root": 2 * (nd - 1) * 2 * psi,
    }
    if kind not in table:
        raise ValueError(kind)
    return table[kind]


def hybrid_state_bytes_per_gpu(psi: float, shard_group: int, k: float = 12.0) -> float:
    """Hybrid sharding ("PyTorch FSDP..." section 3.3): full sharding inside a
    group of F GPUs, so the ZeRO-3 ledger with N_d replaced by F."""
    return (2 * psi + 2 * psi + k * psi) / shard_group


def hybrid_comm_bytes_per_gpu(psi: float, nd: int, shard_group: int, kind: str,
                              exact: bool = False) -> float:
    """Bytes sent per GPU per step under hybrid sharding, ring model, 16-bit
    elements.  "intra": the gradient reduce-scatter and the parameter
    all-gather inside the group of F (2 x 2Psi, factor (F-1)/F);
    "inter": the all-reduce of the GPU's Psi/F shard across the R = N_d/F
    groups (4 Psi/F, factor (R-1)/R).  This is the ZeRO-1/2 volume of the
    "Infra: Data Parallel" ZeRO section applied to the two levels."""
    if shard_group < 1 or nd % shard_group != 0:
        raise ValueError("the sharding factor must divide N_d")
    R = nd // shard_group
    if kind == "intra":
        f = (shard_group - 1) / shard_group if exact else 1.0
        return 2 * (2 * psi * f) if shard_group > 1 else 0.0
    if kind == "inter":
        f = (R - 1) / R if exact else 1.0
        return 4 * (psi / shard_group) * f if R > 1 else 0.0
    raise ValueError(kind)
