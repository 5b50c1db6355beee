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
