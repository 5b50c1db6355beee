"""Reduce-scatter average, AdamW, bf16 cast and micro-batch accumulation.
TEST INFRASTRUCTURE.

numpy float32 arithmetic: every array operation below is one IEEE operation
rounded to nearest (no fused multiply-add: each ufunc call rounds), and the
operations are written in the order they are applied.  The same functions
run in float64 when given float64 arrays, which the pins use for closed
forms and error bounds.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ----------------------------------------------------------------- bf16

def bf16_to_f32(u16) -> np.ndarray:
    """bf16 bits -> fp32: bf16 is the upper half of an fp32, so the upcast is
    exact (the 16 low bits are zero)."""
    u16 = np.ascontiguousarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """fp32 -> bf16 bits, the nearest bf16 value with ties to the even one.

    Plain definition: the two bf16 values around |x| are the truncation ``lo``
    (low 16 bits cleared) and the next bf16 magnitude ``lo + ulp``; both
    distances are exact in double.  Past the largest finite bf16 the next value
    is 2^128, i.e. overflow to infinity happens at max + ulp/2 as IEEE
    round-to-nearest requires.  NaN maps to a quiet NaN, infinities to
    themselves.  "PyTorch FSDP..." section 3.5 (native mixed precision) has a
    single high-to-low cast; bf16 is the low precision the step's parameters
    and communication use ("Infra: Data Parallel": 16-bit parameters and
    gradients).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    sign = b & np.uint32(0x80000000)
    mag = b & np.uint32(0x7FFFFFFF)
    lo = mag & np.uint32(0xFFFF0000)
    lo_val = lo.view(np.float32).astype(np.float64)
    exp = ((lo >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int32)
    ulp = np.ldexp(np.ones(exp.shape, dtype=np.float64), np.maximum(exp, 1) - 127 - 7)
    hi_val = lo_val + ulp
    with np.errstate(invalid="ignore"):
        xv = mag.view(np.float32).astype(np.float64)
        d_lo = xv - lo_val
        d_hi = hi_val - xv
        odd = ((lo >> np.uint32(16)) & np.uint32(1)) == 1
        up = (d_hi < d_lo) | ((d_hi == d_lo) & odd)
    res = (lo >> np.uint32(16)) + up.astype(np.uint32)
    res = np.where(mag == np.uint32(0x7F800000), np.uint32(0x7F80), res)
    res = np.where(mag > np.uint32(0x7F800000), (mag >> np.uint32(16)) | np.uint32(0x40), res)
    res = res | (sign >> np.uint32(16))
    return res.astype(np.uint16)


def _upcast(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_to_f32(a)
    if a.dtype in (np.float32, np.float64):
        return a
    raise TypeError(a.dtype)


# -------------------------------------------------------- accumulation

def grad_accumulate(micro_grads, scale):
    """Local gradient accumulation over M micro-batches with the loss
    normalised by M ("Infra: Data Parallel", section "Naïve Data Parallelism":
    accumulate locally, sync only on the last micro-batch, divide each
    micro-batch loss by the number of micro-batches).  By linearity of the
    backward pass, dividing the loss by M scales each micro-batch gradient by
    1/M, so acc = sum_j fl(g_j * scale), summed in order j = 0..M-1, the first
    term starting the sum; ``scale`` is the fp32 value of 1/M."""
    if len(micro_grads) == 0:
        raise ValueError("need at least one micro-batch")
    g0 = _upcast(micro_grads[0])
    s = g0.dtype.type(scale)
    acc = g0 * s
    for g in micro_grads[1:]:
        acc = acc + _upcast(g) * s
    return acc


# ------------------------------------------------------ reduce-scatter

def rs_avg(contribs, r: int, shard: int):
    """Reduce-scatter average of rank r's slice.

    ``contribs[q]`` is rank q's full flat gradient (bf16 bits, or the fp32
    accumulator when micro-batches were accumulated).  Rank r keeps
    mean_q contribs[q][r*S : (r+1)*S]: the mean of the N_d local-mean
    gradients, which equals the global-batch gradient ("4.1 数据并行详解",
    section 2, the g-bar identity; averaging, not summing).  The sum is taken
    in fp32 in rank order 0..N_d-1 and divided by N_d ("Infra: Data
    Parallel", ZeRO section: reduce-scatter with averaging hands each rank its
    part of the averaged gradient)."""
    nd = len(contribs)
    if nd < 1:
        raise ValueError("need at least one rank")
    sl = [_upcast(c[r * shard:(r + 1) * shard]) for c in contribs]
    s = sl[0].copy()
    for q in range(1, nd):
        s = s + sl[q]
    return s / s.dtype.type(nd)


# ----------------------------------------------------------------- AdamW

@dataclass
class AdamWConfig:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


@dataclass
class _Scalars:
    lr_wd: object
    beta1: object
    omb1: object
    beta2: object
    omb2: object
    step_size: object
    sqrt_bc2: object
    eps: object


def adamw_scalars(hp: AdamWConfig, t: int, dtype=np.float32) -> _Scalars:
    """Per-step scalars, computed in double and rounded once to ``dtype``:
    lr*wd, beta1, 1-beta1, beta2, 1-beta2, lr/bc1 and sqrt(bc2), with
    bc_i = 1 - beta_i^t and beta_i^t the product of t factors beta_i taken
    left to right in double (t >= 1 is the 1-based step count)."""
    if t < 1:
        raise ValueError("step count starts at 1")
    b1t = 1.0
    b2t = 1.0
    for _ in range(t):
        b1t *= hp.beta1
        b2t *= hp.beta2
    bc1 = 1.0 - b1t
    bc2 = 1.0 - b2t
    f = np.dtype(dtype).type
    return _Scalars(lr_wd=f(hp.lr * hp.weight_decay), beta1=f(hp.beta1), omb1=f(1.0 - hp.beta1),
                    beta2=f(hp.beta2), omb2=f(1.0 - hp.beta2), step_size=f(hp.lr / bc1),
                    sqrt_bc2=f(math.sqrt(bc2)), eps=f(hp.eps))


def adamw(p, m, v, g, hp: AdamWConfig, t: int):
    """Elementwise AdamW on a shard ("Infra: Data Parallel", ZeRO section: AdamW
    updates element by element, so a rank needs only its own parameters,
    averaged gradient and moments; fp32 master weights and both moments are
    the k = 12 bytes of optimizer state per parameter).

    The pages print no update formula.  Reading: decoupled weight decay
    (Loshchilov & Hutter) with Adam's bias correction and eps added outside
    the square root, applied in this order, one rounding per operation:
        p <- p - (lr*wd) * p
        m <- beta1*m + (1-beta1)*g
        v <- beta2*v + ((1-beta2)*g)*g
        p <- p - ((lr/bc1) * m) / (sqrt(v)/sqrt(bc2) + eps)
    Returns new (p, m, v); inputs are not modified."""
    c = adamw_scalars(hp, t, dtype=np.asarray(p).dtype)
    p = p - c.lr_wd * p
    m = c.beta1 * m + c.omb1 * g
    v = c.beta2 * v + (c.omb2 * g) * g
    denom = np.sqrt(v) / c.sqrt_bc2 + c.eps
    p = p - (c.step_size * m) / denom
    return p, m, v


def fsdp_shard_step(contribs, r: int, shard: int, p, m, v, hp: AdamWConfig, t: int):
    """One sharded optimizer step on rank r: reduce-scatter average, AdamW on
    the fp32 shard, then the single cast of the updated shard to bf16 (the
    cast precedes the all-gather, so the gather moves bf16: "PyTorch FSDP..."
    section 3.5, all communication in low precision).
    Returns (p, m, v, p_bf16_bits)."""
    g = rs_avg(contribs, r, shard)
    p, m, v = adamw(p, m, v, g, hp, t)
    return p, m, v, f32_to_bf16(p)


# ------------------------------------------------------- hybrid sharding

def hybrid_rs_avg(contribs, shard_group: int, f: int, shard: int):
    """Hybrid sharding with sharding factor F ("PyTorch FSDP..." section 2,
    sharding factor; section 3.3: full sharding inside groups of F GPUs,
    replication across groups; "4.1 数据并行详解" section 6.3, HYBRID_SHARD).

    The N_d = R x F ranks are ordered k = g*F + j (group g, position j).  A
    unit is split into F shards of S elements and rank (g, f) holds shard f.
    Its gradient is reduce-scattered inside its group, then all-reduced across
    the R groups, then averaged over all N_d ranks:
        s_g   = G_{gF} + G_{gF+1} + ... + G_{gF+F-1}      (in order j)
        total = s_0 + s_1 + ... + s_{R-1}                  (in order g)
        mean  = total / N_d
    on elements [f*S, (f+1)*S) of each rank's flat gradient, in fp32.
    F = N_d is rs_avg; F = 1 is the plain all-reduce average."""
    nd = len(contribs)
    if shard_group < 1 or nd % shard_group != 0:
        raise ValueError("the sharding factor must divide N_d")
    R = nd // shard_group
    sl = [_upcast(c[f * shard:(f + 1) * shard]) for c in contribs]
    total = None
    for g in range(R):
        s = sl[g * shard_group].copy()
        for j in range(1, shard_group):
            s = s + sl[g * shard_group + j]
        total = s if total is None else total + s
    return total / total.dtype.type(nd)


def hybrid_shard_step(contribs, shard_group: int, f: int, shard: int, p, m, v,
                      hp: AdamWConfig, t: int):
    """One hybrid-sharded step on shard f (identical on each of the R groups
    that replicate it): hybrid reduce, AdamW, bf16 cast.
    Returns (p, m, v, p_bf16_bits)."""
    g = hybrid_rs_avg(contribs, shard_group, f, shard)
    p, m, v = adamw(p, m, v, g, hp, t)
    return p, m, v, f32_to_bf16(p)
