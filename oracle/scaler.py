"""Sharded gradient scaler for fp16 loss scaling.  TEST INFRASTRUCTURE.

"PyTorch FSDP..." section 3.5: for the gradient overflow of fp16 mixed
precision, FSDP has a sharded gradient scaler adapted to parameter sharding
that keeps gradient scaling mathematically equivalent.  The page gives no
mechanism.  Reading (the plain one, which the dynamic loss scaling it refers
to defines): the loss is multiplied by a scale s before backward, so the fp16
gradients arrive multiplied by s; after the reduce-scatter each rank
multiplies its averaged shard gradient by 1/s and checks it for inf / NaN;
the found-inf flags are OR-ed across all ranks (an all-reduce); if any rank
found one, every rank skips the update (parameters and moments unchanged) and
the scale is multiplied by the backoff factor, otherwise the update runs on
the unscaled gradient and, after growth_interval consecutive clean steps, the
scale is multiplied by the growth factor.
"""
from __future__ import annotations

import numpy as np

from .numerics import AdamWConfig, _upcast, adamw, f32_to_bf16, hybrid_rs_avg


def f16_to_f32(u16) -> np.ndarray:
    """fp16 bits -> fp32 (exact: every fp16 value is an fp32 value)."""
    return np.ascontiguousarray(u16, dtype=np.uint16).view(np.float16).astype(np.float32)


def _as_f32_contribs(contribs):
    """fp16 contributions are passed as (bits, "f16") pairs; bf16 as uint16
    arrays; fp32 as float32 arrays."""
    out = []
    for c in contribs:
        if isinstance(c, tuple):
            out.append(f16_to_f32(c[0]))
        else:
            out.append(_upcast(c))
    return out


def unscaled_mean(contribs, shard_group: int, f: int, shard: int, inv_scale):
    """Reduced (hybrid order; shard_group = N_d is the plain rank order)
    mean of the N_d contributions to shard f, multiplied by 1/s in fp32."""
    with np.errstate(over="ignore", invalid="ignore"):
        g = hybrid_rs_avg(_as_f32_contribs(contribs), shard_group, f, shard)
        return g * np.float32(inv_scale)


def found_inf(contribs, shard_group: int, f: int, shard: int, inv_scale) -> bool:
    """True when any unscaled mean gradient of shard f is inf or NaN."""
    return not bool(np.all(np.isfinite(unscaled_mean(contribs, shard_group, f, shard,
                                                     inv_scale))))


def scaled_shard_step(contribs, shard_group: int, f: int, shard: int, p, m, v, out_prev,
                      hp: AdamWConfig, t: int, inv_scale, skip: bool):
    """The update of shard f under the scaler: unchanged state (and bf16
    output) when ``skip`` (a rank anywhere found inf/NaN), else AdamW on the
    unscaled mean and the bf16 cast.  Returns (p, m, v, out)."""
    if skip:
        return p, m, v, out_prev
    g = unscaled_mean(contribs, shard_group, f, shard, inv_scale)
    p, m, v = adamw(p, m, v, g, hp, t)
    return p, m, v, f32_to_bf16(p)


def scaler_update(scale: float, tracker: int, found: bool, growth_factor: float,
                  backoff_factor: float, growth_interval: int):
    """Next (scale, growth tracker), in fp32 scale arithmetic: a step with
    inf/NaN multiplies the scale by the backoff factor and resets the
    tracker; a clean step counts, and the growth_interval-th clean step in a
    row multiplies the scale by the growth factor (kept only if the product
    is finite) and resets the tracker."""
    scale = np.float32(scale)
    with np.errstate(over="ignore"):
        return _update(scale, tracker, found, growth_factor, backoff_factor, growth_interval)


def _update(scale, tracker, found, growth_factor, backoff_factor, growth_interval):
    if found:
        return np.float32(scale * np.float32(backoff_factor)), 0
    tracker += 1
    if tracker == growth_interval:
        grown = np.float32(scale * np.float32(growth_factor))
        if np.isfinite(grown):
            scale = grown
        tracker = 0
    return scale, tracker
