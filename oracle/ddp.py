"""DDP bucketing and bucketed all-reduce average.  TEST INFRASTRUCTURE.

"4.1 数据并行详解", section 4.2 (bucket mechanism): gradients are grouped into
buckets in the order backward produces them (last layer first), about 25 MB
each by default (bucket_cap_mb), and a bucket's all-reduce starts as soon as
all of its gradients are ready.  "Infra: Data Parallel", section "Naïve Data
Parallelism": every rank averages the full gradients with all-reduce and
then runs the same update.
"""
from __future__ import annotations

import numpy as np

from .numerics import AdamWConfig, adamw, bf16_to_f32, f32_to_bf16

MiB = 1 << 20


def bucket_plan(numels, elem_size: int, cap_bytes: int):
    """Greedy buckets over the parameters in reverse registration order.

    Reading of the pages' rule (they give only the order and the ~25 MB cap):
    a bucket is closed before a parameter that would take it past the cap, a
    parameter larger than the cap gets a bucket of its own, parameters are
    never split and zero-size parameters join the open bucket.

    Returns (param_offset, bucket_of_param, bucket_offsets): the element offset
    of each parameter in the bucketed flat buffer (buckets back to back, each
    bucket holding its parameters in the order they were added), the bucket of
    each parameter, and the element offsets of the buckets (length
    n_buckets + 1)."""
    n = len(numels)
    if cap_bytes <= 0 or elem_size <= 0:
        raise ValueError("cap and element size must be positive")
    buckets = []
    cur, cur_bytes = [], 0
    for i in reversed(range(n)):
        b = int(numels[i]) * elem_size
        if cur and cur_bytes + b > cap_bytes:
            buckets.append(cur)
            cur, cur_bytes = [], 0
        cur.append(i)
        cur_bytes += b
    if cur:
        buckets.append(cur)
    param_offset = [0] * n
    bucket_of = [0] * n
    offsets = [0]
    pos = 0
    for k, bucket in enumerate(buckets):
        for i in bucket:
            param_offset[i] = pos
            bucket_of[i] = k
            pos += int(numels[i])
        offsets.append(pos)
    return param_offset, bucket_of, offsets


def bucket_allreduce_avg(rank_grads, bucket_offsets):
    """Per bucket b, out[a:e] = bf16((sum_q G_q[a:e]) / N_d) with the fp32 sum in
    rank order 0..N_d-1.  The all-reduce keeps the gradient's dtype, so the
    averaged gradient is rounded to bf16 once."""
    nd = len(rank_grads)
    total = bucket_offsets[-1] if bucket_offsets else 0
    out = np.zeros(total, dtype=np.uint16)
    for a, e in zip(bucket_offsets[:-1], bucket_offsets[1:]):
        s = bf16_to_f32(rank_grads[0][a:e]).copy()
        for q in range(1, nd):
            s = s + bf16_to_f32(rank_grads[q][a:e])
        out[a:e] = f32_to_bf16(s / np.float32(nd))
    return out


def ddp_step(rank_grads, bucket_offsets, p, m, v, hp: AdamWConfig, t: int):
    """Replicated step: bucketed all-reduce average, then the full (unsharded)
    AdamW on every parameter with the averaged bf16 gradient upcast to fp32,
    then the bf16 cast of the parameters.  Returns (avg_bf16, p, m, v, p_bf16)."""
    avg = bucket_allreduce_avg(rank_grads, bucket_offsets)
    p, m, v = adamw(p, m, v, bf16_to_f32(avg), hp, t)
    return avg, p, m, v, f32_to_bf16(p)
