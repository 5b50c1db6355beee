"""CPU oracle for the sharded optimizer step.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check in ``__graft_entry__`` and the benchmark's CPU
baseline / reference arm may import or run anything in this package.  The
CUDA library never does, and the two share no code: the oracle is plain numpy
written from the pages' definitions, in the order the pages (or, where they
are silent, the readings listed below) fix, with no blocking, fusion or
reordering.

Sources (titles of the three pages the method is taken from):
  * "Infra: Data Parallel" (pufanyi.com blog) -- ZeRO stages, memory figure,
    FlatParameter worked example, use_orig_params views, loss/num_micro rule.
  * "PyTorch FSDP: 大模型分布式训练的工业级分片并行方案" (2048ai.net summary of
    Zhao et al. 2023) -- FlatParameter, sharded execution, native mixed
    precision.
  * "4.1 数据并行详解" (AIInfraGuide) -- gradient-mean identity (section 2),
    DDP buckets (4.2), AllReduce = ReduceScatter + AllGather (5.1), memory
    ledger (section 7), communication (section 8).

Readings taken where the pages are silent (each is repeated where it is used):
  * AdamW: decoupled weight decay with Adam bias correction, eps outside the
    square root; fp32 state, one IEEE rounding per operation, in the order
    written in ``numerics.adamw``.
  * Reduce: fp32 sum of the upcast rank slices in rank order 0..N_d-1, then
    divide by N_d; the mean is never rounded to bf16 before the update.
  * Cast: one fp32 -> bf16 round-to-nearest-even of the updated shard, before
    the all-gather, so the gather moves bf16.
  * Padding: zeros at the tail of the unit only, to a multiple of N_d.
  * Accumulation: micro-batches in order inside a rank first, each gradient
    scaled by fl32(1/M) as it is added; the first term starts the sum.
  * Hybrid sharding: ranks k = g*F + j; the reduce sums inside each group
    first (the group's reduce-scatter), then across groups (the all-reduce),
    then divides by N_d.
  * FSDP2: c = ceil(d0/N_d) rows of each parameter per rank (possibly none);
    rank-major communication buffers, each rank's rows of every parameter
    zero-padded to c rows.
  * Gradient scaler: the reduced mean is multiplied by 1/s in fp32 and
    checked for inf/NaN; the flags are OR-ed over all ranks; a flagged step
    changes no state; the scale backs off or grows like dynamic loss scaling.
  * Checkpoint: a load at N_d' re-slices the unit's flat state (the saved
    shards concatenated, cut to T) with the FlatParameter layout of N_d'.
  * Buckets: parameters walked in reverse registration order, a bucket is
    closed before a parameter that would take it over the cap, a parameter
    larger than the cap gets a bucket to itself, parameters are never split.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against facts the pages or mathematics fix (worked example, closed forms,
library routines, brute force).  No function is left unpinned.
"""
from .flat import (Layout, layout, flat_pack, shard_of, sharded_views, ag_unpack,
                   unpack_views, element_source, rank_view_sources)
from .numerics import (AdamWConfig, adamw_scalars, adamw, bf16_to_f32, f32_to_bf16,
                       grad_accumulate, rs_avg, fsdp_shard_step, hybrid_rs_avg,
                       hybrid_shard_step)
from .ddp import bucket_plan, bucket_allreduce_avg, ddp_step
from .scaler import (f16_to_f32, unscaled_mean, found_inf, scaled_shard_step,
                     scaler_update)
from . import checkpoint
from .fsdp2 import (Fsdp2Layout, fsdp2_layout, local_shards, chunk_cat, local_buffer,
                    all_gather_copy_out)
from .ledger import (state_bytes_per_gpu, comm_bytes_per_gpu, hybrid_state_bytes_per_gpu,
                     hybrid_comm_bytes_per_gpu, GB)

__all__ = [
    "Layout", "layout", "flat_pack", "shard_of", "sharded_views", "ag_unpack", "unpack_views",
    "element_source", "rank_view_sources",
    "AdamWConfig", "adamw_scalars", "adamw", "bf16_to_f32", "f32_to_bf16", "grad_accumulate",
    "rs_avg", "fsdp_shard_step", "hybrid_rs_avg", "hybrid_shard_step", "bucket_plan",
    "bucket_allreduce_avg", "ddp_step", "state_bytes_per_gpu", "comm_bytes_per_gpu",
    "hybrid_state_bytes_per_gpu", "hybrid_comm_bytes_per_gpu", "GB", "Fsdp2Layout",
    "fsdp2_layout", "local_shards", "chunk_cat", "local_buffer", "all_gather_copy_out",
    "f16_to_f32", "unscaled_mean", "found_inf", "scaled_shard_step", "scaler_update",
    "checkpoint",
]
