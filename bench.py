"""Benchmark of the sharded optimizer step on the Llama-style 7B rank view.

Workload: one rank's shard of a Llama-7B-shaped model wrapped as 33 FSDP units
(32 layers + embedding unit), Psi = 6,738,415,616, N_d = 8 emulated ranks, so
the rank's shard holds S = 842,301,952 fp32 master weights + both moments and
receives 8 bf16 gradient contributions.  One step = one fused
reduce-scatter-average + AdamW + bf16 cast launch over the whole shard, then
the all-gather of one 202,383,360-parameter layer unit.  Inputs are seeded
synthetic values generated on the device before timing (no data set, no
weights); every step consumes the resident gradients with the step count
advancing.  The step moves ~36 GB, far more than the 129 MB L2, so no L2
flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused shard-step HBM GB/s (% of GB300 peak), params/s at Psi=7B, N_d=8"
KERNEL_SOURCES = ["sharded_optimizer_step_gb300/csrc/step_tma.cu",
                  "sharded_optimizer_step_gb300/csrc/common.cuh"]
FUSED_PROFILES = {
    "llama_7b_rank0_nd8": os.path.join(ROOT, "profiles", "fused_step_llama7b_rank_view.md"),
    "llama_7b_hybrid_nd16_f8_rank0": os.path.join(ROOT, "profiles",
                                                  "fused_step_llama7b_hybrid_nd16_f8.md"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-chunks", type=int, default=4)
    ap.add_argument("--e2e-streams", type=int, default=4)
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + [FSDP2_WORKLOAD, CKPT_WORKLOAD],
                    default="llama_7b_rank0_nd8",
                    help="the Llama-7B rank view under full sharding (the default line), or "
                         "under hybrid sharding with N_d = 16, F = 8")
    ap.add_argument("--layers", type=int, default=0,
                    help="smaller case: only the first N layer units (for profiler captures)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------ environment

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    if world > 1:
        import torch.distributed as dist
        # timing control plane only (barrier + max over ranks); the data path
        # has no collective: each GPU runs its own rank view
        dist.init_process_group("gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(world, x: float) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(world, x: float) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name):
    """DRAM bytes per element of the fused kernel recorded from an ncu capture
    of this workload, if the capture was taken on the current kernel source
    (else None)."""
    try:
        text = open(FUSED_PROFILES[workload_name]).read()
    except (OSError, KeyError):
        return None
    m = re.search(r"traffic_bytes_per_element:\s*([0-9.]+)", text)
    h = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


def smi_index(local: int) -> str:
    """nvidia-smi id of this process's GPU (CUDA_VISIBLE_DEVICES may remap)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    items = [x.strip() for x in vis.split(",") if x.strip()]
    return items[local] if local < len(items) else str(local)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the GPU is busy."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ our arm

WORKLOADS = {
    "llama_7b_rank0_nd8": "llama_7b_rank_view",
    "llama_7b_hybrid_nd16_f8_rank0": "llama_7b_hybrid_view",
    "llama_7b_rank0_nd8_fp16_scaled": "llama_7b_rank_view",
}
LOSS_SCALE = 65536.0


def workload(args):
    from synth import workloads as W
    w = getattr(W, WORKLOADS[args.workload])()
    if args.layers:
        # a smaller case of the same kernel: the first N layer units only
        w.units = w.units[:args.layers]
        w.name = f"{w.name}_first{args.layers}layers"
    return w


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    init_dist(world)
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import sharded_optimizer_step_gb300 as ss
    import synth
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    from synth import workloads as W

    w = workload(args)
    nd, F = w.nd, w.F
    r = rank % F                        # GPU k holds shard k mod F of its own replica
    dev = torch.device("cuda", local)
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    # fp16 gradients under dynamic loss scaling: the gradients arrive
    # multiplied by the scale; check, scaled step and scale update per step
    scaled = args.workload.endswith("_fp16_scaled")
    if scaled:
        w.grad_sigma *= LOSS_SCALE
        w.name = args.workload
    opt = RankShardOptimizer(w.units, nd, r, hp, device=dev, shard_group=w.shard_group,
                             grad_dtype=torch.float16 if scaled else torch.bfloat16)
    scaler = ss.GradScaler(LOSS_SCALE, device=dev) if scaled else None
    S = opt.shard_total
    W.dev_fill_rank_master(w, r, opt.master)
    for q in range(nd):
        W.dev_fill_rank_grad(w, 1, r, q, 0, opt.grad_in[q])
    u = w.extra["ag_unit"]
    Su, Pu = w.unit_shard(u), w.unit_padded(u)
    peers = [torch.empty(Su, dtype=torch.bfloat16, device=dev) for _ in range(F)]
    for q in range(F):
        if q != r:
            synth.dev_fill(w.peer_shard_stream(1, q, u), peers[q])
    full = torch.empty(Pu, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    fused_bytes = (2 * nd + 26) * S
    ag_bytes = 4 * Pu                     # read + write every bf16 element of the unit
    check_bytes = 2 * nd * S if scaled else 0   # the non-finite check reads the slices
    step_bytes = check_bytes + fused_bytes + ag_bytes
    stream = torch.cuda.current_stream(dev)

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if scaled:
            scaler.check(opt.grad_in)
        if ev is not None:
            ev[1].record(stream)
        if scaled:
            opt.t += 1
            scaler.step(opt.grad_in, opt.master, opt.m, opt.v, opt.params, hp, opt.t)
            scaler.update()
        else:
            opt.step()
        if ev is not None:
            ev[2].record(stream)
        opt.gather_unit(u, peers, full)
        if ev is not None:
            ev[3].record(stream)

    clocks = ClockSampler(smi_index(local))
    clocks.start()
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = ss.launch_count()
    torch.cuda.nvtx.range_push("timed_region")
    t_start.record(stream)
    for k in range(args.steps):
        one_step(events[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    launches = ss.launch_count() - launches0
    clk = clocks.stop()
    status = ss.device_status()
    if status:
        raise RuntimeError(f"a TMA-staged wait ran out during the timed steps (status {status})")
    total_ms = t_start.elapsed_time(t_end)
    check_ms = [e[0].elapsed_time(e[1]) for e in events]
    fused_ms = [e[1].elapsed_time(e[2]) for e in events]
    ag_ms = [e[2].elapsed_time(e[3]) for e in events]
    total_ms_max = allreduce_max(world, total_ms)
    all_bytes = allreduce_sum(world, step_bytes * args.steps)
    value = all_bytes / (total_ms_max / 1e3) / 1e9
    ms_per_step = total_ms_max / args.steps
    fused_avg = sum(fused_ms) / len(fused_ms)
    ag_avg = sum(ag_ms) / len(ag_ms)
    peak, peak_kind = measured_peak()
    achieved = fused_bytes / (fused_avg / 1e3) / 1e9
    traffic_per_elem = profiled_traffic(args.workload)

    # end to end through the public API: pinned host inputs copied in every
    # step, the gathered unit read back every step
    e2e = None
    if not args.no_e2e and not scaled:
        e2e = run_e2e(args, torch, ss, opt, peers, full, u, r, nd, stream, step_bytes)
        e2e["value"] = round(allreduce_sum(world, e2e.pop("bytes"))
                             / allreduce_max(world, e2e.pop("seconds")) / 1e9, 1)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(w, r, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
            "config": {"workload": w.name,
                       "model_shape": f"Llama-style 7B, {len(w.units)} FSDP units",
                       "psi": w.psi, "nd": nd, "shard_group": F, "rank": r,
                       "shard_elements": S,
                       "grad_dtype": "f16" if scaled else "bf16", "state_dtype": "f32",
                       "ag_unit_params": Pu,
                       "step": ("non-finite check of the unscaled mean (1 launch), scaled fused "
                                "rs_avg+AdamW+bf16 cast (1 launch), loss-scale update (1 launch), "
                                "then all-gather of one layer unit (1 launch)" if scaled else
                                "fused rs_avg+AdamW+bf16 cast over the rank shard (1 launch), "
                                "then all-gather of one layer unit (1 launch)"),
                       "bytes_per_step": step_bytes,
                       "l2": f"no flush: each step streams {step_bytes / 1e9:.1f} GB vs a 129 MB L2"},
            "params_per_s": round(S * world / (ms_per_step / 1e3), 1),
            "kernels": {**({"check_ms": round(sum(check_ms) / len(check_ms), 4),
                           "check_gbs": round(check_bytes / (sum(check_ms) / len(check_ms) / 1e3)
                                              / 1e9, 1)} if scaled else {}),
                        "fused_ms": round(fused_avg, 4),
                        "fused_gbs": round(achieved, 1),
                        "ag_ms": round(ag_avg, 4),
                        "ag_gbs": round(ag_bytes / (ag_avg / 1e3) / 1e9, 1)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": ("measured: MEASURED_PEAKS.json hbm_gbs (copy, burst)"
                                         if peak_kind == "measured" else "fallback 6800 GB/s"),
                         "kernel": f"rs_adamw_cast_tma<{'f16' if scaled else 'bf16'}> (TMA-staged, N_d = {nd}"
                                   + (f", sharding factor {F})" if F != nd else ")"),
                         "algorithmic_bytes_per_launch": fused_bytes,
                         "traffic": (None if traffic_per_elem is None
                                     else round(traffic_per_elem * S))},
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, torch, ss, opt, peers, full, u, r, nd, stream, step_bytes):
    """Host-resident gradients and peer shards copied in every step, the
    gathered unit copied out.  The shard is cut into chunks: each chunk's 8
    contributions are copied on a pool of copy streams while the fused
    update of the previous chunk runs on the compute stream."""
    S = opt.shard_total
    host_g = [torch.empty(S, dtype=torch.bfloat16, pin_memory=True) for _ in range(nd)]
    for q in range(nd):
        host_g[q].copy_(opt.grad_in[q])
    host_p = [torch.empty(peers[0].numel(), dtype=torch.bfloat16, pin_memory=True)
              for _ in range(len(peers))]
    for q in range(len(peers)):
        host_p[q].copy_(peers[q])
    host_out = torch.empty(full.numel(), dtype=torch.bfloat16, pin_memory=True)
    torch.cuda.synchronize()
    h2d = sum(x.numel() * 2 for x in host_g) + sum(x.numel() * 2 for q, x in enumerate(host_p)
                                                   if q != r)
    d2h = host_out.numel() * 2
    n_chunks = max(1, args.e2e_chunks)
    step8 = -(-S // (8 * n_chunks)) * 8
    bounds = [min(S, c * step8) for c in range(n_chunks)] + [S]
    copy_streams = [torch.cuda.Stream(device=stream.device) for _ in range(max(1, args.e2e_streams))]

    def e2e_step():
        prev = stream.record_event()          # last step's kernels are done with the buffers
        k = 0
        chunk_ready = []
        for c in range(n_chunks):
            a, b = bounds[c], bounds[c + 1]
            evs = []
            for q in range(nd):
                cs = copy_streams[k % len(copy_streams)]
                k += 1
                cs.wait_event(prev)
                with torch.cuda.stream(cs):
                    opt.grad_in[q][a:b].copy_(host_g[q][a:b], non_blocking=True)
                evs.append(cs.record_event())
            chunk_ready.append(evs)
        peer_evs = []
        for q in range(len(peers)):
            if q != r:
                cs = copy_streams[k % len(copy_streams)]
                k += 1
                cs.wait_event(prev)
                with torch.cuda.stream(cs):
                    peers[q].copy_(host_p[q], non_blocking=True)
                peer_evs.append(cs.record_event())
        opt.begin_step()
        for c in range(n_chunks):
            for e in chunk_ready[c]:
                stream.wait_event(e)
            opt.update_range(bounds[c], bounds[c + 1], stream=stream)
        for e in peer_evs:
            stream.wait_event(e)
        opt.gather_unit(u, peers, full, stream=stream)
        host_out.copy_(full, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    sec = a.elapsed_time(b) / 1e3
    return {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "ms_per_step": round(sec * 1e3 / args.e2e_steps, 3),
            "h2d_gbs": round(h2d * args.e2e_steps / sec / 1e9, 1),
            "bytes": step_bytes * args.e2e_steps, "seconds": sec,
            "path": (f"pinned host buffers -> {len(copy_streams)} copy streams, shard in "
                     f"{n_chunks} chunks overlapped with the fused update; C-ABI calls")}


# ------------------------------------------------------- CPU baseline / reference

def _oracle_sample(w, r, n, step, rng_seed=0):
    """Inputs of a contiguous sample of n shard elements (plus the matching
    sample of the all-gather), generated on the host."""
    import numpy as np
    from synth import workloads as W
    import synth
    start = (rng_seed * 7919 * n) % max(1, 842_301_952 - n)
    idx = np.arange(start, start + n, dtype=np.int64)
    contribs = [W.host_gather_rank_grad(w, step, r, q, 0, idx) for q in range(w.nd)]
    p = W.host_gather_rank_master(w, r, idx)
    u = w.extra["ag_unit"]
    n_ag = max(1, n // (w.F * 4))
    shards = [synth.host_fill(w.peer_shard_stream(step, q, u), 0, n_ag, "bf16") for q in range(w.F)]
    return contribs, p, shards


def _oracle_step(w, contribs, n, p, m, v, hp, t):
    import oracle
    if w.F == w.nd:
        return oracle.fsdp_shard_step(contribs, 0, n, p, m, v, hp, t)
    return oracle.hybrid_shard_step(contribs, w.F, 0, n, p, m, v, hp, t)


def _time_oracle(w, contribs, p, shards, t):
    import numpy as np
    import oracle
    from oracle.numerics import AdamWConfig
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    n = p.size
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    lay = oracle.layout([w.F * shards[0].size], w.F)
    t0 = time.perf_counter()
    _oracle_step(w, contribs, n, p, m, v, hp, t)
    oracle.ag_unpack(shards, lay)
    dt = time.perf_counter() - t0
    bytes_ = (2 * w.nd + 26) * n + 4 * w.F * shards[0].size
    return dt, bytes_


def cpu_baseline(w, r, budget_s=10.0, n=4_000_000):
    contribs, p, shards = _oracle_sample(w, r, n, 1)
    total_t, total_b, reps = 0.0, 0, 0
    while total_t < budget_s and reps < 50:
        dt, b = _time_oracle(w, contribs, p, shards, reps + 1)
        total_t += dt
        total_b += b
        reps += 1
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{reps} x (fused step on {n} contiguous shard elements of {w.name} "
                      f"+ all-gather of {shards[0].size * w.F} bf16), numpy single-threaded"}


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    w = workload(args)
    r = 0
    n = 2_000_000
    contribs, p, shards = _oracle_sample(w, r, n, 1)
    for k in range(args.warmup):
        _time_oracle(w, contribs, p, shards, k + 1)
    ts, bs = [], []
    for k in range(args.steps):
        dt, b = _time_oracle(w, contribs, p, shards, args.warmup + k + 1)
        ts.append(dt)
        bs.append(b)
    value = sum(bs) / sum(ts) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(ts) / len(ts), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "psi": w.psi, "nd": w.nd, "rank": r,
                   "sample_elements_per_step": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: fused step on {n} shard elements + all-gather of "
                                   f"{shards[0].size * w.F} bf16"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ------------------------------------------------------- FSDP2 layer group

FSDP2_WORKLOAD = "llama_7b_fsdp2_layer_nd8"


def _fsdp2_bytes(shapes, nd, local):
    numel = sum(int(math.prod(s)) for s in shapes)
    cc = nd * 2 * (numel * 2)            # every rank reads and writes its bf16 gradients
    cc += nd * 2 * (nd * local - numel)  # zero padding rows written
    fused = nd * (2 * nd + 26) * local   # nd fused launches over the local buffers
    ag = 2 * (numel * 2)                 # the gathered bf16 rows read and written
    return cc, fused, ag


def run_fsdp2(args):
    """One Llama-7B layer as an FSDP2 group on 8 emulated ranks: every rank's
    full per-parameter bf16 gradients chunk-cat into its reduce-scatter
    input, one fused step per rank on its padded local buffer, then the
    all-gather straight into the 9 full bf16 parameter tensors."""
    import torch
    world, rank, local_rank = dist_env()
    init_dist(world)
    torch.cuda.set_device(local_rank)
    import __graft_entry__
    __graft_entry__.build()
    import sharded_optimizer_step_gb300 as ss
    import synth
    from synth import workloads as W
    w = W.llama_7b_rank_view()
    shapes = w.units[0]
    nd = w.nd
    dev = torch.device("cuda", local_rank)
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    lay = ss.fsdp2_layout(shapes, nd)
    L = lay.local
    grads = [[torch.empty(sh, dtype=torch.bfloat16, device=dev) for sh in shapes]
             for _ in range(nd)]
    for q in range(nd):
        for t, g in enumerate(grads[q]):
            synth.dev_fill(w.grad_stream(1, q, 0, 100 + t), g)
    rs_in = [torch.empty(nd * L, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    masters = [torch.empty(sh, dtype=torch.float32, device=dev) for sh in shapes]
    for t, mt in enumerate(masters):
        synth.dev_fill(w.master_stream(100 + t), mt)
    master = ss.fsdp2_chunk_cat(masters, nd)
    del masters
    m = torch.zeros(nd * L, device=dev)
    v = torch.zeros(nd * L, device=dev)
    out = torch.empty(nd * L, dtype=torch.bfloat16, device=dev)
    params = [torch.empty(sh, dtype=torch.bfloat16, device=dev) for sh in shapes]
    stream = torch.cuda.current_stream(dev)
    cc_b, fused_b, ag_b = _fsdp2_bytes(shapes, nd, L)
    step_b = cc_b + fused_b + ag_b
    t_step = [0]

    def one_step(ev=None):
        t_step[0] += 1
        if ev is not None:
            ev[0].record(stream)
        for q in range(nd):
            ss.fsdp2_chunk_cat(grads[q], nd, out=rs_in[q])
        if ev is not None:
            ev[1].record(stream)
        for r in range(nd):
            sl = slice(r * L, (r + 1) * L)
            ss.fsdp_rs_avg_adamw_cast([x[sl] for x in rs_in], master[sl], m[sl], v[sl], out[sl],
                                      hp, t_step[0])
        if ev is not None:
            ev[2].record(stream)
        ss.fsdp2_all_gather_copy_out([out[r * L:(r + 1) * L] for r in range(nd)], params)
        if ev is not None:
            ev[3].record(stream)

    clocks = ClockSampler(smi_index(local_rank))
    clocks.start()
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = ss.launch_count()
    torch.cuda.nvtx.range_push("timed_region")
    a.record(stream)
    for k in range(args.steps):
        one_step(events[k])
    b.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    launches = ss.launch_count() - launches0
    clk = clocks.stop()
    if ss.device_status():
        raise RuntimeError("a TMA-staged wait ran out during the timed steps")
    total_ms = allreduce_max(world, a.elapsed_time(b))
    ms = [[e[i].elapsed_time(e[i + 1]) for e in events] for i in range(3)]
    avg = [sum(x) / len(x) for x in ms]
    peak, peak_kind = measured_peak()
    fused_launch = fused_b / nd
    achieved = fused_launch / (avg[1] / nd / 1e3) / 1e9
    value = allreduce_sum(world, step_b * args.steps) / (total_ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
            "config": {"workload": FSDP2_WORKLOAD, "group": "one Llama-7B layer (9 parameters, "
                       "202,383,360 elements)", "nd": nd, "local_elements": L,
                       "step": "8 x chunk-cat of a rank's full bf16 gradients, 8 x fused step on "
                               "the padded local buffers, all-gather copy-out into the 9 full "
                               "parameters", "bytes_per_step": step_b,
                       "l2": f"no flush: each step streams {step_b / 1e9:.1f} GB vs a 129 MB L2"},
            "kernels": {"chunk_cat_ms": round(avg[0], 4),
                        "chunk_cat_gbs": round(cc_b / (avg[0] / 1e3) / 1e9, 1),
                        "fused_ms_per_launch": round(avg[1] / nd, 4),
                        "fused_gbs": round(achieved, 1),
                        "copy_out_ms": round(avg[2], 4),
                        "copy_out_gbs": round(ag_b / (avg[2] / 1e3) / 1e9, 1)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": ("measured: MEASURED_PEAKS.json hbm_gbs (copy, burst)"
                                         if peak_kind == "measured" else "fallback 6800 GB/s"),
                         "kernel": "rs_adamw_cast_tma<bf16> on one rank's local buffer",
                         "algorithmic_bytes_per_launch": fused_launch, "traffic": None},
            "e2e": None, "gpu_launches": launches, "clocks": clk, "cpu_baseline": None,
        }))


# ------------------------------------------------------------ checkpoint

CKPT_WORKLOAD = "ckpt_gpt2_small_nd8_to_nd4"


def run_ckpt(args):
    """Sharded checkpoint of the GPT-2-small-shaped model: every one of 8
    ranks saves its fp32 master / m / v shards (device -> pinned host -> its
    own file, ranks in parallel), then 4 ranks of a new layout load their
    resharded state (pieces of the saved files -> pinned host -> device)."""
    import shutil
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    import sharded_optimizer_step_gb300 as ss
    from sharded_optimizer_step_gb300 import checkpoint as ck
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    from synth import workloads as W
    w = W.gpt2_small()
    hp = ss.AdamW()
    old = [RankShardOptimizer(w.units, 8, r, hp, device="cuda:0") for r in range(8)]
    for o in old:
        W.dev_fill_rank_master(w, o.rank, o.master)
        for q in range(8):
            W.dev_fill_rank_grad(w, 1, o.rank, q, 0, o.grad_in[q])
        o.step()
    new = [RankShardOptimizer(w.units, 4, r, hp, device="cuda:0") for r in range(4)]
    torch.cuda.synchronize()
    state_bytes = sum(3 * 4 * o.shard_total for o in old)
    directory = tempfile.mkdtemp(prefix="shst_ckpt_")
    saves, loads = [], []
    try:
        for _ in range(max(1, args.steps)):
            t0 = time.perf_counter()
            ck.save(directory, old)
            t1 = time.perf_counter()
            ck.load(directory, new)
            t2 = time.perf_counter()
            saves.append(t1 - t0)
            loads.append(t2 - t1)
        disk = sum(os.path.getsize(ck.rank_file(directory, r)) for r in range(8))
    finally:
        shutil.rmtree(directory, ignore_errors=True)
    sv, ld = statistics.median(saves), statistics.median(loads)
    print(json.dumps({
        "metric": "sharded checkpoint save / load GB/s (fp32 master + moments)",
        "value": round(state_bytes / sv / 1e9, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": len(saves), "warmup": 0, "ms_per_step": round(1e3 * (sv + ld), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": CKPT_WORKLOAD, "state_bytes": state_bytes,
                                        "file_bytes": disk, "save_ranks": 8, "load_ranks": 4,
                                        "directory": "a temporary directory under /tmp"},
        "save_gbs": round(state_bytes / sv / 1e9, 2), "load_gbs": round(state_bytes / ld / 1e9, 2),
        "save_s": round(sv, 3), "load_s": round(ld, 3),
        "roofline": None, "e2e": None, "gpu_launches": 0, "clocks": None, "cpu_baseline": None,
        "note": "host-IO bound (device <-> pinned host copies and file reads / writes); "
                "no GPU kernel runs"}))


def main():
    args = parse()
    if args.workload == CKPT_WORKLOAD:
        run_ckpt(args)
        return
    if args.workload == FSDP2_WORKLOAD:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the FSDP2 group line has no CPU arm; use the default workload"}))
            return
        run_fsdp2(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
