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
RAGGED_METRIC = ("flat_pack + all-gather HBM GB/s of a ragged Llama-7B layer unit "
                 "(tensors at odd element offsets), N_d=8")
TMA_SOURCES = ["sharded_optimizer_step_gb300/csrc/step_tma.cu",
               "sharded_optimizer_step_gb300/csrc/common.cuh"]
REGISTER_SOURCES = ["sharded_optimizer_step_gb300/csrc/step.cu",
                    "sharded_optimizer_step_gb300/csrc/common.cuh"]
COPY_SOURCES = ["sharded_optimizer_step_gb300/csrc/copy.cu",
                "sharded_optimizer_step_gb300/csrc/common.cuh"]
FSDP2_SOURCES = ["sharded_optimizer_step_gb300/csrc/fsdp2_step.cu",
                 "sharded_optimizer_step_gb300/csrc/common.cuh"]
# per bench line: the ncu summary of its dominant kernel (DRAM bytes per
# element, recorded with the hash of the sources that kernel is built from)
PROFILES = {
    "llama_7b_rank0_nd8": ("fused_step_llama7b_rank_view.md", REGISTER_SOURCES),
    "llama_7b_hybrid_nd16_f8_rank0": ("fused_step_llama7b_hybrid_nd16_f8.md", REGISTER_SOURCES),
    "llama_7b_rank0_nd8_fp16_scaled": ("scaled_step_llama7b_rank_view_fp16.md",
                                       REGISTER_SOURCES),
    "llama_1b_rank0_nd8_m4": ("accumulate_llama1b_rank_view_m4.md",
                              COPY_SOURCES + ["sharded_optimizer_step_gb300/csrc/accum_step.cu"]),
    "ddp_nd8_buckets": ("ddp_buckets_nd8_adamw.md", REGISTER_SOURCES),
    "llama_7b_layer_ragged_nd8": ("pack_gather_llama7b_layer_ragged.md", COPY_SOURCES),
    "llama_7b_fsdp2_layer_nd8": ("fsdp2_llama7b_layer_group.md", FSDP2_SOURCES),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of this node, one process each under torchrun (one replica "
                         "of the line per GPU)")
    ap.add_argument("--steps", type=int, default=200, help="timed steps")
    ap.add_argument("--warmup", type=int, default=5, help="untimed steps before the timing")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="ours: the library on the GPU; reference: the CPU oracle on a "
                         "bounded sample of the same workload")
    ap.add_argument("--e2e-steps", type=int, default=5,
                    help="steps of the end-to-end leg (host buffers in and out)")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="default line's end-to-end leg: chunks of the shard whose copies "
                         "overlap the previous chunk's update")
    ap.add_argument("--e2e-streams", type=int, default=4,
                    help="default line's end-to-end leg: copy streams")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + [FSDP2_WORKLOAD, CKPT_WORKLOAD,
                                                             ACCUM_WORKLOAD, DDP_WORKLOAD,
                                                             RAGGED_WORKLOAD, UNIT9M_WORKLOAD,
                                                             GPT2_WORKLOAD],
                    default="llama_7b_rank0_nd8",
                    help="the Llama-7B rank view under full sharding (the default line); the "
                         "other lines time the other steps of the path")
    ap.add_argument("--layers", type=int, default=0,
                    help="smaller case: only the first N layer units (for profiler captures)")
    ap.add_argument("--nd", type=int, default=0,
                    help="rank-view lines (default, hybrid, fp16), the DDP and the FSDP2 "
                         "lines: another "
                         "number of emulated ranks N_d (0: the workload's own), for kernel "
                         "sweeps and profiler captures")
    ap.add_argument("--shrink", type=int, default=1,
                    help="FSDP2 and ragged lines: a smaller case of the same kernels, every "
                         "parameter's first dimension (ragged: every tensor) divided by this "
                         "(for profiler captures)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--tma-stages", type=int, default=0,
                    help="shared-memory stages of the TMA-staged kernels "
                         "(0: about 128 KB of tiles in flight per SM)")
    ap.add_argument("--kernel-path", choices=["auto", "register", "tma"], default="auto",
                    help="streaming kernels: TMA-staged where they measured faster (auto), "
                         "register-staged only, or TMA-staged wherever the arguments allow")
    ap.add_argument("--graph", action="store_true",
                    help="default / hybrid / accumulation lines and the two whole-job "
                         "lines: the step count and AdamW scalars on the device, the "
                         "accumulate launches, the fused update and the all-gather replayed "
                         "from CUDA graphs captured once")
    ap.add_argument("--no-dependent-launch", action="store_true",
                    help="launch every kernel as an ordinary launch (by default each call's "
                         "first kernel is a programmatic dependent of the kernel before it, "
                         "waiting for it before touching memory, and the later buckets / "
                         "copies of a call overlap the previous one's drain)")
    ap.add_argument("--fsdp2-chunk-cat", action="store_true",
                    help="FSDP2 line: time the step through the chunk-cat (the reduce-scatter "
                         "input a collective needs) and the fused step on its pieces; by "
                         "default the step is read straight from the gradients (same bits) "
                         "and the chunk-cat path is timed beside it")
    ap.add_argument("--accum-two-pass", action="store_true",
                    help="accumulation line: accumulate every micro-batch with its own launch "
                         "and run the fused step on the accumulators (the last micro-batch "
                         "is otherwise accumulated inside the fused step)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true",
                    help="skip the CPU oracle baseline beside the line")
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


def kernel_source_hash(sources=TMA_SOURCES):
    """Hash of the code in `sources` with comments and blank space removed, so
    that a comment-only edit keeps a profile's figures valid."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name):
    """DRAM bytes per element of a bench line's dominant kernel, recorded from
    an ncu capture of this workload, if the capture was taken on the current
    source of that kernel (else None)."""
    try:
        name, sources = PROFILES[workload_name]
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except (OSError, KeyError):
        return None
    m = re.search(r"traffic_bytes_per_element:\s*([0-9.]+)", text)
    h = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash(sources):
        return None
    return float(m.group(1))


def _apply_stages(args):
    import sharded_optimizer_step_gb300 as ss
    ss.set_tma_stages(args.tma_stages)
    ss.set_fused_path(args.kernel_path)
    ss.set_dependent_launch(not args.no_dependent_launch)


def _stages_name(args):
    if args.kernel_path != "auto":
        return f"{args.kernel_path}-staged kernels" + (
            "" if args.tma_stages == 0 else f", {args.tma_stages} stages")
    return "auto" if args.tma_stages == 0 else args.tma_stages


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


def fill_rank_view(opt, buf, stream_of):
    """Seeded inputs of one of a rank's buffers, placed where the library's
    FlatParameter layout puts each tensor's piece (``rank_pieces``, i.e.
    fsdp_shard_pieces); the units' padding stays zero."""
    import synth
    synth.dev_fill_pieces(buf, opt.rank_pieces(), stream_of)


def oracle_rank_values(w, r, idx, stream_of, dtype):
    """CPU-baseline inputs: the values at positions idx of rank r's buffer,
    each traced to its tensor element by the oracle's own layout."""
    import oracle
    import synth
    lays = [oracle.layout(w.unit_numels(u), w.F) for u in range(len(w.units))]
    u, t, k = oracle.rank_view_sources(lays, r, idx)
    return synth.host_gather_sources(u, t, k, stream_of, dtype)


def workload(args):
    from synth import workloads as W
    w = getattr(W, WORKLOADS[args.workload])()
    if args.layers:
        # a smaller case of the same kernel: the first N layer units only
        w.units = w.units[:args.layers]
        w.name = f"{w.name}_first{args.layers}layers"
    if args.nd and args.nd != w.nd:
        if w.shard_group and args.nd % w.shard_group:
            raise SystemExit("--nd must be a multiple of the sharding factor")
        w.nd = args.nd
        w.name = f"{w.name}_nd{args.nd}"
    return w


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    init_dist(world)
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
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
    fill_rank_view(opt, opt.master, w.master_stream)
    for q in range(nd):
        fill_rank_view(opt, opt.grad_in[q], lambda u, k, q=q: w.grad_stream(1, q, 0, u, k))
    u = w.extra["ag_unit"]
    Su, Pu = opt.layouts[u].shard, opt.layouts[u].padded
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

    graph_launches = 0
    if args.graph:
        if scaled:
            raise SystemExit("--graph: the default and hybrid lines only")
        # the step count on the device; the update (advance + fused launch)
        # and the all-gather each captured once, after an eager warm-up
        opt.device_step_state()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            opt.step_on_device()
            opt.gather_unit(u, peers, full)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g_update, g_gather = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        l0 = ss.launch_count()
        with torch.cuda.graph(g_update):
            opt.step_on_device()
        with torch.cuda.graph(g_gather):
            opt.gather_unit(u, peers, full)
        graph_launches = ss.launch_count() - l0     # kernels per replayed step

        def one_step(ev=None):            # noqa: F811 -- the graph form of the step
            if ev is not None:
                ev[0].record(stream)
                ev[1].record(stream)
            g_update.replay()
            if ev is not None:
                ev[2].record(stream)
            g_gather.replay()
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
    launches = ss.launch_count() - launches0 + graph_launches * args.steps
    fused_kernel = ss.last_kernel()     # the fused step is each step's last streaming call
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
    achieved = fused_bytes / (fused_avg / 1e3) / 1e9
    traffic_per_elem = (None if args.layers or args.nd or args.kernel_path != "auto"
                        or args.tma_stages else profiled_traffic(args.workload))

    # the inter-rank bytes the step's emulated collectives stand for (ring
    # model), from one more step issued call by call
    torch.cuda.synchronize()
    ss.comm_counter(reset=True)
    if args.graph:
        opt.step_on_device()
        opt.gather_unit(u, peers, full)
    else:
        one_step()
    torch.cuda.synchronize()
    comm_step = ss.comm_counter(reset=True)

    pack = _time_flat_pack(torch, ss, w, u, nd if F == nd else F, dev, stream)

    # end to end through the public API: pinned host inputs copied in every
    # step, the gathered unit read back every step
    e2e = None
    if not args.no_e2e and not scaled and not args.graph:
        try:
            e2e = run_e2e(args, torch, ss, opt, peers, full, u, r, nd, stream, step_bytes)
            failed = ""
        except RuntimeError as exc:          # e.g. the host cannot pin this much memory
            failed = str(exc).splitlines()[0][:200]
            torch.cuda.synchronize()
        # every rank takes part in the same reductions, whatever happened
        n_failed = allreduce_sum(world, 1.0 if failed else 0.0)
        got_bytes = allreduce_sum(world, 0.0 if failed else float(e2e["bytes"]))
        got_sec = allreduce_max(world, 0.0 if failed else e2e["seconds"])
        if n_failed:
            e2e = {"value": None, "unit": "GB/s", "unavailable":
                   f"end-to-end leg failed on {int(n_failed)} rank(s): {failed or 'another rank'}"}
        else:
            e2e.pop("bytes")
            e2e.pop("seconds")
            e2e["value"] = round(got_bytes / got_sec / 1e9, 1)
    elif not args.no_e2e and scaled and not args.graph:
        # the check must see every contribution before any update, so the
        # copies are not overlapped with the step here
        e2e = _e2e_plain(torch, stream, opt.grad_in + [peers[q] for q in range(F) if q != r],
                         [full], one_step, step_bytes, world, args.e2e_steps,
                         "the 8 scaled fp16 contributions and the peers' shards in, the "
                         "gathered layer unit out")

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu:
        sample = _oracle_sample(w, r, 4_000_000, 1)
        cpu = cpu_baseline(w, r, budget_s=args.cpu_seconds, sample=sample)
        cpu_all = cpu_baseline_all_cores(w, r, budget_s=args.cpu_seconds, sample=sample)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
            "config": {"workload": w.name, "tma_stages": _stages_name(args),
                       "graph": bool(args.graph),
                       "dependent_launch": not args.no_dependent_launch,
                       "model_shape": f"Llama-style 7B, {len(w.units)} FSDP units",
                       "psi": w.psi, "nd": nd, "shard_group": F, "rank": r,
                       "shard_elements": S,
                       "grad_dtype": "f16" if scaled else "bf16", "state_dtype": "f32",
                       "ag_unit_params": Pu,
                       "step": ("non-finite check of the unscaled mean (1 launch), scaled fused "
                                "rs_avg+AdamW+bf16 cast (1 launch), loss-scale update (1 launch), "
                                "then all-gather of one layer unit (1 launch)" if scaled else
                                "step count advanced on the device (1 launch), fused "
                                "rs_avg+AdamW+bf16 cast reading its scalars there (1 launch), "
                                "all-gather of one layer unit (1 launch), replayed from two "
                                "CUDA graphs" if args.graph else
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
                        "ag_gbs": round(ag_bytes / (ag_avg / 1e3) / 1e9, 1),
                        **pack},
            "roofline": _roofline(achieved, f"{fused_kernel}, N_d = {nd}"
                                  + (f", sharding factor {F}" if F != nd else ""), fused_bytes,
                                  None if traffic_per_elem is None
                                  else round(traffic_per_elem * S)),
            "e2e": e2e,
            **({"e2e_note": "the end-to-end leg runs without --graph"} if args.graph else {}),
            "emulated_comm": {
                "bytes_per_step": round(comm_step),
                "link_gbs_to_hide": round(comm_step / (ms_per_step / 1e3) / 1e9, 1),
                "model": "bytes this rank would send per step if each emulated collective ran "
                         "as a ring ((N_d-1)/N_d kept): the reduce-scatter into the fused step "
                         "and the all-gather of one layer unit; link_gbs_to_hide = that over "
                         "the measured step time"},
            "gpu_launches": launches,
            **({"gpu_launches_note": f"{graph_launches} kernels per replayed step, counted "
                                     f"when the graphs were captured"} if args.graph else {}),
            "clocks": clk,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _time_flat_pack(torch, ss, w, u, nd, dev, stream, reps=20):
    """flat_pack of one unit's tensors (a layer unit of the workload) into its
    padded FlatParameter, timed on its own outside the step: the one-time
    layout copy of every unit.  2 B read + 2 B written per element."""
    import synth
    shapes = w.units[u]
    tensors = []
    for k, sh in enumerate(shapes):
        t = torch.empty(sh, dtype=torch.bfloat16, device=dev)
        synth.dev_fill(w.peer_shard_stream(2, k, u), t.view(-1))
        tensors.append(t)
    lay = ss.fsdp_layout([t.numel() for t in tensors], nd)
    flat = torch.empty(lay.padded, dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        ss.fsdp_flat_pack(tensors, nd, flat=flat)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        ss.fsdp_flat_pack(tensors, nd, flat=flat)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    bytes_ = 4 * lay.total
    return {"flat_pack_ms": round(ms, 4), "flat_pack_gbs": round(bytes_ / (ms / 1e3) / 1e9, 1),
            "flat_pack_elements": lay.total}


E2E_WINDOWS = 3                   # timed windows of the default line's end-to-end leg


def run_e2e(args, torch, ss, opt, peers, full, u, r, nd, stream, step_bytes):
    """Host-resident gradients and peer shards copied in every step, the
    gathered unit copied out.  The shard is cut into chunks: each chunk's 8
    contributions are copied on a pool of copy streams while the fused update
    of the previous chunk runs on the compute stream.  Steps overlap as far
    as the buffers allow: a chunk's gradient buffers are refilled as soon as
    the previous step's update of that chunk is done, the peers' shards once
    the previous all-gather has read them, and the gathered unit is read
    back on its own stream while the next step's copies run."""
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
    d2h_stream = torch.cuda.Stream(device=stream.device)
    # events of the previous step that free a buffer for the next one
    free = {"chunk": [None] * n_chunks, "peers": None, "full": None}

    def after(cs, ev, start):
        if ev is not None:
            cs.wait_event(ev)
        if start is not None:
            cs.wait_event(start)

    def e2e_step(start=None):
        k = 0
        chunk_ready = []
        for c in range(n_chunks):
            a, b = bounds[c], bounds[c + 1]
            evs = []
            for q in range(nd):
                cs = copy_streams[k % len(copy_streams)]
                k += 1
                after(cs, free["chunk"][c], start)
                with torch.cuda.stream(cs):
                    opt.grad_in[q][a:b].copy_(host_g[q][a:b], non_blocking=True)
                evs.append(cs.record_event())
            chunk_ready.append(evs)
        peer_evs = []
        for q in range(len(peers)):
            if q != r:
                cs = copy_streams[k % len(copy_streams)]
                k += 1
                after(cs, free["peers"], start)
                with torch.cuda.stream(cs):
                    peers[q].copy_(host_p[q], non_blocking=True)
                peer_evs.append(cs.record_event())
        opt.begin_step()
        for c in range(n_chunks):
            for e in chunk_ready[c]:
                stream.wait_event(e)
            opt.update_range(bounds[c], bounds[c + 1], stream=stream)
            free["chunk"][c] = stream.record_event()
        for e in peer_evs:
            stream.wait_event(e)
        if free["full"] is not None:
            stream.wait_event(free["full"])      # the previous read-back is done with `full`
        opt.gather_unit(u, peers, full, stream=stream)
        gathered = stream.record_event()
        free["peers"] = gathered
        d2h_stream.wait_event(gathered)
        with torch.cuda.stream(d2h_stream):
            host_out.copy_(full, non_blocking=True)
        free["full"] = d2h_stream.record_event()

    e2e_step()
    torch.cuda.synchronize()
    # three windows of e2e_steps steps each: the host link is shared with the
    # machine's other tenants, so one window can catch a slow moment; the
    # median window is the figure, the others are reported beside it
    windows = []
    for _ in range(E2E_WINDOWS):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(args.e2e_steps):
            e2e_step(a if k == 0 else None)
        stream.wait_event(free["full"])          # the last read-back is inside the timing
        b.record(stream)
        torch.cuda.synchronize()
        windows.append(a.elapsed_time(b) / 1e3)
    sec = statistics.median(windows)
    return {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "ms_per_step": round(sec * 1e3 / args.e2e_steps, 3),
            "h2d_gbs": round(h2d * args.e2e_steps / sec / 1e9, 1),
            "windows_ms_per_step": [round(x * 1e3 / args.e2e_steps, 3) for x in windows],
            "bytes": step_bytes * args.e2e_steps, "seconds": sec,
            "path": (f"pinned host buffers -> {len(copy_streams)} copy streams, shard in "
                     f"{n_chunks} chunks overlapped with the fused update; steps overlap per "
                     f"chunk; read-back on its own stream; C-ABI calls; the median of "
                     f"{E2E_WINDOWS} windows of {args.e2e_steps} steps")}


# ------------------------------------------------------- CPU baseline / reference

def _oracle_sample(w, r, n, step, rng_seed=0):
    """Inputs of a contiguous sample of n shard elements (plus the matching
    sample of the all-gather), generated on the host."""
    import numpy as np
    import oracle
    import synth
    total = sum(oracle.layout(w.unit_numels(u), w.F).shard for u in range(len(w.units)))
    start = (rng_seed * 7919 * n) % max(1, total - n)
    idx = np.arange(start, start + n, dtype=np.int64)
    contribs = [oracle_rank_values(w, r, idx, lambda u, k, q=q: w.grad_stream(step, q, 0, u, k),
                                   "bf16") for q in range(w.nd)]
    p = oracle_rank_values(w, r, idx, w.master_stream, "f32")
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


def cpu_baseline(w, r, budget_s=10.0, n=4_000_000, sample=None):
    contribs, p, shards = sample or _oracle_sample(w, r, n, 1)
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


def cpu_baseline_all_cores(w, r, budget_s=10.0, n=4_000_000, sample=None):
    """The same oracle (unchanged) on all host cores: the sample is cut into
    one contiguous element range per thread and each thread runs the fused
    step and its share of the all-gather on its range (numpy releases the
    interpreter lock inside its array operations).  Labelled as such; the
    single-threaded figure is the baseline of record."""
    import concurrent.futures as cf
    threads = max(1, os.cpu_count() or 1)
    contribs, p, shards = sample or _oracle_sample(w, r, n, 1)
    per = -(-n // threads)
    ranges = [(a, min(n, a + per)) for a in range(0, n, per)]
    s_per = -(-shards[0].size // threads)
    pieces = [[s[a:a + s_per] for s in shards] for a in range(0, shards[0].size, s_per)]

    def work(k, t):
        a, e = ranges[k]
        dt, b = _time_oracle(w, [c[a:e] for c in contribs], p[a:e].copy(),
                             pieces[min(k, len(pieces) - 1)], t)
        return b

    total_t, total_b, reps = 0.0, 0, 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while total_t < budget_s and reps < 50:
            t0 = time.perf_counter()
            total_b += sum(ex.map(lambda k: work(k, reps + 1), range(len(ranges))))
            total_t += time.perf_counter() - t0
            reps += 1
    return {"value": round(total_b / total_t / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle, all cores (numpy, one thread per contiguous element range)",
            "sample": f"{reps} x (fused step on {n} contiguous shard elements of {w.name} split "
                      f"over {len(ranges)} threads + their all-gather shares)"}


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
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    import synth
    from synth import workloads as W
    w = W.llama_7b_rank_view()
    shapes = w.units[0]
    if args.shrink > 1:           # a smaller case: every parameter's dim 0 divided
        shapes = [(-(-sh[0] // args.shrink),) + tuple(sh[1:]) for sh in shapes]
    nd = args.nd or w.nd
    dev = torch.device("cuda", local_rank)
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    lay = ss.fsdp2_layout(shapes, nd)
    L = lay.local
    grads = [[torch.empty(sh, dtype=torch.bfloat16, device=dev) for sh in shapes]
             for _ in range(nd)]
    for q in range(nd):
        for t, g in enumerate(grads[q]):
            synth.dev_fill(w.grad_stream(1, q, 0, 100, t), g)
    rs_in = [torch.empty(nd * L, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    masters = [torch.empty(sh, dtype=torch.float32, device=dev) for sh in shapes]
    for t, mt in enumerate(masters):
        synth.dev_fill(w.master_stream(100, t), mt)
    master = ss.fsdp2_chunk_cat(masters, nd)
    del masters
    m = torch.zeros(nd * L, device=dev)
    v = torch.zeros(nd * L, device=dev)
    out = torch.empty(nd * L, dtype=torch.bfloat16, device=dev)
    params = [torch.empty(sh, dtype=torch.bfloat16, device=dev) for sh in shapes]
    stream = torch.cuda.current_stream(dev)
    cc_b, fused_b, ag_b = _fsdp2_bytes(shapes, nd, L)
    t_step = [0]
    fsdp2_step = ss.Fsdp2Step(grads)       # the gradient buffers checked once

    def chunk_cat_step(ev=None):
        """chunk-cat of every rank's gradients, the fused step per rank on the
        pieces, the copy-out"""
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

    def direct_step(ev=None):
        """every rank's step read straight from the ranks' gradients (the same
        bits, no chunk-cat copy), the copy-out"""
        t_step[0] += 1
        if ev is not None:
            ev[0].record(stream)
            ev[1].record(stream)
        for r in range(nd):
            sl = slice(r * L, (r + 1) * L)
            fsdp2_step(r, master[sl], m[sl], v[sl], out[sl], hp, t_step[0])
        if ev is not None:
            ev[2].record(stream)
        ss.fsdp2_all_gather_copy_out([out[r * L:(r + 1) * L] for r in range(nd)], params)
        if ev is not None:
            ev[3].record(stream)

    direct = not args.fsdp2_chunk_cat
    one_step, other_step = ((direct_step, chunk_cat_step) if direct
                            else (chunk_cat_step, direct_step))
    step_b = fused_b + ag_b + (0 if direct else cc_b)
    other_b = fused_b + ag_b + (cc_b if direct else 0)

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
    fused_kernel = ss.last_kernel()
    clk = clocks.stop()
    if ss.device_status():
        raise RuntimeError("a TMA-staged wait ran out during the timed steps")
    total_ms = allreduce_max(world, a.elapsed_time(b))
    ms = [[e[i].elapsed_time(e[i + 1]) for e in events] for i in range(3)]
    avg = [sum(x) / len(x) for x in ms]
    fused_launch = fused_b / nd
    achieved = fused_launch / (avg[1] / nd / 1e3) / 1e9
    value = allreduce_sum(world, step_b * args.steps) / (total_ms / 1e3) / 1e9
    # the other composition of the same step, timed beside it (same bits)
    for _ in range(3):
        other_step()
    da = torch.cuda.Event(enable_timing=True)
    db = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    da.record(stream)
    for _ in range(args.steps):
        other_step()
    db.record(stream)
    torch.cuda.synchronize()
    other_ms = allreduce_max(world, da.elapsed_time(db) / args.steps)
    other_kernel = ss.last_kernel()
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_plain(torch, stream, [g for gs in grads for g in gs], params,
                         lambda: one_step(None), step_b, world, args.e2e_steps,
                         "the 8 ranks' full bf16 gradients of the 9 parameters in, the 9 "
                         "gathered bf16 parameters out")
    cpu = None
    if rank == 0 and not args.no_cpu:
        cv, sec, n_el = _fsdp2_oracle(2, 0, not direct)
        cpu = {"value": round(cv, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"2 x (chunk-cat, 8 fused updates and the copy-out) of the layer group "
                         f"with dimension 0 divided by 16 ({n_el} elements), numpy "
                         f"single-threaded"}
    if rank == 0:
        steps_text = {
            True: "8 x the rank's step read straight from the ranks' per-parameter gradients "
                  "(Fsdp2Step: one launch over its 9 parameters, no chunk-cat copy), all-gather "
                  "copy-out into the 9 full parameters",
            False: "8 x chunk-cat of a rank's full bf16 gradients, 8 x fused step on the padded "
                   "local buffers, all-gather copy-out into the 9 full parameters"}
        kernels = {"fused_ms_per_launch": round(avg[1] / nd, 4),
                   "fused_gbs": round(achieved, 1),
                   "copy_out_ms": round(avg[2], 4),
                   "copy_out_gbs": round(ag_b / (avg[2] / 1e3) / 1e9, 1)}
        if not direct:
            kernels = {"chunk_cat_ms": round(avg[0], 4),
                       "chunk_cat_gbs": round(cc_b / (avg[0] / 1e3) / 1e9, 1), **kernels}
        kernels["with_chunk_cat" if direct else "without_chunk_cat"] = {
            "step": steps_text[not direct], "ms": round(other_ms, 4),
            "gbs": round(other_b / (other_ms / 1e3) / 1e9, 1), "bytes": other_b,
            "time_vs_this_line": round(other_ms / (total_ms / args.steps), 4),
            "kernel": other_kernel, "note": "the same bits as the line's step"}
        print(json.dumps({
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
            "config": {"workload": FSDP2_WORKLOAD + (f"_shrunk{args.shrink}x"
                                                     if args.shrink > 1 else "") +
                                    (f"_nd{nd}" if args.nd else ""),
                       "tma_stages": _stages_name(args),
                       "group": "one Llama-7B layer (9 parameters, "
                       "202,383,360 elements)", "nd": nd, "local_elements": L,
                       "step": steps_text[direct], "bytes_per_step": step_b,
                       "l2": f"no flush: each step streams {step_b / 1e9:.1f} GB vs a 129 MB L2"},
            "kernels": kernels,
            "roofline": _roofline(achieved, f"{fused_kernel}, one rank's local buffer",
                                  fused_launch,
                                  _traffic(FSDP2_WORKLOAD, L, args) if direct else None),
            "e2e": e2e, "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu,
        }))


# ------------------------------------------------------- ragged pack / gather

RAGGED_WORKLOAD = "llama_7b_layer_ragged_nd8"


def _ragged_unit(shrink=1):
    """The Llama-7B layer unit's 9 tensors, each one element longer, so that
    every tensor after the first starts at an odd element offset of the
    FlatParameter and the 8 shard slots sit 4 bytes off 16-byte boundaries
    (shrink > 1: every tensor's length divided by it first, for a smaller
    case of the same copies)."""
    from synth import workloads as W
    w = W.llama_7b_rank_view()
    shapes = w.units[w.extra["ag_unit"]]
    return w, [math.prod(sh) // shrink + 1 for sh in shapes]


def _ragged_oracle(numels, nd, scale, step):
    """The oracle's pack and all-gather on a unit scaled down by `scale`;
    returns (seconds, algorithmic bytes)."""
    import numpy as np
    import oracle
    import synth
    small = [max(1, n // scale) | 1 for n in numels]
    tensors = [synth.host_fill(synth.normal_stream(17, (93, step, k), 0.02), 0, n, "bf16")
               for k, n in enumerate(small)]
    t0 = time.perf_counter()
    flat, lay = oracle.flat_pack(tensors, nd)
    shards = [oracle.shard_of(flat, lay, q) for q in range(nd)]
    oracle.ag_unpack(shards, lay)
    dt = time.perf_counter() - t0
    return dt, 4 * sum(small) + 4 * lay.padded


def run_ragged(args):
    import torch
    world, rank, local = dist_env()
    init_dist(world)
    nd = 8
    w, numels = _ragged_unit(args.shrink)
    if args.impl == "reference":
        if rank == 0:
            tt, tb = 0.0, 0
            for k in range(args.warmup + args.steps):
                dt, b = _ragged_oracle(numels, nd, 64, k)
                if k >= args.warmup:
                    tt, tb = tt + dt, tb + b
            v = tb / tt / 1e9
            print(json.dumps({
                "impl": "reference", "metric": RAGGED_METRIC, "value": round(v, 4),
                "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(tt / args.steps * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": RAGGED_WORKLOAD, "nd": nd, "sample": "unit / 64"},
                "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1,
                                 "kind": "oracle",
                                 "sample": "each step: pack + all-gather of the unit scaled "
                                           "down 64x, numpy single-threaded"},
                "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}))
        _finish_dist(world)
        return
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    import synth
    dev = torch.device("cuda", local)
    tensors = []
    for k, n in enumerate(numels):
        t = torch.empty(n, dtype=torch.bfloat16, device=dev)
        synth.dev_fill(synth.normal_stream(17, (93, 0, k), 0.02), t)
        tensors.append(t)
    lay = ss.fsdp_layout(numels, nd)
    flat = torch.empty(lay.padded, dtype=torch.bfloat16, device=dev)
    S = lay.shard
    shards = [torch.empty(S, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    for q in range(nd):
        synth.dev_fill(synth.normal_stream(17, (94, q), 0.02), shards[q])
    full = torch.empty(nd * S, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    pack_bytes = 4 * lay.total + 2 * (lay.padded - lay.total)   # zero pad written only
    ag_bytes = 4 * nd * S
    step_bytes = pack_bytes + ag_bytes

    def one_step(ev):
        if ev is not None:
            ev[0].record(stream)
        ss.fsdp_flat_pack(tensors, nd, flat=flat)
        if ev is not None:
            ev[1].record(stream)
        ss.fsdp_ag_unpack(shards, full)
        if ev is not None:
            ev[2].record(stream)

    total_ms, events, clk, launches = _timed_loop(torch, stream, args, one_step, 3, world)
    pack_ms, ag_ms = _avg_ms(events, 0, 1), _avg_ms(events, 1, 2)
    ms = total_ms / args.steps
    all_bytes = allreduce_sum(world, step_bytes)
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_plain(torch, stream, tensors + shards, [flat, full], lambda: one_step(None),
                         step_bytes, world, args.e2e_steps, "the unit's 9 bf16 tensors and the "
                         "8 shards in, the packed unit and the gathered unit out")
    if rank != 0:
        _finish_dist(world)
        return
    pack_gbs = pack_bytes / (pack_ms / 1e3) / 1e9
    ag_gbs = ag_bytes / (ag_ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu:
        tt, tb, reps = 0.0, 0, 0
        while tt < args.cpu_seconds and reps < 20:
            dt, b = _ragged_oracle(numels, nd, 64, reps)
            tt, tb, reps = tt + dt, tb + b, reps + 1
        cpu = {"value": round(tb / tt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} x pack + all-gather of the unit scaled down 64x, numpy "
                         f"single-threaded"}
    offs = sorted({(o * 2) % 16 for o in lay.offsets} | {(q * S * 2) % 16 for q in range(nd)})
    print(json.dumps({
        "metric": RAGGED_METRIC,
        "value": round(all_bytes / (ms / 1e3) / 1e9, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
        "config": {"workload": RAGGED_WORKLOAD + (f"_shrunk{args.shrink}x" if args.shrink > 1
                                                  else ""),
                   "tma_stages": _stages_name(args), "nd": nd,
                   "tensors": len(numels), "elements": lay.total, "padded": lay.padded,
                   "shard": S, "byte_offsets_mod_16": offs,
                   "step": "flat_pack of the 9 tensors (1 call), all-gather of the 8 shards "
                           "(1 call)",
                   "bytes_per_step": step_bytes,
                   "l2": f"no flush: each step streams {step_bytes / 1e9:.2f} GB vs a 129 MB L2"},
        "kernels": {"flat_pack_ms": round(pack_ms, 4), "flat_pack_gbs": round(pack_gbs, 1),
                    "ag_ms": round(ag_ms, 4), "ag_gbs": round(ag_gbs, 1)},
        "roofline": _roofline(pack_gbs, "flat_pack: copy16_shift for the tensors at odd "
                              "offsets, copy16 for the congruent ones, copy_segments for "
                              "heads, tails and the zero pad", pack_bytes,
                              _traffic(RAGGED_WORKLOAD, lay.total, args)),
        "e2e": e2e,
        "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu}))
    _finish_dist(world)


def _fsdp2_oracle(steps, warmup=0, with_chunk_cat=False):
    """The oracle's FSDP2 group step (chunk-cat of every rank's gradients,
    the fused update of every rank's local buffer, all-gather copy-out) on
    the Llama-7B layer group with every dimension 0 divided by 16, numpy on
    one core, timed over ``steps`` steps after ``warmup``.  Returns (GB/s of
    the step's algorithmic bytes, seconds per step, elements); the bytes are
    the bench line's: the chunk-cat's only when the line times it."""
    import numpy as np
    import oracle
    import synth
    from oracle.numerics import AdamWConfig
    from synth import workloads as W
    w = W.llama_7b_rank_view()
    shapes = [(max(1, sh[0] // 16),) + tuple(sh[1:]) for sh in w.units[0]]
    nd = w.nd
    lay = oracle.fsdp2_layout(shapes, nd)
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    n = sum(math.prod(sh) for sh in shapes)
    grads = [[synth.host_fill(synth.normal_stream(19, (86, q, k), 1e-3), 0, math.prod(sh),
                              "bf16").reshape(sh) for k, sh in enumerate(shapes)]
             for q in range(nd)]
    master = oracle.chunk_cat([synth.host_fill(synth.normal_stream(19, (85, k), 0.02), 0,
                                               math.prod(sh), "f32").reshape(sh)
                               for k, sh in enumerate(shapes)], lay)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    L = lay.local
    cc_b, fused_b, ag_b = _fsdp2_bytes(shapes, nd, L)
    tt = 0.0
    for k in range(warmup + steps):
        t0 = time.perf_counter()
        rs_in = [oracle.chunk_cat(grads[q], lay) for q in range(nd)]
        outs = []
        for r in range(nd):
            sl = slice(r * L, (r + 1) * L)
            p1, m1, v1, o1 = oracle.fsdp_shard_step([x for x in rs_in], r, L, master[sl],
                                                    m[sl], v[sl], hp, k + 1)
            master[sl], m[sl], v[sl] = p1, m1, v1
            outs.append(o1)
        oracle.all_gather_copy_out(outs, lay)
        if k >= warmup:
            tt += time.perf_counter() - t0
    step_b = fused_b + ag_b + (cc_b if with_chunk_cat else 0)
    return step_b * steps / tt / 1e9, tt / steps, n


def run_fsdp2_reference(args):
    """The oracle arm of the FSDP2 line (``_fsdp2_oracle``); rank 0 alone
    under torchrun."""
    world, rank, _ = dist_env()
    init_dist(world)
    if rank == 0:
        nd = 8
        val, sec, n = _fsdp2_oracle(args.steps, args.warmup, args.fsdp2_chunk_cat)
        tt = sec * args.steps
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": FSDP2_WORKLOAD, "nd": nd,
                       "sample": f"the layer group with dimension 0 divided by 16 ({n} elements)"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "each step: chunk-cat, 8 fused updates and the copy-out "
                                       "of the scaled-down group, numpy single-threaded"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
    _finish_dist(world)


# ------------------------------------------------------------ checkpoint

CKPT_WORKLOAD = "ckpt_gpt2_small_nd8_to_nd4"


def _ckpt_oracle(steps, warmup=0):
    """The checkpoint with numpy on the host: the 8 ranks' fp32 master / m / v
    shards of every GPT-2-small unit written with numpy.save, then the 4 new
    ranks' shards read back and resharded by the oracle; median seconds of
    ``steps`` rounds after ``warmup``.  Returns (save s, load s, state bytes)."""
    import shutil
    import numpy as np
    import synth
    from oracle import checkpoint as oracle_ckpt
    from synth import workloads as W
    w = W.gpt2_small()
    totals = [sum(math.prod(sh) for sh in u) for u in w.units]
    old_nd, new_nd = 8, 4
    shards = {}                     # (rank, unit, kind) -> fp32 array
    for u, T in enumerate(totals):
        S = -(-T // old_nd)
        for kind in range(3):
            flat = np.zeros(S * old_nd, np.float32)
            flat[:T] = synth.host_fill(synth.normal_stream(23, (84, u, kind), 0.02), 0, T, "f32")
            for r in range(old_nd):
                shards[(r, u, kind)] = flat[r * S:(r + 1) * S].copy()
    state_bytes = sum(a.nbytes for a in shards.values())
    root = tempfile.mkdtemp(prefix="shst_ckref_")
    saves, loads = [], []
    try:
        for k in range(warmup + max(1, steps)):
            d = os.path.join(root, f"step{k}")
            os.makedirs(d)
            t0 = time.perf_counter()
            for (r, u, kind), a in shards.items():
                np.save(os.path.join(d, f"{r}_{u}_{kind}.npy"), a)
            t1 = time.perf_counter()
            for u, T in enumerate(totals):
                for kind in range(3):
                    old = [np.load(os.path.join(d, f"{r}_{u}_{kind}.npy"))
                           for r in range(old_nd)]
                    for nr in range(new_nd):
                        oracle_ckpt.reshard(old, T, new_nd, nr)
            t2 = time.perf_counter()
            if k >= warmup:
                saves.append(t1 - t0)
                loads.append(t2 - t1)
            shutil.rmtree(d, ignore_errors=True)
    finally:
        shutil.rmtree(root, ignore_errors=True)
    return statistics.median(saves), statistics.median(loads), state_bytes


def run_ckpt_reference(args):
    """The oracle arm of the checkpoint line (``_ckpt_oracle``); rank 0 alone."""
    world, rank, _ = dist_env()
    init_dist(world)
    if rank == 0:
        old_nd, new_nd = 8, 4
        sv, ld, state_bytes = _ckpt_oracle(args.steps, args.warmup)
        val = state_bytes / sv / 1e9
        print(json.dumps({
            "impl": "reference",
            "metric": "sharded checkpoint save / load GB/s (fp32 master + moments)",
            "value": round(val, 3), "unit": "GB/s", "n_gpus": world, "steps": max(1, args.steps),
            "warmup": args.warmup, "ms_per_step": round(1e3 * (sv + ld), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": CKPT_WORKLOAD, "old_nd": old_nd, "new_nd": new_nd,
                       "state_bytes": state_bytes, "load_gbs": round(state_bytes / ld / 1e9, 3)},
            "cpu_baseline": {"value": round(val, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "the whole GPT-2-small optimizer state: numpy.save per "
                                       "rank, unit and kind, then numpy.load + the oracle's "
                                       "reshard for the 4 new ranks"},
            "e2e": {"value": round(val, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
    _finish_dist(world)


def run_ckpt(args):
    """Sharded checkpoint of the GPT-2-small-shaped model: every one of 8
    ranks saves its fp32 master / m / v shards (device -> pinned host -> its
    own file, ranks in parallel), then 4 ranks of a new layout load their
    resharded state (pieces of the saved files -> pinned host -> device)."""
    import shutil
    import torch
    world, rank, local = dist_env()
    if rank != 0:
        return                          # host-IO line: one process
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    from sharded_optimizer_step_gb300 import checkpoint as ck
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    from synth import workloads as W
    w = W.gpt2_small()
    hp = ss.AdamW()
    old = [RankShardOptimizer(w.units, 8, r, hp, device="cuda:0") for r in range(8)]
    for o in old:
        fill_rank_view(o, o.master, w.master_stream)
        for q in range(8):
            fill_rank_view(o, o.grad_in[q], lambda u, k, q=q: w.grad_stream(1, q, 0, u, k))
        o.step()
    new = [RankShardOptimizer(w.units, 4, r, hp, device="cuda:0") for r in range(4)]
    torch.cuda.synchronize()
    state_bytes = sum(3 * 4 * o.shard_total for o in old)
    root = tempfile.mkdtemp(prefix="shst_ckpt_")
    saves, loads = [], []
    try:
        # every save goes to a new directory (as a training run's periodic
        # checkpoints do); the previous one is removed outside the timing.
        # The first save and load also pin each optimizer's host staging.
        prev = None
        first = None
        for k in range(max(1, args.steps) + 1):
            directory = os.path.join(root, f"step{k}")
            t0 = time.perf_counter()
            ck.save(directory, old)
            t1 = time.perf_counter()
            ck.load(directory, new)
            t2 = time.perf_counter()
            if k == 0:
                first = (t1 - t0, t2 - t1)
            else:
                saves.append(t1 - t0)
                loads.append(t2 - t1)
            if prev is not None:
                shutil.rmtree(prev, ignore_errors=True)
            prev = directory
        disk = sum(os.path.getsize(ck.rank_file(prev, r)) for r in range(8))
    finally:
        shutil.rmtree(root, ignore_errors=True)
    sv, ld = statistics.median(saves), statistics.median(loads)
    cpu = None
    if not args.no_cpu:
        csv, cld, cbytes = _ckpt_oracle(1)
        cpu = {"value": round(cbytes / csv / 1e9, 3), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "load_gbs": round(cbytes / cld / 1e9, 3),
               "sample": "the whole optimizer state once: numpy.save per rank, unit and kind, "
                         "then numpy.load + the oracle's reshard for the 4 new ranks"}
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
        "first_save_s": round(first[0], 3), "first_load_s": round(first[1], 3),
        "staging": "pinned host buffers per optimizer, pinned by the first save / load "
                   "(untimed, reported as first_*) and reused",
        "roofline": None,
        "e2e": {"value": round(state_bytes / sv / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": state_bytes, "d2h_bytes_per_step": state_bytes,
                "note": "the line is itself end to end: the save copies the device state out "
                        "and writes the files, the load reads them and copies the new ranks' "
                        "state in, through the public checkpoint calls, timed on the host"},
        "gpu_launches": 0, "clocks": None, "cpu_baseline": cpu,
        "note": "host-IO bound (device <-> pinned host copies and file reads / writes); "
                "no GPU kernel runs"}))


# ------------------------------------------- micro-batch accumulation (fp32)

ACCUM_WORKLOAD = "llama_1b_rank0_nd8_m4"


def _timed_loop(torch, stream, args, one_step, n_events, world=1):
    """Warm-up, then args.steps timed steps with n_events CUDA events each,
    bracketed by a barrier and a device synchronize on both sides; returns
    (total ms, max over ranks; per-step event lists; clocks; launches)."""
    import sharded_optimizer_step_gb300 as ss
    clocks = ClockSampler(smi_index(torch.cuda.current_device()))
    clocks.start()
    for _ in range(args.warmup):
        one_step(None)
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)]
              for _ in range(args.steps)]
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
    return allreduce_max(world, a.elapsed_time(b)), events, clk, launches


def _avg_ms(events, i, j):
    return sum(e[i].elapsed_time(e[j]) for e in events) / len(events)


def _traffic(workload_name, elements, args):
    """ncu DRAM bytes of one launch of the line's dominant kernel, scaled from
    the profile's bytes per element (None for smaller cases, other kernel
    choices or a kernel changed since the capture)."""
    per = profiled_traffic(workload_name)
    if (per is None or args.layers or args.nd or args.kernel_path != "auto" or args.tma_stages
            or getattr(args, "shrink", 1) > 1):
        return None
    return round(per * elements)


# GB300 HBM3e nominal bandwidth (8 stacks, NVIDIA's published 7.9 TB/s per
# GPU).  The roofline's `peak` is the measured copy bandwidth instead, so
# `frac` can read a little above 1 for a read-heavy kernel; `frac_of_nominal`
# puts the same bytes against the nominal figure.
HBM_NOMINAL_GBS = 7900.0


def _roofline(achieved, kernel, bytes_per_launch, traffic=None):
    peak, kind = measured_peak()
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "frac_of": ("the measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs: b.copy_ of "
                        "1 Gi bf16, read + write bytes, burst)" if kind == "measured"
                        else "the fallback 6800 GB/s"),
            "peak_source": ("measured: MEASURED_PEAKS.json hbm_gbs (copy, burst)"
                            if kind == "measured" else "fallback 6800 GB/s"),
            "frac_of_nominal": round(achieved / HBM_NOMINAL_GBS, 4),
            "nominal_gbs": HBM_NOMINAL_GBS,
            "nominal_source": "GB300 HBM3e nominal 7.9 TB/s (NVIDIA specification)",
            "kernel": kernel, "algorithmic_bytes_per_launch": bytes_per_launch,
            "traffic": traffic}


def _accum_oracle_sample(w, n, t):
    """Oracle time of a contiguous sample of n shard elements of one rank's
    view: M micro-batch accumulations of the N_d contributions, then the
    fused step on the fp32 accumulators."""
    import numpy as np
    import oracle
    from oracle.numerics import AdamWConfig
    idx = np.arange(1_000_000, 1_000_000 + n, dtype=np.int64)
    micro = [[oracle_rank_values(w, 0, idx, lambda u, k, q=q, j=j: w.grad_stream(1, q, j, u, k),
                                 "bf16") for j in range(w.micro)] for q in range(w.nd)]
    p = oracle_rank_values(w, 0, idx, w.master_stream, "f32")
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    t0 = time.perf_counter()
    accs = [oracle.grad_accumulate(micro[q], np.float32(1.0 / w.micro)) for q in range(w.nd)]
    oracle.fsdp_shard_step(accs, 0, n, p, m, v, hp, t)
    dt = time.perf_counter() - t0
    acc_b, fused_b = _accum_bytes(w.nd, w.micro, True)
    return dt, (acc_b + fused_b) * n


def _accum_bytes(nd, M, fused_last):
    """Algorithmic bytes per shard element of the accumulation (all launches
    over the nd contributions) and of the fused step.  Each micro-batch
    accumulate reads bf16 and writes fp32 (6 B), after the first also reads
    fp32 (10 B).  fused_last: the last micro-batch is accumulated inside the
    fused step, which reads per contribution the fp32 accumulator and the
    bf16 gradient (6 B) and no accumulator is written for it."""
    if fused_last:
        return (6 + 10 * (M - 2)) * nd, 6 * nd + 26
    return (6 + 10 * (M - 1)) * nd, 4 * nd + 26


def run_accum(args):
    """One rank's view of the Llama-style 1B model (17 units, N_d = 8) with
    M = 4 micro-batches: every one of the 8 contributions to this rank's
    shard is accumulated in fp32 over the bf16 micro-batch gradients
    (acc = g*(1/M), then acc += g*(1/M); one launch per micro-batch over the
    8 contributions side by side).  By default micro-batches 0..M-2 are
    accumulated so and the last one is added inside the fused step, which
    reads the 8 fp32 accumulators and the 8 last bf16 gradients; with
    --accum-two-pass all M are accumulated and the fused step reads the
    accumulators only.  Then one layer unit is all-gathered.  The
    accumulate work per step equals a real rank's (N_d shard slices = one
    full gradient)."""
    world, rank, local = dist_env()
    if args.impl == "reference":
        return _accum_reference(args) if rank == 0 else None
    init_dist(world)
    import torch
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    import synth
    from sharded_optimizer_step_gb300.engine import RankShardOptimizer
    from synth import workloads as W
    w = W.llama_1b()
    if args.layers:
        w.units = w.units[:args.layers]      # smaller case: the first N layer units
    nd, M = w.nd, w.micro
    r = rank % nd                       # GPU k holds rank k mod N_d's view of its own replica
    dev = torch.device("cuda", local)
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    opt = RankShardOptimizer(w.units, nd, r, hp, device=dev, grad_dtype=torch.float32)
    S = opt.shard_total
    acc = torch.empty(nd * S, dtype=torch.float32, device=dev)
    opt.grad_in = [acc[q * S:(q + 1) * S] for q in range(nd)]
    micro = [torch.empty(nd * S, dtype=torch.bfloat16, device=dev) for _ in range(M)]
    for j in range(M):
        for q in range(nd):
            fill_rank_view(opt, micro[j][q * S:(q + 1) * S],
                           lambda u, k, q=q, j=j: w.grad_stream(1, q, j, u, k))
    fill_rank_view(opt, opt.master, w.master_stream)
    u = 0
    Su, Pu = opt.layouts[u].shard, opt.layouts[u].padded
    peers = [torch.empty(Su, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    for q in range(1, nd):
        synth.dev_fill(w.peer_shard_stream(1, q, u), peers[q])
    full = torch.empty(Pu, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    inv_m = float(1.0 / M)
    fused_last = not args.accum_two_pass
    n_acc = M - 1 if fused_last else M        # accumulate launches per step
    acc_b, fused_b = _accum_bytes(nd, M, fused_last)
    acc_bytes, fused_bytes = acc_b * S, fused_b * S
    ag_bytes = 4 * Pu
    step_bytes = acc_bytes + fused_bytes + ag_bytes
    kernel_names = {}
    last = [micro[M - 1][q * S:(q + 1) * S] for q in range(nd)]

    def one_step(ev):
        if ev is not None:
            ev[0].record(stream)
        for j in range(n_acc):
            ss.fsdp_grad_accumulate(micro[j], acc, inv_m, j == 0, stream=stream)
        kernel_names["accumulate"] = ss.last_kernel()
        if ev is not None:
            ev[1].record(stream)
        if fused_last:
            opt.step_with_last_micro_batch(last, inv_m, stream=stream)
        else:
            opt.step(stream=stream)
        kernel_names["fused"] = ss.last_kernel()
        if ev is not None:
            ev[2].record(stream)
        opt.gather_unit(u, peers, full, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    graph_launches = 0
    if args.graph:
        if not fused_last:
            raise SystemExit("--graph: the accumulation line with the fused last micro-batch")
        # the step count on the device; the accumulate launches, the update
        # (advance + fused launch) and the all-gather each captured once,
        # after an eager warm-up
        opt.device_step_state()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for j in range(n_acc):
                ss.fsdp_grad_accumulate(micro[j], acc, inv_m, j == 0)
            opt.step_with_last_micro_batch_on_device(last, inv_m)
            opt.gather_unit(u, peers, full)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g_acc, g_update, g_gather = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                     torch.cuda.CUDAGraph())
        l0 = ss.launch_count()
        with torch.cuda.graph(g_acc):
            for j in range(n_acc):
                ss.fsdp_grad_accumulate(micro[j], acc, inv_m, j == 0)
        kernel_names["accumulate"] = ss.last_kernel()
        with torch.cuda.graph(g_update):
            opt.step_with_last_micro_batch_on_device(last, inv_m)
        kernel_names["fused"] = ss.last_kernel()
        with torch.cuda.graph(g_gather):
            opt.gather_unit(u, peers, full)
        graph_launches = ss.launch_count() - l0     # kernels per replayed step

        def one_step(ev):                 # noqa: F811 -- the graph form of the step
            if ev is not None:
                ev[0].record(stream)
            g_acc.replay()
            if ev is not None:
                ev[1].record(stream)
            g_update.replay()
            if ev is not None:
                ev[2].record(stream)
            g_gather.replay()
            if ev is not None:
                ev[3].record(stream)

    total_ms, events, clk, launches = _timed_loop(torch, stream, args, one_step, 4, world)
    if args.graph:
        launches = graph_launches * args.steps
    acc_ms, fused_ms, ag_ms = _avg_ms(events, 0, 1), _avg_ms(events, 1, 2), _avg_ms(events, 2, 3)
    ms = total_ms / args.steps
    all_bytes = allreduce_sum(world, step_bytes)
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_plain(torch, stream, micro, [full], lambda: one_step(None), step_bytes, world,
                         args.e2e_steps, f"the {M} micro-batches' bf16 gradients of the {nd} "
                         f"contributions in, the gathered layer unit out")
    if rank != 0:
        _finish_dist(world)
        return
    acc_gbs = acc_bytes / (acc_ms / 1e3) / 1e9
    fused_gbs = fused_bytes / (fused_ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu:
        n, tt, tb, reps = 1_000_000, 0.0, 0, 0
        while tt < args.cpu_seconds and reps < 20:
            dt, b = _accum_oracle_sample(w, n, reps + 1)
            tt, tb, reps = tt + dt, tb + b, reps + 1
        cpu = {"value": round(tb / tt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} x (accumulate 4 micro-batches of 8 contributions + fused "
                         f"step) on {n} contiguous shard elements, numpy single-threaded"}
    print(json.dumps({
        "metric": "micro-batch accumulate + fused fp32-accumulator step HBM GB/s, "
                  "Llama-1B rank view, N_d=8, M=4",
        "value": round(all_bytes / (ms / 1e3) / 1e9, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
        "config": {"workload": ACCUM_WORKLOAD + (f"_first{args.layers}layers" if args.layers
                                                 else ""),
                   "tma_stages": _stages_name(args), "graph": bool(args.graph),
                   "model_shape": f"Llama-style 1B, {len(w.units)} FSDP units",
                   "psi": w.psi, "nd": nd, "micro_batches": M, "rank": r, "shard_elements": S,
                   "grad_dtype": "bf16 micro-batch gradients, fp32 accumulators",
                   "step": (f"{n_acc} accumulate launches over the {nd} contributions (first "
                            "writes, then read-add-write), "
                            + ("the last micro-batch accumulated inside the fused rs_avg+AdamW+"
                               "bf16 cast launch (reads the fp32 accumulators and the bf16 "
                               "gradients)" if fused_last else
                               "fused rs_avg+AdamW+bf16 cast on the fp32 accumulators (1 "
                               "launch)")
                            + ", all-gather of one layer unit (1 launch)"),
                   "bytes_per_step": step_bytes,
                   "l2": f"no flush: each step streams {step_bytes / 1e9:.1f} GB vs a 129 MB L2"},
        "params_per_s": round(S * world / (ms / 1e3), 1),
        "kernels": {"accumulate_ms": round(acc_ms, 4), "accumulate_gbs": round(acc_gbs, 1),
                    "fused_kernel": kernel_names["fused"],
                    "fused_ms": round(fused_ms, 4), "fused_gbs": round(fused_gbs, 1),
                    "fused_frac": round(fused_gbs / measured_peak()[0], 4),
                    "ag_ms": round(ag_ms, 4),
                    "ag_gbs": round(ag_bytes / (ag_ms / 1e3) / 1e9, 1)},
        "roofline": _roofline(acc_gbs, f"{kernel_names['accumulate']} "
                                       f"({n_acc} launches over {nd} x {S} elements)",
                              acc_bytes // n_acc, _traffic(ACCUM_WORKLOAD, nd * S, args)
                              if fused_last else None),
        "e2e": e2e,
        "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu}))
    _finish_dist(world)


def _finish_dist(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _accum_reference(args):
    from synth import workloads as W
    w = W.llama_1b()
    n = 500_000
    for k in range(args.warmup):
        _accum_oracle_sample(w, n, k + 1)
    ts, bs = [], []
    for k in range(args.steps):
        dt, b = _accum_oracle_sample(w, n, args.warmup + k + 1)
        ts.append(dt)
        bs.append(b)
    value = round(sum(bs) / sum(ts) / 1e9, 4)
    print(json.dumps({
        "impl": "reference", "metric": "micro-batch accumulate + fused fp32-accumulator step "
                                       "HBM GB/s, Llama-1B rank view, N_d=8, M=4",
        "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * sum(ts) / len(ts), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": ACCUM_WORKLOAD, "sample_elements_per_step": n},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {n} contiguous shard elements"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


# ------------------------------------------------- DDP buckets + full AdamW

DDP_WORKLOAD = "ddp_nd8_buckets"


def _ddp_oracle_sample(w, numels, n_params, t):
    """Oracle time of the DDP step on the first n_params parameters (whole
    parameters, one bucket each at the default cap's plan order)."""
    import numpy as np
    import oracle
    import synth
    from oracle.numerics import AdamWConfig
    sel = numels[:n_params]
    total = sum(sel)
    grads = [np.concatenate([synth.host_fill(w.grad_stream(1, q, 0, 0, i), 0, n, "bf16")
                             for i, n in enumerate(sel)]) for q in range(w.nd)]
    p = np.concatenate([synth.host_fill(w.master_stream(0, i), 0, n, "f32")
                        for i, n in enumerate(sel)])
    z = np.zeros(total, np.float32)
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    bounds = [0]
    for n in sel:
        bounds.append(bounds[-1] + n)
    t0 = time.perf_counter()
    oracle.ddp_step(grads, bounds, p, z, z.copy(), hp, t)
    return time.perf_counter() - t0, (2 * w.nd + 2) * total + 28 * total, total


def run_ddp(args):
    """Replicated DDP on 8 emulated ranks: 80 blocks' worth of parameters
    (Psi = 351,035,392 bf16) bucketed in reverse registration order at a
    25 MiB cap; each bucket's 8 rank gradients are averaged (fp32 sum in rank
    order, bf16 out; one launch per bucket), then one full AdamW + bf16 cast
    over all Psi parameters.  The caps 1, 4, 64 and 256 MiB are timed too
    (all-reduce only)."""
    from synth import workloads as W
    w = W.ddp_sweep()
    if args.nd:
        w.nd = args.nd
    numels = w.unit_numels(0)
    if args.layers:
        numels = numels[:5 * args.layers]    # smaller case: the first N blocks' parameters
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return
        n_params = 4
        ts, bs = [], []
        for k in range(args.warmup + args.steps):
            dt, b, total = _ddp_oracle_sample(w, numels, n_params, k + 1)
            if k >= args.warmup:
                ts.append(dt)
                bs.append(b)
        value = round(sum(bs) / sum(ts) / 1e9, 4)
        print(json.dumps({
            "impl": "reference", "metric": "DDP bucket all-reduce avg + full AdamW HBM GB/s, "
                                           "Psi=351M, N_d=8, 25 MiB buckets",
            "value": value, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * sum(ts) / len(ts), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": DDP_WORKLOAD,
                                            "sample_params": n_params, "sample_elements": total},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"the first {n_params} parameters ({total} elements)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return
    init_dist(world)
    import torch
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    import synth
    nd = w.nd
    total = sum(numels)
    dev = torch.device("cuda", local)
    grads = [torch.empty(total, dtype=torch.bfloat16, device=dev) for _ in range(nd)]
    hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    plans = {}
    for mib in w.extra["caps_mib"]:
        plans[mib] = ss.ddp_bucket_plan(numels, 2, mib << 20)
    off, _, boff = plans[25]
    for q in range(nd):
        for i, n in enumerate(numels):
            synth.dev_fill(w.grad_stream(1, q, 0, 0, i), grads[q][off[i]:off[i] + n])
    out = torch.empty(total, dtype=torch.bfloat16, device=dev)
    master = torch.empty(total, dtype=torch.float32, device=dev)
    for i, n in enumerate(numels):
        synth.dev_fill(w.master_stream(0, i), master[off[i]:off[i] + n])
    mm = torch.zeros(total, device=dev)
    vv = torch.zeros(total, device=dev)
    pb = torch.empty(total, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    ar_bytes = (2 * nd + 2) * total
    adam_bytes = 28 * total
    step_bytes = ar_bytes + adam_bytes
    t = [0]
    kernel_names = {}

    def one_step(ev):
        if ev is not None:
            ev[0].record(stream)
        ss.ddp_bucket_allreduce_avg(grads, boff, out, stream=stream)
        kernel_names["allreduce"] = ss.last_kernel()
        if ev is not None:
            ev[1].record(stream)
        t[0] += 1
        ss.fsdp_rs_avg_adamw_cast([out], master, mm, vv, pb, hp, t[0], stream=stream)
        kernel_names["adamw"] = ss.last_kernel()
        if ev is not None:
            ev[2].record(stream)

    total_ms, events, clk, launches = _timed_loop(torch, stream, args, one_step, 3, world)
    ar_ms, adam_ms = _avg_ms(events, 0, 1), _avg_ms(events, 1, 2)
    ms = total_ms / args.steps
    all_bytes = allreduce_sum(world, step_bytes)
    # the other caps: all-reduce only, same gradients (the values per bucket
    # differ in placement, not in amount of work)
    by_cap = {}
    for mib, (_, _, bo) in plans.items():
        for _ in range(3):
            ss.ddp_bucket_allreduce_avg(grads, bo, out, stream=stream)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record(stream)
        for _ in range(reps):
            ss.ddp_bucket_allreduce_avg(grads, bo, out, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        cap_ms = a.elapsed_time(b) / reps
        by_cap[f"{mib}MiB"] = {"buckets": len(bo) - 1, "ms": round(cap_ms, 4),
                               "gbs": round(ar_bytes / (cap_ms / 1e3) / 1e9, 1)}
    # the same step fused: the all-reduce of all buckets and the replicated
    # AdamW + cast in one launch (ddp_bucket_allreduce_avg_adamw_cast), with
    # and without the averaged gradient kept; back to back, same gradients
    fused = {}
    for keep in (False, True):
        def fused_call():
            t[0] += 1
            ss.ddp_bucket_allreduce_avg_adamw_cast(grads, boff, master, mm, vv, pb, hp, t[0],
                                                   mean_out=out if keep else None,
                                                   stream=stream)
        for _ in range(3):
            fused_call()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fused_call()
        b.record(stream)
        torch.cuda.synchronize()
        f_ms = allreduce_max(world, a.elapsed_time(b) / args.steps)
        f_bytes = (2 * nd + 26 + (2 if keep else 0)) * total
        fused["keep_mean" if keep else "no_mean"] = {
            "ms": round(f_ms, 4), "gbs": round(f_bytes / (f_ms / 1e3) / 1e9, 1),
            "bytes": f_bytes, "time_vs_two_calls": round(f_ms / ms, 4),
            "kernel": ss.last_kernel()}
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_plain(torch, stream, grads, [pb], lambda: one_step(None), step_bytes, world,
                         args.e2e_steps, "the 8 ranks' bucketed bf16 gradients in, the "
                         "bf16 parameters out")
    if rank != 0:
        _finish_dist(world)
        return
    ar_gbs = ar_bytes / (ar_ms / 1e3) / 1e9
    adam_gbs = adam_bytes / (adam_ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu:
        tt, tb, reps, n_params = 0.0, 0, 0, 4
        while tt < args.cpu_seconds and reps < 20:
            dt, b, n_el = _ddp_oracle_sample(w, numels, n_params, reps + 1)
            tt, tb, reps = tt + dt, tb + b, reps + 1
        cpu = {"value": round(tb / tt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} x the DDP step on the first {n_params} parameters "
                         f"({n_el} elements), numpy single-threaded"}
    print(json.dumps({
        "metric": "DDP bucket all-reduce avg + full AdamW HBM GB/s, Psi=351M, N_d=8, "
                  "25 MiB buckets",
        "value": round(all_bytes / (ms / 1e3) / 1e9, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator on the device; no data set or weights)",
        "config": {"workload": DDP_WORKLOAD + (f"_first{args.layers}blocks" if args.layers
                                               else "") + (f"_nd{nd}" if nd != 8 else ""),
                   "tma_stages": _stages_name(args),
                   "dependent_launch": not args.no_dependent_launch,
                   "psi": total, "nd": nd, "cap_mib": 25,
                   "buckets": len(boff) - 1,
                   "step": "one all-reduce-avg launch per bucket (8 bf16 rank gradients -> "
                           "bf16 mean), then fused AdamW + bf16 cast over all parameters "
                           "(1 launch, N_d = 1)",
                   "bytes_per_step": step_bytes,
                   "l2": f"no flush: each step streams {step_bytes / 1e9:.1f} GB vs a 129 MB L2"},
        "kernels": {"allreduce_ms": round(ar_ms, 4), "allreduce_gbs": round(ar_gbs, 1),
                    "allreduce_frac": round(ar_gbs / measured_peak()[0], 4),
                    "adamw_ms": round(adam_ms, 4), "adamw_gbs": round(adam_gbs, 1),
                    "allreduce_by_cap": by_cap,
                    "fused_step": {**fused, "note": "ddp_bucket_allreduce_avg_adamw_cast over "
                                   "the 25 MiB plan's buckets in one launch: the same bits as "
                                   "the two calls timed above"}},
        "roofline_fused": _roofline(fused["no_mean"]["gbs"], fused["no_mean"]["kernel"],
                                    fused["no_mean"]["bytes"]),
        "roofline": _roofline(adam_gbs, f"{kernel_names['adamw']} at N_d = 1 (full AdamW)",
                              adam_bytes, _traffic(DDP_WORKLOAD, total, args)),
        "roofline_allreduce": _roofline(ar_gbs, f"{kernel_names['allreduce']} at N_d = {nd} "
                                                f"({len(boff) - 1} launches, one per bucket; "
                                                f"the last bucket's kernel named)", ar_bytes),
        "e2e": e2e,
        "note": "buckets after the first of the call are launched as programmatic dependents "
                "of the previous bucket's kernel" if not args.no_dependent_launch else
                "every bucket an ordinary launch",
        "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu}))
    _finish_dist(world)


def _e2e_plain(torch, stream, inputs, outputs, step_fn, step_bytes, world, steps, what):
    """End to end through the public calls with host buffers: every step
    copies the step's inputs in from pinned host memory, issues the step's
    calls and reads its outputs back, all on the compute stream, with no
    overlap.  ``inputs`` / ``outputs`` are the device tensors the step reads
    / produces; ``step_fn()`` issues the step.  Every rank takes part in the
    same reductions, whatever happened; returns the line's ``e2e`` object
    (GB/s of the step's algorithmic bytes)."""
    failed, ms, h2d, d2h = "", 0.0, 0, 0
    try:
        pairs = [(d, torch.empty(d.shape, dtype=d.dtype, pin_memory=True)) for d in inputs]
        for d, h in pairs:
            h.copy_(d)
        host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outputs]
        h2d = sum(d.numel() * d.element_size() for d in inputs)
        d2h = sum(o.numel() * o.element_size() for o in outputs)
        n = max(1, steps)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            for d, h in pairs:
                d.copy_(h, non_blocking=True)
            step_fn()
            for o, h in zip(outputs, host_out):
                h.copy_(o, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n
        del pairs, host_out
    except RuntimeError as exc:          # e.g. the host cannot pin this much memory
        failed = str(exc).splitlines()[0][:200]
        torch.cuda.synchronize()
    n_failed = allreduce_sum(world, 1.0 if failed else 0.0)
    ms = allreduce_max(world, ms)
    total = allreduce_sum(world, float(step_bytes))
    if n_failed:
        return {"value": None, "unit": "GB/s",
                "unavailable": f"end-to-end leg failed on {int(n_failed)} rank(s): "
                               f"{failed or 'another rank'}"}
    return {"value": round(total / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "path": f"{what}: pinned host inputs copied in, the step's C-ABI calls, the "
                    f"outputs read back, every step on the compute stream, no overlap"}


# ------------------------------------ small workloads: the whole job

UNIT9M_WORKLOAD = "unit_9m_nd4_m4"
GPT2_WORKLOAD = "gpt2_small_nd8"
SMALL_METRICS = {
    UNIT9M_WORKLOAD: ("whole-job step HBM GB/s: 3 micro-batch accumulations of the 4 ranks' "
                      "gradients + the 4 ranks' fused last micro-batch rs_avg+AdamW+bf16 cast "
                      "(one launch over their side-by-side shards) + all-gather, one "
                      "9.4M-param unit, N_d=4, M=4"),
    GPT2_WORKLOAD: ("whole-job step HBM GB/s: 8 rank-view fused rs_avg+AdamW+bf16 cast launches "
                    "over 13 units + all-gather of one block unit, GPT-2 small, N_d=8"),
}
L2_FLUSH_BYTES = 256 << 20          # written between timed steps: twice the 129 MB L2


class _SmallJob:
    """The whole data-parallel job of a small workload on one GPU: every
    emulated rank's step, so that launch latency and the small arrays are what
    is measured.  Inputs (gradients of every rank and micro-batch, fp32
    master) are seeded, packed / placed by the library's layout and resident
    before timing."""

    def __init__(self, name, torch, ss, dev):
        import synth
        from synth import workloads as W
        from sharded_optimizer_step_gb300.engine import RankShardOptimizer
        self.name, self.torch, self.ss, self.dev = name, torch, ss, dev
        w = self.w = W.unit_9m() if name == UNIT9M_WORKLOAD else W.gpt2_small()
        self.hp = ss.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
        nd, M = w.nd, w.micro
        bf16, f32 = torch.bfloat16, torch.float32
        if name == UNIT9M_WORKLOAD:
            shapes = w.units[0]
            lay = self.lay = ss.fsdp_layout(w.unit_numels(0), nd)
            S, P = lay.shard, lay.padded
            # micro-batch j's gradients of all N_d ranks side by side (rank q's
            # packed unit at q*P), like the accumulators: one accumulate
            # launch per micro-batch covers the whole job
            tens = [torch.empty(s, dtype=bf16, device=dev) for s in shapes]
            self.g = []
            for j in range(M):
                flat = torch.empty(nd * P, dtype=bf16, device=dev)
                for q in range(nd):
                    for t, x in enumerate(tens):
                        synth.dev_fill(w.grad_stream(1, q, j, 0, t), x.view(-1))
                    ss.fsdp_flat_pack(tens, nd, flat=flat[q * P:(q + 1) * P])
                self.g.append(flat)
            mt = [torch.empty(s, dtype=f32, device=dev) for s in shapes]
            for t, x in enumerate(mt):
                synth.dev_fill(w.master_stream(0, t), x.view(-1))
            self.master = ss.fsdp_flat_pack(mt, nd)
            self.m = torch.zeros(P, dtype=f32, device=dev)
            self.v = torch.zeros(P, dtype=f32, device=dev)
            self.acc = torch.empty(nd * P, dtype=f32, device=dev)
            # the ranks' bf16 shards side by side (rank r's at r*S), as their
            # fp32 state is: one fused launch updates every rank's shard
            self.shards = torch.empty(P, dtype=bf16, device=dev)
            self.outs = [self.shards[r * S:(r + 1) * S] for r in range(nd)]
            self.full = torch.empty(P, dtype=bf16, device=dev)
            self.S, self.P = S, P
            acc_b = nd * (6 + 10 * (M - 2)) * P
            fused_b = (6 * nd + 26) * P             # every rank's shard: P elements
            self.parts = [("accumulate", acc_b), ("fused", fused_b), ("all-gather", 4 * P)]
            self.shard_elements = P
        else:
            self.opts = [RankShardOptimizer(w.units, nd, r, self.hp, device=dev)
                         for r in range(nd)]
            for o in self.opts:
                fill_rank_view(o, o.master, w.master_stream)
                for q in range(nd):
                    fill_rank_view(o, o.grad_in[q], lambda u, k, q=q: w.grad_stream(1, q, 0, u, k))
            S = self.opts[0].shard_total
            self.u = 0
            Pu = self.opts[0].layouts[self.u].padded
            self.full = torch.empty(Pu, dtype=bf16, device=dev)
            self.S, self.P = S, Pu
            self.parts = [("fused", (2 * nd + 26) * S * nd), ("all-gather", 4 * Pu)]
            self.shard_elements = S * nd
        self.step_bytes = sum(b for _, b in self.parts)
        self.state = None
        self.t = 0

    def device_state(self):
        """Step count and AdamW scalars on the device, for graph capture: one
        state that every rank's launch reads (the ranks step in lockstep)."""
        self.state = self.ss.AdamWState(self.hp, self.t, device=self.dev)

    def run(self, ev=None, graph_form=False):
        """One step of the whole job; ev: 4 events (start, after the
        accumulation, after the fused steps, after the all-gather)."""
        ss, w = self.ss, self.w
        nd, M = w.nd, w.micro
        if ev is not None:
            ev[0].record()
        if self.name == UNIT9M_WORKLOAD:
            S, P = self.S, self.P
            inv_m = float(1.0 / M)
            for j in range(M - 1):
                ss.fsdp_grad_accumulate(self.g[j], self.acc, inv_m, j == 0)
            if ev is not None:
                ev[1].record()
            if graph_form:
                self.state.advance()
            else:
                self.t += 1
            # rank r's shard is positions r*S..(r+1)*S of the state; its N_d
            # reduce inputs are the same positions of every rank's packed
            # accumulator and last micro-batch, so one launch over P positions
            # makes every rank's fused step with the same per-element sums
            args = ([self.acc[q * P:(q + 1) * P] for q in range(nd)],
                    [self.g[M - 1][q * P:(q + 1) * P] for q in range(nd)],
                    inv_m, self.master, self.m, self.v, self.shards)
            if graph_form:
                ss.fsdp_state_accumulate_rs_avg_adamw_cast(*args, self.state)
            else:
                ss.fsdp_accumulate_rs_avg_adamw_cast(*args, self.hp, self.t)
            if ev is not None:
                ev[2].record()
            ss.fsdp_ag_unpack(self.outs, self.full)
        else:
            if ev is not None:
                ev[1].record()
            if graph_form:
                self.state.advance()
                for o in self.opts:
                    ss.fsdp_state_rs_avg_adamw_cast(o.grad_in, o.master, o.m, o.v, o.params,
                                                    self.state)
            else:
                for o in self.opts:
                    o.step()
            if ev is not None:
                ev[2].record()
            u = self.u
            peers = [o.unit_slice(o.params, u) for o in self.opts]
            self.opts[0].gather_unit(u, peers, self.full)
        if ev is not None:
            ev[3].record()

    def inputs(self):
        """The device buffers of every gradient input: what an end-to-end step
        brings in from the host."""
        return (list(self.g) if self.name == UNIT9M_WORKLOAD
                else [x for o in self.opts for x in o.grad_in])


def _small_oracle(w_name, budget_s):
    """The oracle on the host: the whole step of the 9.4M unit (all ranks'
    accumulations, fused steps, the all-gather), or a contiguous sample of
    rank 0's GPT-2 view (fused step) plus the matching all-gather share.
    Returns (GB/s of algorithmic bytes, sample description)."""
    import numpy as np
    import oracle
    import synth
    from oracle.numerics import AdamWConfig
    from synth import workloads as W
    if w_name == UNIT9M_WORKLOAD:
        w = W.unit_9m()
        nd, M = w.nd, w.micro
        numels = w.unit_numels(0)
        hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
        g = [[oracle.flat_pack([synth.host_fill(w.grad_stream(1, q, j, 0, t), 0, n, "bf16")
                                for t, n in enumerate(numels)], nd)[0] for j in range(M)]
             for q in range(nd)]
        p, lay = oracle.flat_pack([synth.host_fill(w.master_stream(0, t), 0, n, "f32")
                                   for t, n in enumerate(numels)], nd)
        S, P = lay.shard, lay.padded
        step_b = nd * (6 + 10 * (M - 2)) * P + (6 * nd + 26) * P + 4 * P
        total_t, total_b, reps = 0.0, 0, 0
        while total_t < budget_s and reps < 20:
            t0 = time.perf_counter()
            accs = [oracle.grad_accumulate(g[q], np.float32(1.0 / M)) for q in range(nd)]
            outs = []
            for r in range(nd):
                z = np.zeros(S, np.float32)
                outs.append(oracle.fsdp_shard_step(accs, r, S, p[r * S:(r + 1) * S], z, z, hp,
                                                   1)[3])
            oracle.ag_unpack(outs, lay)
            total_t += time.perf_counter() - t0
            total_b += step_b
            reps += 1
        return total_b / total_t / 1e9, (f"{reps} x the whole step (4 ranks' accumulations of 4 "
                                         f"micro-batches, 4 fused steps, the all-gather), numpy "
                                         f"single-threaded")
    w = W.gpt2_small()
    n = 2_000_000
    hp = AdamWConfig(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    idx = np.arange(n, dtype=np.int64)
    contribs = [oracle_rank_values(w, 0, idx, lambda u, k, q=q: w.grad_stream(1, q, 0, u, k),
                                   "bf16") for q in range(w.nd)]
    p = oracle_rank_values(w, 0, idx, w.master_stream, "f32")
    shards = [synth.host_fill(w.peer_shard_stream(1, q, 0), 0, n // 64, "bf16")
              for q in range(w.nd)]
    lay = oracle.layout([w.nd * (n // 64)], w.nd)
    total_t, total_b, reps = 0.0, 0, 0
    while total_t < budget_s and reps < 50:
        z = np.zeros(n, np.float32)
        t0 = time.perf_counter()
        oracle.fsdp_shard_step(contribs, 0, n, p, z, z, hp, reps + 1)
        oracle.ag_unpack(shards, lay)
        total_t += time.perf_counter() - t0
        total_b += (2 * w.nd + 26) * n + 4 * w.nd * (n // 64)
        reps += 1
    return total_b / total_t / 1e9, (f"{reps} x (fused step on the first {n} elements of rank "
                                     f"0's view + all-gather of {w.nd * (n // 64)} bf16), numpy "
                                     f"single-threaded")


def run_small(args):
    """The two small model-shaped workloads: a 9.4M-parameter unit (N_d = 4,
    M = 4) and the GPT-2 small model (N_d = 8), each as its whole job on one
    GPU.  At these sizes (a step of 1.5 GB and 5.3 GB) launch latency is part
    of the answer, so the line gives the eager step and, with --graph, the
    same launches replayed from one CUDA graph.  L2 is flushed (256 MB
    written) between timed steps, outside the timed events."""
    world, rank, local = dist_env()
    name = args.workload
    metric = SMALL_METRICS[name]
    if args.impl == "reference":
        if rank != 0:
            return
        value, sample = _small_oracle(name, max(1.0, args.cpu_seconds))
        print(json.dumps({
            "impl": "reference", "metric": metric, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": name},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return
    init_dist(world)
    import torch
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    _apply_stages(args)
    import sharded_optimizer_step_gb300 as ss
    dev = torch.device("cuda", local)
    job = _SmallJob(name, torch, ss, dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    run = job.run
    graph_launches = 0
    if args.graph:
        job.device_state()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            job.run(graph_form=True)          # warm-up outside the capture
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        l0 = ss.launch_count()
        with torch.cuda.graph(graph):
            job.run(graph_form=True)
        graph_launches = ss.launch_count() - l0

        def run(ev=None):                     # noqa: F811 -- the replayed step
            if ev is not None:
                ev[0].record()
                ev[1].record()
                ev[2].record()
            graph.replay()
            if ev is not None:
                ev[3].record()

    def one_step(ev):
        flush.zero_()                         # L2 holds nothing of the previous step
        run(ev)

    total_ms, events, clk, launches = _timed_loop(torch, stream, args, one_step, 4, world)
    launches += graph_launches * args.steps
    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    ms_per_step = allreduce_max(world, sum(step_ms) / len(step_ms))
    value = allreduce_sum(world, job.step_bytes) / (ms_per_step / 1e3) / 1e9
    parts = {}
    if not args.graph:
        for k, (pname, b) in enumerate(job.parts if name == UNIT9M_WORKLOAD
                                       else [("accumulate", 0)] + job.parts):
            if pname == "accumulate" and b == 0:
                continue
            ms = _avg_ms(events, k, k + 1)
            parts[pname] = {"ms": round(ms, 4), "gbs": round(b / (ms / 1e3) / 1e9, 1)}
    dom_name, dom_bytes = max(job.parts, key=lambda x: x[1])
    if parts:
        dom_ms = parts[dom_name]["ms"]
        dom_kernel = ("accumulate_vec8 (register-staged)" if dom_name == "accumulate"
                      else "rs_adamw_cast_vec4<8, bf16> (register-staged)")
        n_launch = job.w.micro - 1 if dom_name == "accumulate" else job.w.nd
        roof = _roofline(dom_bytes / (dom_ms / 1e3) / 1e9, f"{dom_kernel}, {n_launch} launches "
                         f"per step ({dom_name})", dom_bytes // n_launch)
    else:
        roof = _roofline(job.step_bytes / (ms_per_step / 1e3) / 1e9,
                         "the whole step replayed from one CUDA graph (per-kernel times not "
                         "separable)", job.step_bytes)

    # end to end: every gradient input copied in from pinned host memory and
    # the gathered unit copied out, inside the timing, each step
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_plain(torch, stream, job.inputs(), [job.full], lambda: run(None),
                         job.step_bytes, world, args.e2e_steps,
                         "every rank's gradients (every micro-batch) in, the gathered unit out")

    cpu = None
    if rank == 0 and not args.no_cpu:
        cv, sample = _small_oracle(name, args.cpu_seconds)
        cpu = {"value": round(cv, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": sample}
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator on the device; no data set or "
                    "weights)",
            "config": {"workload": name, "graph": bool(args.graph), "psi": job.w.psi,
                       "nd": job.w.nd, "micro_batches": job.w.micro,
                       "units": len(job.w.units), "ranks_per_gpu": job.w.nd,
                       "elements_updated_per_step": job.shard_elements,
                       "bytes_per_step": job.step_bytes,
                       "roofline_ms": round(job.step_bytes / measured_peak()[0] / 1e6, 4),
                       "l2": "flushed between steps (256 MB written, outside the timed events)",
                       "tma_stages": _stages_name(args),
                       "dependent_launch": not args.no_dependent_launch},
            "params_per_s": round(job.shard_elements * world / (ms_per_step / 1e3), 1),
            "kernels": parts,
            "roofline": roof,
            "e2e": e2e,
            "gpu_launches": launches,
            **({"gpu_launches_note": f"{graph_launches} kernels per replayed step, counted when "
                                     f"the graph was captured"} if args.graph else {}),
            "clocks": clk,
            "cpu_baseline": cpu,
        }))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.workload in SMALL_METRICS:
        run_small(args)
        return
    if args.workload == ACCUM_WORKLOAD:
        run_accum(args)
        return
    if args.workload == DDP_WORKLOAD:
        run_ddp(args)
        return
    if args.workload == CKPT_WORKLOAD:
        if args.impl == "reference":
            run_ckpt_reference(args)
        else:
            run_ckpt(args)
        return
    if args.workload == RAGGED_WORKLOAD:
        run_ragged(args)
        return
    if args.workload == FSDP2_WORKLOAD:
        if args.impl == "reference":
            run_fsdp2_reference(args)
            return
        run_fsdp2(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
