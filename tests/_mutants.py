"""Planted mistakes in the oracle, to show that its pins catch them.

Each mutant is a plausible slip in one oracle module (a dropped term, a wrong
sign or index, a transposed operand, a rounding or ordering mistake), written
as an exact text edit of that module's source.  ``python -m tests._mutants``
runs, in one process: the pins of every module unmodified (they must pass),
then, for each mutant, the module re-executed with the edit and its pins run
again (at least one must fail), then the module restored.  It prints one JSON
object {mutant: pytest exit code}.  Everything here runs on the CPU and
touches only the oracle; nothing under the library is imported."""
from __future__ import annotations

import contextlib
import importlib
import io
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# the pin files that call each oracle module's functions
PINS = {
    "oracle.numerics": ["tests/test_oracle_numerics.py", "tests/test_oracle_hybrid.py",
                        "tests/test_oracle_ddp_ledger.py", "tests/test_oracle_scaler.py",
                        "tests/test_oracle_fsdp2.py"],
    "oracle.flat": ["tests/test_oracle_layout.py", "tests/test_oracle_checkpoint.py"],
    "oracle.fsdp2": ["tests/test_oracle_fsdp2.py"],
    "oracle.scaler": ["tests/test_oracle_scaler.py"],
    "oracle.ddp": ["tests/test_oracle_ddp_ledger.py"],
    "oracle.ledger": ["tests/test_oracle_ddp_ledger.py", "tests/test_oracle_hybrid.py"],
    "oracle.checkpoint": ["tests/test_oracle_checkpoint.py"],
}

# name -> (module, [(old, new), ...])
MUTANTS = {
    # ---- bf16 cast and upcast
    "bf16_ties_away_from_zero": ("oracle.numerics", [
        ("up = (d_hi < d_lo) | ((d_hi == d_lo) & odd)", "up = d_hi <= d_lo")]),
    "bf16_truncates": ("oracle.numerics", [
        ("res = (lo >> np.uint32(16)) + up.astype(np.uint32)", "res = lo >> np.uint32(16)")]),
    "bf16_ulp_off_by_one_binade": ("oracle.numerics", [
        ("np.maximum(exp, 1) - 127 - 7", "np.maximum(exp, 1) - 127 - 8")]),
    "bf16_nan_not_quieted": ("oracle.numerics", [
        ("(mag >> np.uint32(16)) | np.uint32(0x40)", "(mag >> np.uint32(16))")]),
    "bf16_sign_dropped": ("oracle.numerics", [
        ("res = res | (sign >> np.uint32(16))", "res = res")]),
    "bf16_upcast_wrong_shift": ("oracle.numerics", [
        ("(u16.astype(np.uint32) << np.uint32(16))", "(u16.astype(np.uint32) << np.uint32(15))")]),
    # ---- accumulation
    "accumulate_first_term_unscaled": ("oracle.numerics", [
        ("acc = g0 * s", "acc = g0.copy()")]),
    "accumulate_later_terms_unscaled": ("oracle.numerics", [
        ("acc = acc + _upcast(g) * s", "acc = acc + _upcast(g)")]),
    "accumulate_drops_last_micro_batch": ("oracle.numerics", [
        ("for g in micro_grads[1:]:", "for g in micro_grads[1:-1]:")]),
    # ---- reduce-scatter average
    "rs_sum_not_mean": ("oracle.numerics", [
        ("return s / s.dtype.type(nd)", "return s")]),
    "rs_divides_by_nd_minus_1": ("oracle.numerics", [
        ("return s / s.dtype.type(nd)", "return s / s.dtype.type(max(nd - 1, 1))")]),
    "rs_takes_rank_0_slice": ("oracle.numerics", [
        ("sl = [_upcast(c[r * shard:(r + 1) * shard]) for c in contribs]",
         "sl = [_upcast(c[0:shard]) for c in contribs]")]),
    "rs_reverse_rank_order": ("oracle.numerics", [
        ("    s = sl[0].copy()\n    for q in range(1, nd):\n        s = s + sl[q]",
         "    s = sl[nd - 1].copy()\n    for q in range(1, nd):\n        s = s + sl[nd - 1 - q]")]),
    "rs_multiplies_by_reciprocal": ("oracle.numerics", [
        ("return s / s.dtype.type(nd)", "return s * (s.dtype.type(1) / s.dtype.type(nd))")]),
    # ---- AdamW
    "adamw_no_weight_decay": ("oracle.numerics", [
        ("p = p - c.lr_wd * p", "p = p")]),
    "adamw_weight_decay_wrong_sign": ("oracle.numerics", [
        ("p = p - c.lr_wd * p", "p = p + c.lr_wd * p")]),
    "adamw_weight_decay_after_update": ("oracle.numerics", [
        ("    p = p - c.lr_wd * p\n", ""),
        ("    p = p - (c.step_size * m) / denom\n",
         "    p = p - (c.step_size * m) / denom\n    p = p - c.lr_wd * p\n")]),
    "adamw_betas_swapped_in_m": ("oracle.numerics", [
        ("m = c.beta1 * m + c.omb1 * g", "m = c.omb1 * m + c.beta1 * g")]),
    "adamw_v_of_g_not_g2": ("oracle.numerics", [
        ("v = c.beta2 * v + (c.omb2 * g) * g", "v = c.beta2 * v + c.omb2 * np.abs(g)")]),
    "adamw_beta1_in_v": ("oracle.numerics", [
        ("v = c.beta2 * v + (c.omb2 * g) * g", "v = c.beta1 * v + (c.omb1 * g) * g")]),
    "adamw_no_v_bias_correction": ("oracle.numerics", [
        ("denom = np.sqrt(v) / c.sqrt_bc2 + c.eps", "denom = np.sqrt(v) + c.eps")]),
    "adamw_no_m_bias_correction": ("oracle.numerics", [
        ("step_size=f(hp.lr / bc1)", "step_size=f(hp.lr)")]),
    "adamw_eps_inside_sqrt": ("oracle.numerics", [
        ("denom = np.sqrt(v) / c.sqrt_bc2 + c.eps",
         "denom = np.sqrt(v / (c.sqrt_bc2 * c.sqrt_bc2) + c.eps)")]),
    "adamw_step_count_off_by_one": ("oracle.numerics", [
        ("    for _ in range(t):\n        b1t *= hp.beta1",
         "    for _ in range(t + 1):\n        b1t *= hp.beta1")]),
    "adamw_lr_times_wd_as_wd": ("oracle.numerics", [
        ("lr_wd=f(hp.lr * hp.weight_decay)", "lr_wd=f(hp.weight_decay)")]),
    "shard_step_casts_old_master": ("oracle.numerics", [
        ("    g = rs_avg(contribs, r, shard)\n    p, m, v = adamw(p, m, v, g, hp, t)\n"
         "    return p, m, v, f32_to_bf16(p)",
         "    g = rs_avg(contribs, r, shard)\n    out = f32_to_bf16(p)\n"
         "    p, m, v = adamw(p, m, v, g, hp, t)\n    return p, m, v, out")]),
    # ---- hybrid sharding
    "hybrid_divides_by_f": ("oracle.numerics", [
        ("return total / total.dtype.type(nd)", "return total / total.dtype.type(shard_group)")]),
    "hybrid_groups_transposed": ("oracle.numerics", [
        ("s = sl[g * shard_group].copy()", "s = sl[g].copy()"),
        ("s = s + sl[g * shard_group + j]", "s = s + sl[j * R + g]")]),
    "hybrid_takes_shard_0": ("oracle.numerics", [
        ("sl = [_upcast(c[f * shard:(f + 1) * shard]) for c in contribs]",
         "sl = [_upcast(c[0:shard]) for c in contribs]")]),
    # ---- FlatParameter layout, pack, gather
    "layout_no_padding": ("oracle.flat", [
        ("padded = -(-total // nd) * nd", "padded = total")]),
    "layout_pads_a_whole_extra_row": ("oracle.flat", [
        ("padded = -(-total // nd) * nd", "padded = (total // nd + 1) * nd")]),
    "layout_offsets_shifted": ("oracle.flat", [
        ("        offsets.append(acc)\n        acc += n", "        acc += n\n        offsets.append(acc)")]),
    "layout_piece_end_unclamped": ("oracle.flat", [
        ("hi.append([min(max(off + n - base, 0), shard)", "hi.append([max(off + n - base, 0)")]),
    "layout_piece_start_unclamped_below": ("oracle.flat", [
        ("lo.append([min(max(off - base, 0), shard)", "lo.append([min(off - base, shard)")]),
    "pack_padding_not_zero": ("oracle.flat", [
        ("flat = np.zeros(lay.padded, dtype=dtype)", "flat = np.ones(lay.padded, dtype=dtype)")]),
    "gather_reverse_rank_order": ("oracle.flat", [
        ("np.concatenate([np.asarray(s).reshape(-1) for s in shards])",
         "np.concatenate([np.asarray(s).reshape(-1) for s in shards[::-1]])")]),
    "element_source_absolute_index": ("oracle.flat", [
        ("k[sel] = flat_idx[sel] - off", "k[sel] = flat_idx[sel]")]),
    "rank_view_forgets_rank_offset": ("oracle.flat", [
        ("element_source(lay, r * lay.shard + (idx[sel] - start))",
         "element_source(lay, idx[sel] - start)")]),
    # ---- FSDP2 Shard(0)
    "fsdp2_chunk_floor": ("oracle.fsdp2", [
        ("c = -(-d0 // nd)", "c = max(1, d0 // nd)")]),
    "fsdp2_every_rank_full_chunk": ("oracle.fsdp2", [
        ("return max(0, min(c, d0 - r * c))", "return c if r * c < d0 else 0")]),
    "fsdp2_chunk_cat_param_major": ("oracle.fsdp2", [
        ("dst = r * lay.local + lay.offset[t]",
         "dst = lay.offset[t] * lay.nd + r * lay.chunk[t] * lay.row[t]")]),
    "fsdp2_copy_out_uses_own_rows": ("oracle.fsdp2", [
        ("            dst = r * lay.chunk[t] * lay.row[t]\n            full[dst:dst + n]",
         "            dst = r * n\n            full[dst:dst + n]")]),
    # ---- gradient scaler
    "scaler_ignores_nan": ("oracle.scaler", [
        ("return not bool(np.all(np.isfinite(", "return not bool(np.all(~np.isinf(")]),
    "scaler_multiplies_by_scale": ("oracle.scaler", [
        ("return g * np.float32(inv_scale)", "return g / np.float32(inv_scale)")]),
    "scaler_skip_still_updates": ("oracle.scaler", [
        ("    if skip:\n        return p, m, v, out_prev", "    if False:\n        return p, m, v, out_prev")]),
    "scaler_backoff_keeps_tracker": ("oracle.scaler", [
        ("return np.float32(scale * np.float32(backoff_factor)), 0",
         "return np.float32(scale * np.float32(backoff_factor)), tracker")]),
    "scaler_growth_keeps_tracker": ("oracle.scaler", [
        ("            scale = grown\n        tracker = 0", "            scale = grown")]),
    "scaler_grows_to_inf": ("oracle.scaler", [
        ("if np.isfinite(grown):", "if True:")]),
    # ---- DDP buckets
    "ddp_forward_order": ("oracle.ddp", [
        ("for i in reversed(range(n)):", "for i in range(n):")]),
    "ddp_cap_exclusive": ("oracle.ddp", [
        ("if cur and cur_bytes + b > cap_bytes:", "if cur and cur_bytes + b >= cap_bytes:")]),
    "ddp_allreduce_sum_not_mean": ("oracle.ddp", [
        ("out[a:e] = f32_to_bf16(s / np.float32(nd))", "out[a:e] = f32_to_bf16(s)")]),
    "ddp_step_uses_fp32_mean": ("oracle.ddp", [
        ("p, m, v = adamw(p, m, v, bf16_to_f32(avg), hp, t)",
         "p, m, v = adamw(p, m, v, sum(bf16_to_f32(g) for g in rank_grads) "
         "/ np.float32(len(rank_grads)), hp, t)")]),
    # ---- memory and communication ledger
    "ledger_zero2_as_zero1": ("oracle.ledger", [
        ("return 2 * psi + (2 * psi + k * psi) / nd", "return 2 * psi + 2 * psi + k * psi / nd")]),
    "ledger_ddp_one_pass": ("oracle.ledger", [
        ('"ddp": 2 * one,', '"ddp": one,')]),
    "ledger_zero3_two_passes": ("oracle.ledger", [
        ('"zero3": one + one + one,', '"zero3": one + one,')]),
    "ledger_hybrid_grads_replicated": ("oracle.ledger", [
        ("return (2 * psi + 2 * psi + k * psi) / shard_group",
         "return 2 * psi + (2 * psi + k * psi) / shard_group")]),
    "ledger_hybrid_inter_whole_model": ("oracle.ledger", [
        ("return 4 * (psi / shard_group) * f if R > 1 else 0.0", "return 4 * psi * f if R > 1 else 0.0")]),
    # ---- sharded checkpoint
    "ckpt_keeps_old_padding": ("oracle.checkpoint", [
        ("return np.concatenate([np.asarray(s).reshape(-1) for s in old_shards])[:total]",
         "return np.concatenate([np.asarray(s).reshape(-1) for s in old_shards])")]),
    "ckpt_plan_floor_shard": ("oracle.checkpoint", [
        ("S_old = -(-total // old_nd)", "S_old = max(1, total // old_nd)")]),
    "ckpt_reshard_wrong_rank": ("oracle.checkpoint", [
        ("return full[new_rank * S:(new_rank + 1) * S]", "return full[0:S]")]),
}


def _oracle_modules():
    return {k: m for k, m in sys.modules.items() if k == "oracle" or k.startswith("oracle.")}


_CLASS_UNDO = []      # (class, attribute, original value) of patched methods


def _apply(modname, edits):
    """Re-execute ``modname`` with the edits; point every reference that other
    oracle modules (and the package's re-exports) hold to its old functions
    at the new ones.  Classes stay the original objects (instances made
    before keep working); their methods take the edited bodies."""
    mod = importlib.import_module(modname)
    with open(mod.__file__, encoding="utf-8") as f:
        src = f.read()
    for old, new in edits:
        n = src.count(old)
        if n != 1:
            raise ValueError(f"{modname}: edit text found {n} times: {old!r}")
        src = src.replace(old, new)
    old_objs = dict(vars(mod))
    exec(compile(src, mod.__file__, "exec"), mod.__dict__)
    for k, v in old_objs.items():
        if isinstance(v, type):
            edited = mod.__dict__[k]
            for a, f in vars(edited).items():
                if callable(f) and not a.startswith("__") and vars(v).get(a) is not f:
                    _CLASS_UNDO.append((v, a, vars(v).get(a)))
                    setattr(v, a, f)
            mod.__dict__[k] = v
    swap = {id(v): mod.__dict__[k] for k, v in old_objs.items()
            if callable(v) and not isinstance(v, type) and mod.__dict__.get(k) is not v}
    for m in _oracle_modules().values():
        for k, v in list(vars(m).items()):
            if id(v) in swap:
                setattr(m, k, swap[id(v)])


def _run(files):
    import pytest
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf), contextlib.redirect_stderr(buf):
        return int(pytest.main([*files, "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                                "--rootdir", ROOT]))


def main():
    os.chdir(ROOT)
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle                          # noqa: F401 -- every submodule loaded
    for name in sorted(PINS):
        importlib.import_module(name)
    snapshot = {k: dict(vars(m)) for k, m in _oracle_modules().items()}
    all_pins = sorted({f for fs in PINS.values() for f in fs})
    result = {"<none>": _run(all_pins)}
    only = sys.argv[1:]
    for name, (modname, edits) in MUTANTS.items():
        if only and name not in only:
            continue
        try:
            _apply(modname, edits)
            result[name] = _run(PINS[modname])
        finally:
            for k, m in _oracle_modules().items():
                d = m.__dict__
                d.clear()
                d.update(snapshot[k])
            while _CLASS_UNDO:
                cls, a, f = _CLASS_UNDO.pop()
                setattr(cls, a, f)
    print(json.dumps(result))


if __name__ == "__main__":
    main()
