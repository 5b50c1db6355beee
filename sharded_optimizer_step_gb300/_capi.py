"""ctypes declarations of libshardstep.so (include/shardstep.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any entry point."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_i32, c_i64, c_u64, c_f32, c_f64, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                           ctypes.c_float, ctypes.c_double, ctypes.c_void_p)
P_i64 = ctypes.POINTER(ctypes.c_int64)
P_i32 = ctypes.POINTER(ctypes.c_int32)
P_vp = ctypes.POINTER(ctypes.c_void_p)

OK = 0
ERR_INVALID = -1
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_CAPACITY = -5
ERR_IO = -6
PATH_AUTO = 0
PATH_REGISTER = 1
PATH_TMA = 2
DTYPE_BF16 = 0
DTYPE_F32 = 1
DTYPE_F16 = 2
MAX_ND = 64
COMM_KINDS = {"reduce_scatter": 0, "all_gather": 1, "all_reduce": 2, "ddp": 2,
              "zero1": 3, "zero2": 4, "zero3": 5}


class AdamWHP(ctypes.Structure):
    _fields_ = [("lr", c_f64), ("beta1", c_f64), ("beta2", c_f64), ("eps", c_f64),
                ("weight_decay", c_f64), ("step", c_i64)]


class LayoutInfo(ctypes.Structure):
    _fields_ = [("total", c_i64), ("padded", c_i64), ("shard", c_i64), ("n_tensors", c_i32),
                ("nd", c_i32)]


class CkptSection(ctypes.Structure):
    _fields_ = [("unit", c_i32), ("kind", c_i32), ("bytes", c_i64), ("data", c_vp)]


class CkptInfo(ctypes.Structure):
    _fields_ = [("nd", c_i32), ("rank", c_i32), ("n_units", c_i32), ("n_sections", c_i32),
                ("step", c_i64)]


class CkptPiece(ctypes.Structure):
    _fields_ = [("old_rank", c_i32), ("pad_", c_i32), ("old_offset", c_i64),
                ("new_offset", c_i64), ("count", c_i64)]


# name -> (restype, argtypes), exactly the declarations of include/shardstep.h
SIGNATURES = {
    "fsdp_layout": (c_i32, [P_i64, c_i32, c_i32, ctypes.POINTER(LayoutInfo), P_i64, P_i64, P_i64]),
    "fsdp_flat_pack": (c_i32, [P_vp, P_i64, c_i32, c_i32, c_i32, c_vp, c_vp]),
    "fsdp_views": (c_i32, [P_i64, c_i32, c_i32, c_i32, c_vp, c_i32, P_vp, P_i64]),
    "fsdp_shard_pieces": (c_i32, [P_i64, c_i32, c_i32, c_i32, P_i64, P_i64, P_i64]),
    "fsdp_grad_accumulate": (c_i32, [c_vp, c_vp, c_i64, c_f32, c_i32, c_vp]),
    "fsdp_rs_avg_adamw_cast": (c_i32, [P_vp, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp, c_vp,
                                       ctypes.POINTER(AdamWHP), c_vp]),
    "fsdp_hybrid_rs_avg_adamw_cast": (c_i32, [P_vp, c_i32, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp,
                                              c_vp, ctypes.POINTER(AdamWHP), c_vp]),
    "fsdp_accumulate_rs_avg_adamw_cast": (c_i32, [P_vp, P_vp, c_i32, c_i32, c_i64, c_f32, c_vp,
                                                  c_vp, c_vp, c_vp, ctypes.POINTER(AdamWHP),
                                                  c_vp]),
    "fsdp_state_accumulate_rs_avg_adamw_cast": (c_i32, [P_vp, P_vp, c_i32, c_i32, c_i64, c_f32,
                                                        c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fsdp_grad_unscale_check": (c_i32, [P_vp, c_i32, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp]),
    "fsdp_scaled_rs_avg_adamw_cast": (c_i32, [P_vp, c_i32, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp,
                                              c_vp, ctypes.POINTER(AdamWHP), c_vp, c_vp, c_vp]),
    "fsdp_grad_scaler_update": (c_i32, [c_vp, c_vp, c_vp, c_f32, c_f32, c_i32, c_vp]),
    "fsdp_ag_unpack": (c_i32, [P_vp, c_i32, c_i64, c_vp, c_vp]),
    "fsdp2_layout": (c_i32, [P_i64, P_i64, c_i32, c_i32, P_i64, P_i64, P_i64]),
    "fsdp2_local_views": (c_i32, [P_i64, P_i64, c_i32, c_i32, c_i32, c_vp, c_i32, P_vp, P_i64]),
    "fsdp2_rs_avg_adamw_cast": (c_i32, [P_vp, c_i32, P_i64, P_i64, c_i32, c_i32, c_i32, c_vp,
                                        c_vp, c_vp, c_vp, ctypes.POINTER(AdamWHP), c_vp]),
    "fsdp2_state_rs_avg_adamw_cast": (c_i32, [P_vp, c_i32, P_i64, P_i64, c_i32, c_i32, c_i32,
                                              c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fsdp2_chunk_cat": (c_i32, [P_vp, P_i64, P_i64, c_i32, c_i32, c_i32, c_vp, c_vp]),
    "fsdp2_all_gather_copy_out": (c_i32, [P_vp, P_i64, P_i64, c_i32, c_i32, c_i32, P_vp, c_vp]),
    "ddp_bucket_plan": (c_i32, [P_i64, c_i32, c_i32, c_i64, P_i64, P_i32, P_i64, P_i32]),
    "ddp_bucket_allreduce_avg": (c_i32, [P_vp, c_i32, P_i64, c_i32, c_i32, c_vp, c_vp]),
    "ddp_bucket_allreduce_avg_adamw_cast": (c_i32, [P_vp, c_i32, P_i64, c_i32, c_i32, c_vp, c_vp,
                                                    c_vp, c_vp, c_vp, ctypes.POINTER(AdamWHP),
                                                    c_vp]),
    "shardstep_state_bytes": (c_f64, [c_f64, c_i32, c_i32, c_f64]),
    "shardstep_comm_bytes": (c_f64, [c_f64, c_i32, c_i32, c_i32]),
    "shardstep_comm_counter": (c_f64, [c_i32]),
    "shardstep_hybrid_state_bytes": (c_f64, [c_f64, c_i32, c_f64]),
    "shardstep_hybrid_comm_bytes": (c_f64, [c_f64, c_i32, c_i32, c_i32, c_i32]),
    "shardstep_ckpt_save_rank": (c_i32, [ctypes.c_char_p, c_i32, c_i32, c_i64, P_i64, c_i32,
                                         ctypes.POINTER(CkptSection), c_i32]),
    "shardstep_ckpt_info": (c_i32, [ctypes.c_char_p, ctypes.POINTER(CkptInfo), P_i64, c_i32]),
    "shardstep_ckpt_read": (c_i32, [ctypes.c_char_p, c_i32, c_i32, c_i64, c_i64, c_vp]),
    "shardstep_ckpt_verify": (c_i32, [ctypes.c_char_p]),
    "fsdp_reshard_plan": (c_i32, [c_i64, c_i32, c_i32, c_i32, ctypes.POINTER(CkptPiece), c_i32,
                                  P_i32]),
    "shardstep_last_error": (ctypes.c_char_p, []),
    "ddp_ready_bytes": (c_i64, [c_i32, c_i32, c_i32]),
    "ddp_ready_init": (c_i32, [c_vp, c_i64, c_vp, c_i32, c_i32, c_i32]),
    "ddp_ready_mark": (c_i32, [c_vp, c_i32, c_i32, c_vp]),
    "ddp_ready_wait": (c_i32, [c_vp, c_i32, c_i64, c_vp, c_vp]),
    "ddp_ready_reset": (c_i32, [c_vp]),
    "shardstep_set_fused_path": (c_i32, [c_i32]),
    "shardstep_set_tma_stages": (c_i32, [c_i32]),
    "shardstep_set_dependent_launch": (c_i32, [c_i32]),
    "shardstep_device_status": (c_i32, [ctypes.POINTER(ctypes.c_uint32), c_i32]),
    "shardstep_set_tma_wait_ns": (c_i64, [c_i64]),
    "shardstep_check_mean_division": (c_i32, [c_i32, c_vp, c_vp, c_vp]),
    "shardstep_launch_count": (c_u64, []),
    "shardstep_last_kernel": (ctypes.c_char_p, []),
    "shardstep_adamw_state_init": (c_i32, [c_vp, ctypes.POINTER(AdamWHP), c_i64, c_vp]),
    "shardstep_adamw_state_advance": (c_i32, [c_vp, ctypes.POINTER(AdamWHP), c_vp, c_vp]),
    "fsdp_state_scaled_rs_avg_adamw_cast": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i64, c_vp, c_vp,
                                                    c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fsdp_state_rs_avg_adamw_cast": (c_i32, [c_vp, c_i32, c_i32, c_i32, c_i64, c_vp, c_vp, c_vp,
                                             c_vp, c_vp, c_vp]),
}

# Size in bytes of shardstep_adamw_state_t (int64 step, two doubles, 8 floats).
ADAMW_STATE_BYTES = 56

_lib = None


class ShardstepError(RuntimeError):
    def __init__(self, name, code, msg):
        super().__init__(f"{name} failed ({code}): {msg}")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library.  Raises if it was not built (call ``build()``)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: the CUDA library has not been built "
                "(run sharded_optimizer_step_gb300.build()); there is no fallback")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(name: str, rc: int) -> None:
    if rc != OK:
        raise ShardstepError(name, rc, lib().shardstep_last_error().decode())


def i64_array(values):
    values = [int(x) for x in values]
    return (c_i64 * max(1, len(values)))(*values)


def ptr_array(ptrs):
    ptrs = [int(p) if p is not None else 0 for p in ptrs]
    return (c_vp * max(1, len(ptrs)))(*ptrs)
