"""ctypes declarations of ``libfused_adamw.so`` (mirrors include/fused_adamw.h).

Loading fails loudly when the library has not been built: there is no
fallback of any kind.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

from .build import LIB_PATH

c_i32, c_i64, c_u64, c_f64, c_vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_double, ctypes.c_void_p)

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_DTYPE", 3: "FA_ERR_SIZE",
                4: "FA_ERR_OPTION", 5: "FA_ERR_ALIAS", 6: "FA_ERR_POINTER", 7: "FA_ERR_ALIGN",
                8: "FA_ERR_PLAN", 9: "FA_ERR_CUDA", 10: "FA_ERR_SEGMENTS"}
FA_F32, FA_F16, FA_BF16 = 0, 1, 2


class FaOptions(ctypes.Structure):
    _fields_ = [("lr", c_f64), ("beta1", c_f64), ("beta2", c_f64), ("eps", c_f64),
                ("weight_decay", c_f64), ("amsgrad", c_i32), ("maximize", c_i32)]


class FaStepControl(ctypes.Structure):
    _fields_ = [("gradient_scale", c_f64), ("skip_update", c_i32)]


class FaStats(ctypes.Structure):
    _fields_ = [("sum_sq", ctypes.c_float), ("nonfinite", ctypes.c_uint32),
                ("sum_sq_lo", ctypes.c_float)]


class FaBucketUpdate(ctypes.Structure):
    _fields_ = [("seg_offsets", ctypes.POINTER(c_i64)), ("nseg", c_i32), ("n_total", c_i64),
                ("p", c_vp), ("g", c_vp), ("gdt", c_i32), ("m", c_vp), ("v", c_vp),
                ("vmax", c_vp), ("t", c_u64), ("grad_mult", c_f64),
                ("seg_grad_mult", ctypes.POINTER(c_f64)), ("report", c_vp),
                ("seg_reports", c_vp), ("max_grad_norm", c_f64), ("p_model", c_vp),
                ("model_dtype", c_i32), ("seg_decided", c_vp), ("seg_decided_elements", c_i64)]


class FaStepReport(ctypes.Structure):
    _fields_ = [("updated", c_i32), ("skipped_nonfinite", c_i32), ("nonfinite", c_u64),
                ("grad_norm", c_f64), ("clip_coef", c_f64)]


P = c_vp
PI64 = ctypes.POINTER(c_i64)
PU64 = ctypes.POINTER(c_u64)
PI32 = ctypes.POINTER(c_i32)
PF64 = ctypes.POINTER(c_f64)

# name -> (restype, argtypes)
SIGNATURES = {
    "fa_abi_version": (c_i32, []),
    "fa_stats_sum_sq": (c_i32, [ctypes.POINTER(FaStats), PF64]),
    "fa_status_string": (ctypes.c_char_p, [c_i32]),
    "fa_options_default": (FaOptions, []),
    "fa_device_error": (c_i32, [PI32, c_i32]),
    "fa_bounds_check_report": (c_i32, [PI32, PU64, c_i32]),
    "fa_pipeline_selftest": (c_i32, [c_i64, P, P, c_i32, P, P, PI32, P]),
    "fa_step_coefficients": (c_i32, [ctypes.POINTER(FaOptions), c_u64, c_f64, c_f64,
                                     ctypes.POINTER(ctypes.c_float)]),
    "fa_adamw_step": (c_i32, [c_i64, P, P, c_i32, P, P, P, c_u64, ctypes.POINTER(FaOptions),
                              FaStepControl, P, P, P, P, PU64, PI32, P]),
    "fa_adamw_step_inplace": (c_i32, [c_i64, P, P, c_i32, P, P, P, PU64,
                                      ctypes.POINTER(FaOptions), FaStepControl, c_f64, PI32, P]),
    "fa_bucket_step": (c_i32, [PI64, c_i32, c_i64, P, P, c_i32, P, P, P, PU64,
                               ctypes.POINTER(FaOptions), FaStepControl, c_f64, PI32, P]),
    "fa_bucket_update": (c_i32, [ctypes.POINTER(FaBucketUpdate), ctypes.POINTER(FaOptions),
                                 FaStepControl, PI32, P]),
    "fa_adamw_step_staged": (c_i32, [c_i64, P, P, c_i32, P, P, P, PU64,
                                     ctypes.POINTER(FaOptions), FaStepControl, c_f64, P, PI32,
                                     P]),
    "fa_bucket_step_clipped_gated": (c_i32, [PI64, c_i32, c_i64, P, P, c_i32, P, P, P, PU64,
                                             ctypes.POINTER(FaOptions), FaStepControl, c_f64,
                                             c_i32, P, c_i64, P, c_i64, P, P,
                                             ctypes.POINTER(FaStepReport), P]),
    "fa_stats_plan": (c_i32, [c_i64, PI32, PI64]),
    "fa_stats_rows": (c_i32, [c_i64, c_i32, PI64, c_i32, PI64]),
    "fa_analyze_gradient": (c_i32, [P, c_i32, c_i64, c_i32, PI64, c_i32, P, c_i64, P]),
    "fa_merge_gradient_stats": (c_i32, [P, c_i64, P, c_i64, P, P]),
    "fa_merge_gradient_stats_static": (c_i32, [P, c_i64, P, P]),
    "fa_stats_chunk_scratch": (c_i32, [PI64, c_i32, PI64]),
    "fa_merge_gradient_stats_chunks": (c_i32, [P, PI64, c_i32, P, c_i64, P, P]),
    "fa_bucket_step_clipped_per_segment": (c_i32, [PI64, c_i32, c_i64, P, P, c_i32, P, P, P,
                                                   PU64, ctypes.POINTER(FaOptions),
                                                   FaStepControl, c_f64, c_i32, P, c_i64, P,
                                                   c_i64, P, PF64, PF64,
                                                   ctypes.POINTER(FaStepReport), P]),
    "fa_bucket_step_clipped_per_segment_gated": (c_i32, [PI64, c_i32, c_i64, P, P, c_i32, P, P,
                                                         P, c_u64, ctypes.POINTER(FaOptions),
                                                         FaStepControl, c_f64, c_i32, P, c_i64,
                                                         P, c_i64, P, P, P]),
    "fa_read_report": (c_i32, [P, ctypes.POINTER(FaStats), P]),
    "fa_clip_decision": (c_i32, [c_f64, c_u64, c_f64, c_f64, PI32, PF64, PF64]),
    "fa_clip_decide": (c_i32, [P, c_f64, c_f64, PI32, PF64, PF64, P]),
    "fa_bucket_step_clipped": (c_i32, [PI64, c_i32, c_i64, P, P, c_i32, P, P, P, PU64,
                                       ctypes.POINTER(FaOptions), FaStepControl, c_f64, c_i32,
                                       P, c_i64, P, c_i64, P, ctypes.POINTER(FaStepReport), P]),
}

_LIB = None
_OVERRIDE = None  # a library variant used in place of the normal one (see ``using``)


def open_library(path: str) -> ctypes.CDLL:
    """Loads a build of the library at ``path`` with every signature declared."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built: run amsgrad_optimizer_step_gb300.build.build() "
            "(nvcc, sm_103a). There is no CPU or library fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _OVERRIDE is not None:
        return _OVERRIDE
    if _LIB is None:
        _LIB = open_library(path)
    return _LIB


@contextlib.contextmanager
def using(lib: ctypes.CDLL):
    """Routes every binding call through ``lib`` (e.g. the bounds-checked build)."""
    global _OVERRIDE
    prev = _OVERRIDE
    _OVERRIDE = lib
    try:
        yield lib
    finally:
        _OVERRIDE = prev


class FusedAdamWError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = load().fa_status_string(status).decode()
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({msg})")


def check(fn: str, status: int) -> None:
    if status != FA_OK:
        raise FusedAdamWError(fn, status)
