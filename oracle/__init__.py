"""ORACLE -- TEST INFRASTRUCTURE ONLY.

A plain FP64 CPU restatement of the fused AdamW / AMSGrad step and of the
gradient statistics around it, used to check the CUDA library.  Only the
tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import
this package; the product path never does, and the two share no code.

The arithmetic lives in ``adamw_oracle.c`` and ``stats_oracle.c`` (plain C,
single-threaded, built with gcc -O2 -ffp-contract=off).  This module builds
them, loads them through ctypes, and adds the host-side control flow that the
pages state around one update call:

* RUDA "实验性融合 AdamW / AMSGrad" (zh/docs/fused-adamw), "增加的实际能力": an empty
  tensor or skip_update = true changes nothing and does not advance the step;
  the first update initialises the moments without reading them.
* RUDA "実験的なデバイス上の融合 AdamW / AMSGrad" (ja/docs/fused-adamw),
  "この演算子を使用する理由": the update is indexed by the 1-based step t.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ("adamw_oracle.c", "stats_oracle.c")
LIB_NAME = "liboracle.so"

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {"f32": F32, "f16": F16, "bf16": BF16}

# The page's reduction limits (ja/docs/fused-adamw, "ネイティブ PyTorch ストレージと階層統計").
FAN_IN = 1024
MAX_ROWS = 4_194_304


class _Options(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("amsgrad", ctypes.c_int32),
                ("maximize", ctypes.c_int32)]


def _native(path: str) -> bool:
    """True when the shared object at ``path`` was built for this machine (its ELF
    e_machine matches), so that one copied from another architecture is rebuilt."""
    import platform
    want = {"x86_64": 62, "amd64": 62, "aarch64": 183, "arm64": 183}.get(
        platform.machine().lower())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return want is None or int.from_bytes(head[18:20], "little") == want


def build(src_dir: str = HERE, out_path: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle C sources into a shared library; returns its path."""
    out_path = out_path or os.path.join(src_dir, LIB_NAME)
    srcs = [os.path.join(src_dir, s) for s in SOURCES]
    if (not force and os.path.exists(out_path) and _native(out_path)
            and all(os.path.getmtime(out_path) >= os.path.getmtime(s)
                    for s in srcs + [os.path.join(src_dir, "oracle.h")])):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-I", src_dir, "-o", tmp, *srcs, "-lm"],
                   check=True)
    os.replace(tmp, out_path)
    return out_path


class OracleLib:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: Optional[str] = None):
        path = path or build()
        self.path = path
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_widen.argtypes = [P, ctypes.c_int, ctypes.c_int64]
        lib.oracle_widen.restype = ctypes.c_double
        lib.oracle_int_pow.argtypes = [ctypes.c_double, ctypes.c_uint64]
        lib.oracle_int_pow.restype = ctypes.c_double
        lib.oracle_adamw_update.argtypes = [
            ctypes.c_int64, P, ctypes.c_int, ctypes.POINTER(_Options), ctypes.c_double,
            ctypes.c_double, ctypes.c_uint64, ctypes.c_int, ctypes.c_int, P, P, P, P]
        lib.oracle_adamw_update.restype = None
        lib.oracle_model_copy.argtypes = [ctypes.c_int64, P, ctypes.c_int, P]
        lib.oracle_model_copy.restype = None
        lib.oracle_gradient_stats.argtypes = [ctypes.c_int64, P, ctypes.c_int, ctypes.c_double,
                                              P, P]
        lib.oracle_gradient_stats.restype = None
        lib.oracle_row_stats.argtypes = [ctypes.c_int64, P, ctypes.c_int, ctypes.c_int64,
                                         P, ctypes.c_int64, P, P]
        lib.oracle_row_stats.restype = ctypes.c_int64
        lib.oracle_stats_plan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                          P, P, P]
        lib.oracle_stats_plan.restype = ctypes.c_int
        lib.oracle_clip_decision.argtypes = [ctypes.c_double, ctypes.c_uint64, ctypes.c_double,
                                             P, P, P]
        lib.oracle_clip_decision.restype = None
        self._lib = lib

    # ---- element-level helpers ----------------------------------------------
    def widen(self, g: np.ndarray, dtype: str) -> np.ndarray:
        g = np.ascontiguousarray(g)
        code = _DTYPE_CODE[dtype]
        return np.array([self._lib.oracle_widen(g.ctypes.data, code, i) for i in range(g.size)],
                        dtype=np.float64)

    def int_pow(self, beta: float, t: int) -> float:
        return self._lib.oracle_int_pow(beta, t)

    def update(self, g: np.ndarray, dtype: str, opts: dict, gradient_scale: float,
               clip_coef: float, t: int, have_state: bool, round_fp32: bool,
               p: np.ndarray, m: np.ndarray, v: np.ndarray, vmax: np.ndarray) -> None:
        """One update on FP64 state arrays, in place (see adamw_oracle.c)."""
        n = p.size
        g = np.ascontiguousarray(g)
        for a in (p, m, v, vmax):
            assert a.dtype == np.float64 and a.flags.c_contiguous and a.size == n
        o = _Options(opts["lr"], opts["beta1"], opts["beta2"], opts["eps"],
                     opts["weight_decay"], int(opts["amsgrad"]), int(opts["maximize"]))
        self._lib.oracle_adamw_update(n, g.ctypes.data, _DTYPE_CODE[dtype], ctypes.byref(o),
                                      gradient_scale, clip_coef, t, int(have_state),
                                      int(round_fp32), p.ctypes.data, m.ctypes.data,
                                      v.ctypes.data, vmax.ctypes.data)

    def model_copy(self, p: np.ndarray, dtype: str) -> np.ndarray:
        """BF16/FP16 bit patterns of FP32 values, rounded to nearest, ties to even."""
        p = np.ascontiguousarray(p, dtype=np.float32)
        out = np.zeros(p.size, dtype=np.uint16)
        self._lib.oracle_model_copy(p.size, p.ctypes.data, _DTYPE_CODE[dtype], out.ctypes.data)
        return out

    # ---- statistics ---------------------------------------------------------
    def gradient_stats(self, g: np.ndarray, dtype: str, gradient_scale: float = 1.0):
        g = np.ascontiguousarray(g)
        s = ctypes.c_double()
        c = ctypes.c_uint64()
        self._lib.oracle_gradient_stats(g.size, g.ctypes.data, _DTYPE_CODE[dtype],
                                        gradient_scale, ctypes.addressof(s), ctypes.addressof(c))
        return s.value, c.value

    def row_stats(self, g: np.ndarray, dtype: str, row_len: int, segments=None):
        g = np.ascontiguousarray(g)
        seg = (np.ascontiguousarray(segments, dtype=np.int64) if segments is not None
               else np.zeros(1, dtype=np.int64))
        nseg = seg.size - 1 if segments is not None else 0
        rows = self._lib.oracle_row_stats(g.size, g.ctypes.data, _DTYPE_CODE[dtype], row_len,
                                          seg.ctypes.data, nseg, None, None)
        if rows < 0:
            raise ValueError("malformed segment table")
        s = np.zeros(rows, dtype=np.float64)
        c = np.zeros(rows, dtype=np.uint64)
        self._lib.oracle_row_stats(g.size, g.ctypes.data, _DTYPE_CODE[dtype], row_len,
                                   seg.ctypes.data, nseg, s.ctypes.data, c.ctypes.data)
        return s, c

    def stats_plan(self, rows: int, fan_in: int = FAN_IN, max_rows: int = MAX_ROWS):
        """(merge kernels, scratch FP32 elements, records per level) or None if rejected."""
        k = ctypes.c_int()
        e = ctypes.c_int64()
        lv = np.zeros(64, dtype=np.int64)
        rc = self._lib.oracle_stats_plan(rows, fan_in, max_rows, ctypes.addressof(k),
                                         ctypes.addressof(e), lv.ctypes.data)
        if rc != 0:
            return None
        return k.value, e.value, [int(x) for x in lv[:k.value]]

    def clip_decision(self, sum_sq: float, nonfinite: int, max_grad_norm: float):
        skip = ctypes.c_int()
        norm = ctypes.c_double()
        coef = ctypes.c_double()
        self._lib.oracle_clip_decision(sum_sq, nonfinite, max_grad_norm, ctypes.addressof(skip),
                                       ctypes.addressof(norm), ctypes.addressof(coef))
        return bool(skip.value), norm.value, coef.value


_DEFAULT: Optional[OracleLib] = None


def lib() -> OracleLib:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = OracleLib()
    return _DEFAULT


@dataclasses.dataclass
class OracleState:
    """Optimizer state: the step count t and the moment arrays (None before step 1)."""
    t: int = 0
    m: Optional[np.ndarray] = None
    v: Optional[np.ndarray] = None
    vmax: Optional[np.ndarray] = None


class OracleAdamW:
    """Host control flow around one oracle update, on FP32-stored (or FP64) state.

    ``storage`` = "f32" keeps parameters and moments in FP32 between calls, as
    the device does; "f64" keeps them in FP64 (used by the closed-form pins).
    """

    def __init__(self, p0: np.ndarray, opts: dict, storage: str = "f32",
                 lib_: Optional[OracleLib] = None):
        self.lib = lib_ or lib()
        self.opts = dict(opts)
        self.storage = storage
        self.p = np.array(p0, dtype=np.float32 if storage == "f32" else np.float64)
        self.state = OracleState()

    def step(self, g: np.ndarray, dtype: str, gradient_scale: float = 1.0,
             skip_update: bool = False, clip_coef: float = 1.0) -> bool:
        """Returns True when an update ran (False for skip or an empty tensor)."""
        n = self.p.size
        if n == 0 or skip_update:
            return False
        t = self.state.t + 1
        have = self.state.t > 0
        f64 = lambda a: np.array(a, dtype=np.float64) if a is not None else np.zeros(n)  # noqa
        p, m, v = f64(self.p), f64(self.state.m), f64(self.state.v)
        vmax = f64(self.state.vmax) if self.opts["amsgrad"] else np.zeros(n)
        self.lib.update(g, dtype, self.opts, gradient_scale, clip_coef, t, have,
                        self.storage == "f32", p, m, v, vmax)
        dt = np.float32 if self.storage == "f32" else np.float64
        self.p = p.astype(dt)
        self.state = OracleState(t=t, m=m.astype(dt), v=v.astype(dt),
                                 vmax=vmax.astype(dt) if self.opts["amsgrad"] else None)
        return True
