"""GB300 fused AdamW / AMSGrad step: thin Python binding of ``libfused_adamw.so``.

Every function here marshals torch tensors into the C ABI of
``include/fused_adamw.h`` under the same name; all arithmetic runs in the CUDA
kernels of the library.  PyTorch supplies device memory and streams only.
Layout checks that raw pointers cannot express (contiguity, strides, dtype,
device) are made here, as the adapter's job ("実験的なデバイス上の融合 AdamW /
AMSGrad", section "ネイティブ PyTorch ストレージと階層統計": the adapter validates
shape, alias, lifetime and queue).
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import (FA_BF16, FA_F16, FA_F32, FaOptions, FaStats, FaStepControl,  # noqa: F401
                   FaStepReport, FusedAdamWError, check)

__all__ = [
    "fa_abi_version", "fa_device_error", "fa_bounds_check_report", "fa_pipeline_selftest",
    "fa_options_default", "fa_step_coefficients", "fa_adamw_step", "fa_adamw_step_inplace",
    "fa_bucket_step", "fa_bucket_update", "fa_adamw_step_staged", "fa_stats_plan",
    "fa_stats_rows", "fa_analyze_gradient", "fa_merge_gradient_stats",
    "fa_merge_gradient_stats_static", "fa_read_report", "fa_stats_sum_sq", "fa_clip_decision",
    "fa_stats_chunk_scratch", "fa_merge_gradient_stats_chunks",
    "fa_bucket_step_clipped_per_segment", "fa_bucket_step_clipped_per_segment_gated",
    "segment_rows", "fa_clip_decide", "fa_bucket_step_clipped", "fa_bucket_step_clipped_gated",
    "report_mailbox", "options", "control", "stats_buffer", "scratch_buffer",
    "FusedAdamWError", "FaStats", "FaStepReport", "bytes_per_param",
]

_TORCH_GRAD = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}
STATS_WORDS = 3  # a 12-byte record is three 32-bit words


def _L():
    return _lib.load()


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dense(name: str, t: torch.Tensor, n: int, dtypes, device=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.layout != torch.strided:
        raise ValueError(f"{name}: sparse or non-strided tensors are not supported")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous() or (t.numel() > 1 and 0 in t.stride()):
        raise ValueError(f"{name}: must be dense and contiguous (no strides, no broadcast)")
    if t.numel() != n:
        raise ValueError(f"{name}: {t.numel()} elements, expected {n}")
    if device is not None and t.numel() and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


def options(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=1e-4, amsgrad=False,
            maximize=False) -> FaOptions:
    return FaOptions(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                     int(bool(amsgrad)), int(bool(maximize)))


def control(gradient_scale: float = 1.0, skip_update: bool = False) -> FaStepControl:
    return FaStepControl(float(gradient_scale), int(bool(skip_update)))


def bytes_per_param(grad_bytes: int, amsgrad: bool, first_step: bool) -> int:
    """Algorithmic HBM bytes one update moves per parameter.

    FP32 parameter read and write; gradient read; m and v written, and read
    unless this is the first step; AMSGrad adds the max state the same way
    ("実験的なデバイス上の融合 AdamW / AMSGrad", section "割り当てとパフォーマンスのモデル":
    28 bytes = 4 FP32 reads + 3 FP32 writes for an FP32 gradient).
    """
    states = 3 if amsgrad else 2
    reads = 4 + grad_bytes + (0 if first_step else 4 * states)
    writes = 4 + 4 * states
    return reads + writes


# ---- host-only -----------------------------------------------------------------

def fa_abi_version() -> int:
    return _L().fa_abi_version()


def fa_device_error(clear: bool = False) -> int:
    """1 when an update kernel's bounded pipeline wait gave up on this device."""
    v = ctypes.c_int32()
    check("fa_device_error", _L().fa_device_error(ctypes.byref(v), int(bool(clear))))
    return v.value


def fa_bounds_check_report(clear: bool = False) -> tuple[bool, int]:
    """(checked build?, out-of-range accesses counted and skipped since the last clear)."""
    en = ctypes.c_int32()
    n = ctypes.c_uint64()
    check("fa_bounds_check_report",
          _L().fa_bounds_check_report(ctypes.byref(en), ctypes.byref(n), int(bool(clear))))
    return bool(en.value), int(n.value)


def fa_pipeline_selftest(p, g, m, v, stream=None) -> int:
    """Runs the bounded-wait self-test on these buffers; returns the flag (1 expected)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    flag = ctypes.c_int32()
    check("fa_pipeline_selftest", _L().fa_pipeline_selftest(
        n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), ctypes.byref(flag),
        _stream(stream)))
    return flag.value


def fa_options_default() -> FaOptions:
    return _L().fa_options_default()


def fa_step_coefficients(opts: FaOptions, t: int, gradient_scale: float = 1.0,
                         grad_mult: float = 1.0) -> list[float]:
    out = (ctypes.c_float * 9)()
    check("fa_step_coefficients",
          _L().fa_step_coefficients(ctypes.byref(opts), t, gradient_scale, grad_mult, out))
    return list(out)


def fa_stats_plan(rows: int) -> tuple[int, int]:
    k = ctypes.c_int32()
    e = ctypes.c_int64()
    check("fa_stats_plan", _L().fa_stats_plan(rows, ctypes.byref(k), ctypes.byref(e)))
    return k.value, e.value


def _segments(seg_offsets: Optional[Sequence[int]]):
    if seg_offsets is None:
        return None, 0
    arr = (ctypes.c_int64 * len(seg_offsets))(*[int(x) for x in seg_offsets])
    return arr, len(seg_offsets) - 1


def fa_stats_rows(n: int, row_len: int, seg_offsets: Optional[Sequence[int]] = None) -> int:
    seg, nseg = _segments(seg_offsets)
    r = ctypes.c_int64()
    check("fa_stats_rows", _L().fa_stats_rows(n, row_len, seg, nseg, ctypes.byref(r)))
    return r.value


def fa_stats_sum_sq(record: FaStats) -> float:
    """The sum of squares a 12-byte record stands for (either of its two forms)."""
    out = ctypes.c_double()
    check("fa_stats_sum_sq", _L().fa_stats_sum_sq(ctypes.byref(record), ctypes.byref(out)))
    return out.value


def fa_clip_decision(sum_sq_stored: float, nonfinite: int, gradient_scale: float,
                     max_grad_norm: float) -> tuple[bool, float, float]:
    s = ctypes.c_int32()
    nrm = ctypes.c_double()
    c = ctypes.c_double()
    check("fa_clip_decision",
          _L().fa_clip_decision(sum_sq_stored, nonfinite, gradient_scale, max_grad_norm,
                                ctypes.byref(s), ctypes.byref(nrm), ctypes.byref(c)))
    return bool(s.value), nrm.value, c.value


# ---- the update ------------------------------------------------------------------

def fa_adamw_step(p: torch.Tensor, g: torch.Tensor, m: Optional[torch.Tensor],
                  v: Optional[torch.Tensor], vmax: Optional[torch.Tensor], t: int,
                  opts: FaOptions, ctl: FaStepControl, stream=None):
    """Out-of-place step.  Returns (p, m, v, vmax, t, updated).

    Skip and empty steps allocate nothing and return the inputs unchanged.
    """
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    for name, x in (("m", m), ("v", v), ("vmax", vmax)):
        if x is not None:
            _dense(name, x, n, (torch.float32,), p.device)
    if n == 0 or ctl.skip_update:
        # the library still validates; no output buffer is allocated
        tout, upd = ctypes.c_uint64(), ctypes.c_int32()
        check("fa_adamw_step", _L().fa_adamw_step(
            n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax), t,
            ctypes.byref(opts), ctl, None, None, None, None, ctypes.byref(tout),
            ctypes.byref(upd), _stream(stream)))
        return p, m, v, vmax, tout.value, False
    p_out = torch.empty_like(p)
    m_out = torch.empty_like(p)
    v_out = torch.empty_like(p)
    vmax_out = torch.empty_like(p) if opts.amsgrad else None
    tout, upd = ctypes.c_uint64(), ctypes.c_int32()
    check("fa_adamw_step", _L().fa_adamw_step(
        n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax), t,
        ctypes.byref(opts), ctl, _ptr(p_out), _ptr(m_out), _ptr(v_out), _ptr(vmax_out),
        ctypes.byref(tout), ctypes.byref(upd), _stream(stream)))
    return p_out, m_out, v_out, vmax_out, tout.value, bool(upd.value)


def fa_adamw_step_inplace(p, g, m, v, vmax, t: int, opts: FaOptions, ctl: FaStepControl,
                          grad_mult: float = 1.0, stream=None) -> tuple[int, bool]:
    """In-place step on preallocated storage.  Returns (t, updated)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    tt, upd = ctypes.c_uint64(t), ctypes.c_int32()
    check("fa_adamw_step_inplace", _L().fa_adamw_step_inplace(
        n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, grad_mult, ctypes.byref(upd),
        _stream(stream)))
    return tt.value, bool(upd.value)


def fa_bucket_step(seg_offsets, p, g, m, v, vmax, t: int, opts: FaOptions, ctl: FaStepControl,
                   grad_mult: float = 1.0, stream=None) -> tuple[int, bool]:
    """One update launch over a pre-flattened bucket.  Returns (t, updated)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    seg, nseg = _segments(seg_offsets)
    tt, upd = ctypes.c_uint64(t), ctypes.c_int32()
    check("fa_bucket_step", _L().fa_bucket_step(
        seg, nseg, n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, grad_mult, ctypes.byref(upd),
        _stream(stream)))
    return tt.value, bool(upd.value)


def fa_bucket_update(seg_offsets, p, g, m, v, vmax, t: int, opts: FaOptions,
                     ctl: FaStepControl, *, grad_mult: float = 1.0,
                     seg_grad_mult: Optional[Sequence[float]] = None,
                     report: Optional[torch.Tensor] = None,
                     seg_reports: Optional[torch.Tensor] = None, max_grad_norm: float = 0.0,
                     p_model: Optional[torch.Tensor] = None,
                     seg_decided: Optional[torch.Tensor] = None, stream=None) -> bool:
    """One update of a pre-flattened bucket in any variant (the fa_bucket_update_args record):
    a host multiplier (``grad_mult``, or ``seg_grad_mult`` per segment) or the decision on
    the device from ``report`` / ``seg_reports`` with ``max_grad_norm``, and optionally the
    BF16/FP16 model copy ``p_model``.  ``seg_decided`` (FP32 device scratch of at least
    nseg + 1 elements, with ``seg_reports``): where every segment's decision is taken once
    before the update.  The update is step t + 1; t is not changed.
    Returns True when an update kernel was enqueued."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    if p_model is not None:
        _dense("p_model", p_model, n, (torch.float16, torch.bfloat16), p.device)
    if report is not None:
        _stats_tensor("report", report)
    if seg_decided is not None:
        _dense("seg_decided", seg_decided, seg_decided.numel(), (torch.float32,), p.device)
    seg, nseg = _segments(seg_offsets)
    if seg_reports is not None:
        _stats_tensor("seg_reports", seg_reports)
        if seg_reports.shape[0] < nseg:
            raise ValueError(f"seg_reports: {seg_reports.shape[0]} records for {nseg} segments")
    mult = None
    if seg_grad_mult is not None:
        if len(seg_grad_mult) != nseg:
            raise ValueError("one multiplier per segment")
        mult = (ctypes.c_double * nseg)(*[float(x) for x in seg_grad_mult])
    u = _lib.FaBucketUpdate(
        seg_offsets=seg, nseg=nseg, n_total=n, p=_ptr(p), g=_ptr(g), gdt=_TORCH_GRAD[g.dtype],
        m=_ptr(m), v=_ptr(v), vmax=_ptr(vmax), t=t, grad_mult=grad_mult, seg_grad_mult=mult,
        report=_ptr(report), seg_reports=_ptr(seg_reports), max_grad_norm=max_grad_norm,
        p_model=_ptr(p_model),
        model_dtype=_TORCH_GRAD[p_model.dtype] if p_model is not None else FA_BF16,
        seg_decided=_ptr(seg_decided),
        seg_decided_elements=seg_decided.numel() if seg_decided is not None else 0)
    enq = ctypes.c_int32()
    check("fa_bucket_update", _L().fa_bucket_update(ctypes.byref(u), ctypes.byref(opts), ctl,
                                                    ctypes.byref(enq), _stream(stream)))
    return bool(enq.value)


def fa_adamw_step_staged(p, g, m, v, vmax, t: int, opts: FaOptions, ctl: FaStepControl,
                         delta: torch.Tensor, grad_mult: float = 1.0,
                         stream=None) -> tuple[int, bool]:
    """The 4/5-kernel staged comparison (benchmarks only).  Returns (t, updated)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    _dense("delta", delta, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    tt, upd = ctypes.c_uint64(t), ctypes.c_int32()
    check("fa_adamw_step_staged", _L().fa_adamw_step_staged(
        n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, grad_mult, _ptr(delta), ctypes.byref(upd),
        _stream(stream)))
    return tt.value, bool(upd.value)


def report_mailbox() -> torch.Tensor:
    """A report mailbox (fa_report_mailbox: the 12-byte report and a sequence word) in
    pinned host memory, as int32 [4]; one per caller thread, reused across calls."""
    return torch.zeros(4, dtype=torch.int32).pin_memory()


def _check_mailbox(mailbox) -> None:
    if (not isinstance(mailbox, torch.Tensor) or mailbox.device.type != "cpu"
            or mailbox.nbytes < 16 or not mailbox.is_contiguous() or not mailbox.is_pinned()):
        raise ValueError("mailbox: expected a pinned, contiguous host tensor of 16 bytes")


def fa_bucket_step_clipped_gated(seg_offsets, p, g, m, v, vmax, t: int, opts: FaOptions,
                                 ctl: FaStepControl, max_grad_norm: float, row_len: int,
                                 rows_buf: torch.Tensor, scratch: Optional[torch.Tensor],
                                 report: torch.Tensor, mailbox: torch.Tensor,
                                 stream=None) -> tuple[int, FaStepReport]:
    """The statistics-guarded step with the update gated on the device; the report
    comes back through ``mailbox`` (see ``report_mailbox``).  Returns (t, report)."""
    _check_mailbox(mailbox)
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    _stats_tensor("rows_buf", rows_buf)
    _stats_tensor("report", report)
    seg, nseg = _segments(seg_offsets)
    tt = ctypes.c_uint64(t)
    rep = FaStepReport()
    check("fa_bucket_step_clipped_gated", _L().fa_bucket_step_clipped_gated(
        seg, nseg, n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, max_grad_norm, row_len, _ptr(rows_buf),
        rows_buf.shape[0], _ptr(scratch), 0 if scratch is None else scratch.numel(),
        _ptr(report), _ptr(mailbox), ctypes.byref(rep), _stream(stream)))
    return tt.value, rep


# ---- statistics ------------------------------------------------------------------

def stats_buffer(rows: int, device) -> torch.Tensor:
    """Device buffer of ``rows`` 12-byte records, as int32 [rows, 3]."""
    return torch.empty((max(rows, 1), STATS_WORDS), dtype=torch.int32, device=device)


def scratch_buffer(rows: int, device) -> torch.Tensor:
    """Device scratch (FP32 elements) for merging ``rows`` records."""
    _, e = fa_stats_plan(rows)
    return torch.empty(max(e, 1), dtype=torch.float32, device=device)


def _stats_tensor(name, t):
    if t.dtype != torch.int32 or t.dim() != 2 or t.shape[1] != STATS_WORDS or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous int32 [rows, 3] stats buffer")


def fa_analyze_gradient(g: torch.Tensor, row_len: int, rows_out: torch.Tensor,
                        seg_offsets: Optional[Sequence[int]] = None, stream=None) -> int:
    """Per-row statistics of ``g`` into ``rows_out``.  Returns the row count."""
    _dense("g", g, g.numel(), tuple(_TORCH_GRAD))
    _stats_tensor("rows_out", rows_out)
    seg, nseg = _segments(seg_offsets)
    rows = fa_stats_rows(g.numel(), row_len, seg_offsets)
    check("fa_analyze_gradient", _L().fa_analyze_gradient(
        _ptr(g), _TORCH_GRAD[g.dtype], g.numel(), row_len, seg, nseg, _ptr(rows_out),
        rows_out.shape[0], _stream(stream)))
    return rows


def fa_merge_gradient_stats(rows_in: torch.Tensor, rows: int, scratch: Optional[torch.Tensor],
                            report: torch.Tensor, stream=None) -> None:
    _stats_tensor("rows_in", rows_in)
    _stats_tensor("report", report)
    if scratch is not None and (scratch.dtype != torch.float32 or not scratch.is_contiguous()):
        raise ValueError("scratch: expected contiguous float32")
    check("fa_merge_gradient_stats", _L().fa_merge_gradient_stats(
        _ptr(rows_in), rows, _ptr(scratch), 0 if scratch is None else scratch.numel(),
        _ptr(report), _stream(stream)))


def fa_merge_gradient_stats_static(rows_in: torch.Tensor, rows: int, report: torch.Tensor,
                                   stream=None) -> None:
    """Merge into ``report`` using the library's fixed scratch (allocates nothing).

    For callers that cannot allocate device memory; calls on streams that are
    not ordered with each other race on the shared scratch.
    """
    _stats_tensor("rows_in", rows_in)
    _stats_tensor("report", report)
    check("fa_merge_gradient_stats_static", _L().fa_merge_gradient_stats_static(
        _ptr(rows_in), rows, _ptr(report), _stream(stream)))


def fa_stats_chunk_scratch(chunk_rows: Sequence[int]) -> int:
    arr = (ctypes.c_int64 * len(chunk_rows))(*[int(x) for x in chunk_rows])
    e = ctypes.c_int64()
    check("fa_stats_chunk_scratch",
          _L().fa_stats_chunk_scratch(arr, len(chunk_rows) - 1, ctypes.byref(e)))
    return e.value


def segment_rows(seg_offsets: Sequence[int], row_len: int) -> list[int]:
    """Row offsets of each segment's statistics rows (rows never span segments)."""
    out = [0]
    for a, b in zip(seg_offsets[:-1], seg_offsets[1:]):
        out.append(out[-1] + (int(b) - int(a) + row_len - 1) // row_len)
    return out


def fa_merge_gradient_stats_chunks(rows_in: torch.Tensor, chunk_rows: Sequence[int],
                                   scratch: torch.Tensor, chunk_reports: torch.Tensor,
                                   stream=None) -> None:
    _stats_tensor("rows_in", rows_in)
    _stats_tensor("chunk_reports", chunk_reports)
    arr = (ctypes.c_int64 * len(chunk_rows))(*[int(x) for x in chunk_rows])
    check("fa_merge_gradient_stats_chunks", _L().fa_merge_gradient_stats_chunks(
        _ptr(rows_in), arr, len(chunk_rows) - 1, _ptr(scratch), scratch.numel(),
        _ptr(chunk_reports), _stream(stream)))


def fa_bucket_step_clipped_per_segment(seg_offsets, p, g, m, v, vmax, t: int, opts: FaOptions,
                                       ctl: FaStepControl, max_grad_norm: float, row_len: int,
                                       rows_buf: torch.Tensor, scratch: torch.Tensor,
                                       seg_reports: torch.Tensor, stream=None):
    """Per-parameter clipped step.  Returns (t, report, segment norms, coefficients)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    _stats_tensor("rows_buf", rows_buf)
    _stats_tensor("seg_reports", seg_reports)
    seg, nseg = _segments(seg_offsets)
    norms = (ctypes.c_double * nseg)()
    coefs = (ctypes.c_double * nseg)()
    tt = ctypes.c_uint64(t)
    rep = FaStepReport()
    check("fa_bucket_step_clipped_per_segment", _L().fa_bucket_step_clipped_per_segment(
        seg, nseg, n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, max_grad_norm, row_len, _ptr(rows_buf),
        rows_buf.shape[0], _ptr(scratch), scratch.numel(), _ptr(seg_reports), norms, coefs,
        ctypes.byref(rep), _stream(stream)))
    return tt.value, rep, list(norms), list(coefs)


def fa_bucket_step_clipped_per_segment_gated(seg_offsets, p, g, m, v, vmax, t: int,
                                             opts: FaOptions, ctl: FaStepControl,
                                             max_grad_norm: float, row_len: int,
                                             rows_buf: torch.Tensor, scratch: torch.Tensor,
                                             seg_reports: torch.Tensor,
                                             mailbox: Optional[torch.Tensor] = None,
                                             stream=None) -> None:
    """Enqueues analysis, per-segment merges and the device-decided per-segment update.
    When ``scratch`` holds nseg + 1 elements, the decisions are taken there once (its
    contents are scratch either way).  Without ``mailbox`` nothing is read back: the
    caller reads ``seg_reports`` and advances t.  With a mailbox (``report_mailbox()``)
    the call returns once the bucket's record is posted there (its count decides the
    skip; ``fa_stats_sum_sq`` of it is the total sum of squares), while the update may
    still run."""
    if mailbox is not None:
        _check_mailbox(mailbox)
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    _stats_tensor("rows_buf", rows_buf)
    _stats_tensor("seg_reports", seg_reports)
    seg, nseg = _segments(seg_offsets)
    if seg_reports.shape[0] < nseg:
        raise ValueError(f"seg_reports: {seg_reports.shape[0]} records for {nseg} segments")
    check("fa_bucket_step_clipped_per_segment_gated",
          _L().fa_bucket_step_clipped_per_segment_gated(
              seg, nseg, n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v),
              _ptr(vmax), t, ctypes.byref(opts), ctl, max_grad_norm, row_len, _ptr(rows_buf),
              rows_buf.shape[0], _ptr(scratch), scratch.numel(), _ptr(seg_reports),
              _ptr(mailbox), _stream(stream)))


def fa_read_report(report: torch.Tensor, stream=None) -> FaStats:
    _stats_tensor("report", report)
    h = FaStats()
    check("fa_read_report", _L().fa_read_report(_ptr(report), ctypes.byref(h), _stream(stream)))
    return h


def fa_clip_decide(report: torch.Tensor, gradient_scale: float, max_grad_norm: float,
                   stream=None) -> tuple[bool, float, float]:
    _stats_tensor("report", report)
    s = ctypes.c_int32()
    nrm = ctypes.c_double()
    c = ctypes.c_double()
    check("fa_clip_decide", _L().fa_clip_decide(
        _ptr(report), gradient_scale, max_grad_norm, ctypes.byref(s), ctypes.byref(nrm),
        ctypes.byref(c), _stream(stream)))
    return bool(s.value), nrm.value, c.value


def fa_bucket_step_clipped(seg_offsets, p, g, m, v, vmax, t: int, opts: FaOptions,
                           ctl: FaStepControl, max_grad_norm: float, row_len: int,
                           rows_buf: torch.Tensor, scratch: Optional[torch.Tensor],
                           report: torch.Tensor, stream=None) -> tuple[int, FaStepReport]:
    """Analyse, merge, read back, decide, then update or skip.  Returns (t, report)."""
    n = p.numel()
    _dense("p", p, n, (torch.float32,))
    _dense("g", g, n, tuple(_TORCH_GRAD), p.device)
    _dense("m", m, n, (torch.float32,), p.device)
    _dense("v", v, n, (torch.float32,), p.device)
    if vmax is not None:
        _dense("vmax", vmax, n, (torch.float32,), p.device)
    _stats_tensor("rows_buf", rows_buf)
    _stats_tensor("report", report)
    seg, nseg = _segments(seg_offsets)
    tt = ctypes.c_uint64(t)
    rep = FaStepReport()
    check("fa_bucket_step_clipped", _L().fa_bucket_step_clipped(
        seg, nseg, n, _ptr(p), _ptr(g), _TORCH_GRAD[g.dtype], _ptr(m), _ptr(v), _ptr(vmax),
        ctypes.byref(tt), ctypes.byref(opts), ctl, max_grad_norm, row_len, _ptr(rows_buf),
        rows_buf.shape[0], _ptr(scratch), 0 if scratch is None else scratch.numel(),
        _ptr(report), ctypes.byref(rep), _stream(stream)))
    return tt.value, rep
