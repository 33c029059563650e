"""A torch.optim-style optimizer over the fused step, and a matching GradScaler.

Follows "训练与状态保存" (zh/docs/training), section "在 ruda:0 上进行原生 PyTorch 训练":
an AdamW whose fused path reads back a 12-byte gradient report before updating,
skips the whole step on any non-finite gradient, optionally clips by the global
L2 norm of the unscaled gradient over every active parameter group
(``max_grad_norm``; clipping requires the fused step), keeps ``.grad``, keeps
master parameters and moments in FP32, and is used with a GradScaler as
``scaler.scale(loss).backward(); scaler.step(opt); scaler.update()``.  Its
state_dict keeps ``fused_step`` and ``max_grad_norm`` and uses step-options
version 2 when hierarchical statistics are on; an older state_dict without
these options restores with the fused / hierarchical modes off.

GB300 layout: every parameter group is packed into one contiguous bucket.  The
parameters (or, for BF16/FP16 parameters, an FP32 master copy) and their
gradients become views into flat device buffers, so a step is one analysis and
one update launch per group over the whole bucket (the pages launch one update
per active parameter).  Elements of one launch share the group's options and step
count, as a pre-flattened bucket must ("実験的なデバイス上の融合 AdamW / AMSGrad",
section "サポートされている契約").  Each parameter keeps its own step count: a
parameter whose ``.grad`` is None is inactive, is not updated and does not advance,
as in torch.optim; the update then covers each run of consecutive active
parameters with equal counts in one launch.  All arithmetic runs in the library's
kernels; this module only allocates buffers and calls the C ABI.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import (FaStats, fa_analyze_gradient, fa_bucket_step, fa_bucket_update,
               fa_clip_decision, fa_stats_sum_sq, fa_merge_gradient_stats,
               fa_read_report, fa_stats_rows, options, control, scratch_buffer, stats_buffer)
from . import sharded

MAX_ROWS = 4_194_304
STEP_OPTIONS_VERSION_HIERARCHICAL = 2
STEP_OPTIONS_VERSION_PLAIN = 1


def active_runs(active: list[bool], steps: list[int], offsets: list[int],
                n: int) -> list[tuple[int, int, int, int]]:
    """Maximal runs of consecutive active parameters with equal step counts, as
    (first parameter, end parameter, first element, end element): each run is one
    update launch over a contiguous slice of the bucket, and when every parameter is
    active with one step count (the usual case) the single run is the whole bucket.
    A run ends at the next parameter's offset, so it includes its alignment padding."""
    out = []
    i = 0
    count = len(active)
    while i < count:
        if not active[i]:
            i += 1
            continue
        j = i + 1
        while j < count and active[j] and steps[j] == steps[i]:
            j += 1
        out.append((i, j, offsets[i], offsets[j] if j < count else n))
        i = j
    return out


class _Bucket:
    """Flat device buffers of one parameter group."""

    def __init__(self, params: list[torch.Tensor], amsgrad: bool):
        dev = params[0].device
        if dev.type != "cuda":
            raise ValueError("FusedAdamW needs CUDA parameters (there is no CPU path)")
        if any(p.device != dev for p in params):
            raise ValueError("a parameter group must hold parameters of one CUDA device")
        dtypes = {p.dtype for p in params}
        if len(dtypes) != 1 or not dtypes <= {torch.float32, torch.float16, torch.bfloat16}:
            raise TypeError("a parameter group must hold parameters of one float dtype "
                            "(float32, float16 or bfloat16)")
        self.param_dtype = params[0].dtype
        self.params = params
        sizes = [p.numel() for p in params]
        # segment starts rounded up to 8 elements keep every segment 16-byte aligned
        offs, pos = [], 0
        for sz in sizes:
            offs.append(pos)
            pos += (sz + 7) // 8 * 8
        self.offsets = offs
        self.n = pos
        self.segments = sorted(set(offs + [pos]))
        self.master_separate = self.param_dtype != torch.float32
        self.model = None
        if self.master_separate:
            self.model = torch.zeros(self.n, dtype=self.param_dtype, device=dev)
        self.master = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.grad = torch.zeros(self.n, dtype=self.param_dtype, device=dev)
        self.m = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.v = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.vmax = torch.zeros(self.n, dtype=torch.float32, device=dev) if amsgrad else None
        with torch.no_grad():
            for p, off in zip(params, offs):
                k = p.numel()
                self.master[off:off + k].copy_(p.detach().reshape(-1))
                if self.master_separate:
                    self.model[off:off + k].copy_(p.detach().reshape(-1))
                    p.data = self.model[off:off + k].view_as(p)
                else:
                    p.data = self.master[off:off + k].view_as(p)
                if p.grad is not None:
                    self.grad[off:off + k].copy_(p.grad.reshape(-1))
                p.grad = self.grad[off:off + k].view_as(p)
        # one step count per parameter: a parameter without a gradient is not updated
        # and its count does not advance, as in torch.optim and the pages' adapter
        self.steps = [0] * len(params)

    def view(self, buf: torch.Tensor, i: int) -> torch.Tensor:
        p = self.params[i]
        return buf[self.offsets[i]:self.offsets[i] + p.numel()].view_as(p)

    def gather_grads(self) -> list[bool]:
        """Autograd normally accumulates into the bucket views in place; a gradient
        that was replaced by a new tensor is copied back into the bucket.  Returns
        which parameters are active (have a gradient); an inactive one's slice of the
        bucket gradient is zeroed, so it adds nothing to the statistics."""
        active = []
        with torch.no_grad():
            for i, p in enumerate(self.params):
                mine = self.view(self.grad, i)
                if p.grad is None:
                    mine.zero_()
                    active.append(False)
                    continue
                if p.grad.data_ptr() != mine.data_ptr():
                    mine.copy_(p.grad)
                    p.grad = mine
                active.append(True)
        return active

    def runs(self, active: list[bool]) -> list[tuple[int, int, int, int]]:
        return active_runs(active, self.steps, self.offsets, self.n)

    def slices(self, lo: int, hi: int):
        """(master, grad, m, v, vmax, model) views of elements [lo, hi)."""
        cut = lambda t: None if t is None else t[lo:hi]  # noqa: E731
        return (cut(self.master), cut(self.grad), cut(self.m), cut(self.v), cut(self.vmax),
                cut(self.model))


def statistics_decision(rep, gradient_scale: float, max_grad_norm: float,
                        shard_group=None) -> tuple[bool, float, float]:
    """(skip, norm, clip coefficient) from this process's 12-byte report.

    Without ``shard_group`` the report covers the whole gradient: one process, or
    data-parallel replicas whose gradients were already reduced (each replica's norm is
    the global norm, as with ``torch.nn.utils.clip_grad_norm_``).  With a process group,
    this optimizer's parameters are one rank's shard of the model: the ranks' totals
    are summed in rank order and every rank takes the same decision.
    """
    if shard_group is None:
        s, c = sharded.report_totals(rep)
        return fa_clip_decision(s, c, gradient_scale, max_grad_norm)
    return sharded.global_clip_decision(rep, gradient_scale, max_grad_norm, group=shard_group)


class FusedAdamW(torch.optim.Optimizer):
    """AdamW / AMSGrad on GB300 through the fused step.

    ``step(gradient_scale=..., found_inf=...)``: the stored gradients are divided by
    ``gradient_scale``; ``found_inf`` (an externally computed flag) skips the step.
    With ``max_grad_norm`` set, or ``hierarchical_stats=True``, or when a
    ``GradScaler`` asks for it, the step first analyses every group's gradient,
    merges the statistics (fan-in 1024) and reads back the 12-byte report: a
    non-finite value skips the step, and the global norm sets the clip.

    ``shard_group``: a ``torch.distributed`` process group when each rank's optimizer
    holds a different shard of the model's parameters; the statistics are then summed
    over the group before the decision.  Leave it None for one process or for
    replicas with reduced gradients (the decision is then local, and taken on the
    device).
    """

    def __init__(self, params, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-5,
                 weight_decay: float = 1e-4, amsgrad: bool = False, maximize: bool = False,
                 fused_step: bool = True, max_grad_norm: Optional[float] = None,
                 hierarchical_stats: bool = False, row_len: Optional[int] = None,
                 shard_group=None):
        if not fused_step:
            raise ValueError("FusedAdamW implements the fused step only (fused_step=True)")
        if max_grad_norm is not None and not max_grad_norm > 0:
            raise ValueError("max_grad_norm must be positive or None")
        defaults = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                        amsgrad=amsgrad, maximize=maximize)
        self._buckets = None
        super().__init__(params, defaults)
        self.fused_step = True
        self.max_grad_norm = max_grad_norm
        self.hierarchical_stats = hierarchical_stats
        self.shard_group = shard_group
        self._buckets = [_Bucket(list(g["params"]), g["amsgrad"]) for g in self.param_groups]
        self._row_len_fixed = row_len is not None
        self.row_len = row_len if row_len is not None else self._auto_row_len()
        self._stats = None
        self.last_report: dict = {}
        self._bind_state()

    def add_param_group(self, param_group: dict) -> None:
        """As torch.optim: a group added after construction gets its own bucket (its
        parameters become views into it) and starts at step 0."""
        super().add_param_group(param_group)
        if getattr(self, "_buckets", None) is None:  # called from the constructor
            return
        g = self.param_groups[-1]
        self._buckets.append(_Bucket(list(g["params"]), g["amsgrad"]))
        if not self._row_len_fixed:
            self.row_len = self._auto_row_len()
        self._stats = None
        self._bind_state()

    # ---- state -------------------------------------------------------------------
    def _bind_state(self) -> None:
        """Per-parameter state entries are views into the group buckets."""
        for b in self._buckets:
            for i, p in enumerate(b.params):
                st = {"step": torch.tensor(float(b.steps[i])),
                      "exp_avg": b.view(b.m, i), "exp_avg_sq": b.view(b.v, i)}
                if b.vmax is not None:
                    st["max_exp_avg_sq"] = b.view(b.vmax, i)
                if b.master_separate:
                    st["master_param"] = b.view(b.master, i)
                self.state[p] = st

    def _sync_steps(self) -> None:
        for b in self._buckets:
            for i, p in enumerate(b.params):
                self.state[p]["step"] = torch.tensor(float(b.steps[i]))

    def state_dict(self):
        self._sync_steps()
        sd = super().state_dict()
        sd["fused_options"] = {
            "fused_step": True, "max_grad_norm": self.max_grad_norm,
            "hierarchical_stats": self.hierarchical_stats, "row_len": self.row_len,
            "step_options_version": (STEP_OPTIONS_VERSION_HIERARCHICAL if self.hierarchical_stats
                                     else STEP_OPTIONS_VERSION_PLAIN)}
        return sd

    def load_state_dict(self, state_dict) -> None:
        """Restores hyper-parameters, step counts and moments into the buckets.

        The saved moments are copied as they are (FP32), never cast to the
        parameter dtype.  A record without ``fused_options`` (an older format)
        restores with clipping and hierarchical statistics off.
        """
        fo = state_dict.get("fused_options")
        if fo is None:
            self.max_grad_norm = None
            self.hierarchical_stats = False
        else:
            self.max_grad_norm = fo.get("max_grad_norm")
            self.hierarchical_stats = (bool(fo.get("hierarchical_stats", False))
                                       and int(fo.get("step_options_version", 1))
                                       >= STEP_OPTIONS_VERSION_HIERARCHICAL)
            self.row_len = int(fo.get("row_len", self.row_len))
        saved_groups = state_dict["param_groups"]
        if len(saved_groups) != len(self.param_groups):
            raise ValueError("state_dict has a different number of parameter groups")
        saved_state = state_dict["state"]
        with torch.no_grad():
            for group, saved, b in zip(self.param_groups, saved_groups, self._buckets):
                if len(saved["params"]) != len(group["params"]):
                    raise ValueError("a parameter group has a different size in the state_dict")
                for k, val in saved.items():
                    if k != "params":
                        group[k] = tuple(val) if k == "betas" else val
                for i, idx in enumerate(saved["params"]):
                    st = saved_state.get(idx, {})
                    b.steps[i] = int(float(st.get("step", 0)))
                    for key, buf in (("exp_avg", b.m), ("exp_avg_sq", b.v),
                                     ("max_exp_avg_sq", b.vmax), ("master_param", b.master)):
                        if buf is not None and key in st:
                            b.view(buf, i).copy_(st[key])
        self._bind_state()

    def zero_grad(self, set_to_none: bool = False) -> None:
        """Clears the bucket gradients.  By default ``.grad`` stays the bucket view, so
        backward accumulates in place and every parameter counts as active.  With
        ``set_to_none=True`` every ``.grad`` becomes None, as in torch.optim: a parameter
        that backward then leaves without a gradient is skipped by the next step, at the
        cost of one copy of each new gradient into the bucket."""
        for b in self._buckets:
            b.grad.zero_()
            for i, p in enumerate(b.params):
                p.grad = None if set_to_none else b.view(b.grad, i)

    # ---- the step ------------------------------------------------------------------
    def _stats_buffers(self):
        total = sum(self._rows(b) for b in self._buckets)
        if total > MAX_ROWS:
            raise ValueError(f"{total} statistics rows exceed the plan maximum {MAX_ROWS}; "
                             f"use a larger row_len")
        if self._stats is None or self._stats[0] != total:
            dev = self._buckets[0].master.device
            self._stats = (total, stats_buffer(total, dev), scratch_buffer(total, dev),
                           stats_buffer(1, dev))
        return self._stats

    def _auto_row_len(self) -> int:
        """Smallest 256 * 2^k whose rows over every bucket fit the statistics plan."""
        row_len = 256
        while sum(fa_stats_rows(b.n, row_len, b.segments) for b in self._buckets) > MAX_ROWS:
            row_len *= 2
        return row_len

    def _rows(self, b: _Bucket) -> int:
        return fa_stats_rows(b.n, self.row_len, b.segments)

    def _enqueue_statistics(self) -> torch.Tensor:
        """Analyses every group and merges into the one 12-byte device report."""
        total, rows_buf, scratch, report = self._stats_buffers()
        off = 0
        for b in self._buckets:
            r = self._rows(b)
            fa_analyze_gradient(b.grad, self.row_len, rows_buf[off:off + r], b.segments)
            off += r
        fa_merge_gradient_stats(rows_buf, total, scratch, report)
        return report

    def statistics(self, gradient_scale: float = 1.0):
        """Analyse every group, merge, read back: (skip, global norm, clip coefficient,
        non-finite count), over every shard of ``shard_group`` when one is set."""
        rep = fa_read_report(self._enqueue_statistics())
        skip, norm, coef = statistics_decision(
            rep, gradient_scale, self.max_grad_norm if self.max_grad_norm else 0.0,
            self.shard_group)
        return skip, norm, coef, int(rep.nonfinite)

    @torch.no_grad()
    def step(self, closure=None, gradient_scale: float = 1.0, found_inf: bool = False,
             check_finite: bool = False):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        active = [b.gather_grads() for b in self._buckets]
        report = {"skipped": bool(found_inf), "nonfinite": 0, "grad_norm": None, "clip_coef": 1.0}
        use_stats = not found_inf and (self.max_grad_norm is not None or self.hierarchical_stats
                                       or check_finite)
        if use_stats and self._can_gate():
            self.last_report = self._gated_step(gradient_scale, active)
            return loss
        if use_stats:
            skip, norm, coef, bad = self.statistics(gradient_scale)
            report.update(skipped=skip, nonfinite=bad, grad_norm=norm, clip_coef=coef)
        if not report["skipped"]:
            ctl = control(gradient_scale)
            for group, b, act in zip(self.param_groups, self._buckets, active):
                o = self._options(group)
                for i, j, lo, hi in b.runs(act):
                    pm, g, m, v, vm, model = b.slices(lo, hi)
                    if b.master_separate:
                        fa_bucket_update(None, pm, g, m, v, vm, b.steps[i], o, ctl,
                                         grad_mult=report["clip_coef"], p_model=model)
                    else:
                        fa_bucket_step(None, pm, g, m, v, vm, b.steps[i], o, ctl,
                                       report["clip_coef"])
                    for k in range(i, j):
                        b.steps[k] += 1
        self.last_report = report
        return loss

    def _options(self, group):
        return options(lr=group["lr"], beta1=group["betas"][0], beta2=group["betas"][1],
                       eps=group["eps"], weight_decay=group["weight_decay"],
                       amsgrad=group["amsgrad"], maximize=group["maximize"])

    def _can_gate(self) -> bool:
        """The device can take the decision itself when this process holds the whole
        gradient; shards need every rank's totals first."""
        return self.shard_group is None

    def _gated_step(self, gradient_scale: float, active: list[list[bool]]) -> dict:
        """Statistics, then every group's update gated on the device by the same report
        (bit-identical to deciding on the host), while the host reads the report back
        through pinned memory to advance the step counts."""
        report_dev = self._enqueue_statistics()
        if getattr(self, "_pinned_report", None) is None:
            self._pinned_report = torch.empty((1, 3), dtype=torch.int32).pin_memory()
            self._report_event = torch.cuda.Event()
        stream = torch.cuda.current_stream(report_dev.device)
        self._pinned_report.copy_(report_dev, non_blocking=True)
        self._report_event.record(stream)
        ctl = control(gradient_scale)
        max_norm = self.max_grad_norm if self.max_grad_norm else 0.0
        launched = []
        for group, b, act in zip(self.param_groups, self._buckets, active):
            o = self._options(group)
            for i, j, lo, hi in b.runs(act):
                pm, g, m, v, vm, model = b.slices(lo, hi)
                if b.master_separate:
                    fa_bucket_update(None, pm, g, m, v, vm, b.steps[i], o, ctl,
                                     report=report_dev, max_grad_norm=max_norm, p_model=model)
                else:
                    fa_bucket_update(None, pm, g, m, v, vm, b.steps[i], o, ctl,
                                     report=report_dev, max_grad_norm=max_norm)
                launched.append((b, i, j))
        self._report_event.synchronize()
        rep = FaStats.from_buffer_copy(self._pinned_report.numpy().tobytes())
        total = fa_stats_sum_sq(rep)
        skip, norm, coef = fa_clip_decision(total, int(rep.nonfinite), gradient_scale, max_norm)
        if not skip:
            for b, i, j in launched:
                for k in range(i, j):
                    b.steps[k] += 1
        return {"skipped": skip, "nonfinite": int(rep.nonfinite), "grad_norm": norm,
                "clip_coef": coef}


class GradScaler:
    """Dynamic loss scaling for FusedAdamW.

    ``scale(loss)`` multiplies the loss; ``step(opt)`` runs the optimizer with
    ``gradient_scale`` = the current scale and the finiteness check of the fused
    statistics (no separate gradient scan); ``update()`` halves the scale after a
    skipped step and doubles it after ``growth_interval`` clean steps.
    """

    def __init__(self, init_scale: float = 2.0 ** 16, growth_factor: float = 2.0,
                 backoff_factor: float = 0.5, growth_interval: int = 2000):
        self._scale = float(init_scale)
        self.growth_factor = growth_factor
        self.backoff_factor = backoff_factor
        self.growth_interval = growth_interval
        self._good = 0
        self._last_skipped: Optional[bool] = None

    def get_scale(self) -> float:
        return self._scale

    def scale(self, loss: torch.Tensor) -> torch.Tensor:
        return loss * self._scale

    def step(self, optimizer: FusedAdamW, *args, **kwargs):
        out = optimizer.step(*args, gradient_scale=self._scale, check_finite=True, **kwargs)
        self._last_skipped = bool(optimizer.last_report["skipped"])
        return out

    def update(self) -> None:
        if self._last_skipped is None:
            return
        if self._last_skipped:
            self._scale *= self.backoff_factor
            self._good = 0
        else:
            self._good += 1
            if self._good >= self.growth_interval:
                self._scale *= self.growth_factor
                self._good = 0
        self._last_skipped = None

    def state_dict(self) -> dict:
        return {"scale": self._scale, "growth_factor": self.growth_factor,
                "backoff_factor": self.backoff_factor, "growth_interval": self.growth_interval,
                "good_steps": self._good}

    def load_state_dict(self, sd: dict) -> None:
        self._scale = float(sd["scale"])
        self.growth_factor = sd["growth_factor"]
        self.backoff_factor = sd["backoff_factor"]
        self.growth_interval = sd["growth_interval"]
        self._good = int(sd["good_steps"])
