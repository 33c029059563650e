"""Runs a seeded workload through the C ABI on the GPU and checks it against the oracle.

Two comparisons per call:

* one step from identical state: the oracle takes the device's own state from
  just before the call (at the checked indices) and the clip coefficient the
  device used, and must agree with the device after the call within
  |d| <= 1e-6 * max(1, |x|) AND within an error bound derived from FP32
  rounding of the update's arithmetic (``tight_bound``);
* trajectory: an oracle run that never sees device values (its own state, its
  own clip decision from the full gradient) must agree within
  |d| <= 1e-5 * max(1, |x|).

Non-finite counts, skip decisions and the step count must match exactly; the
gradient norm within relative 1e-5.
"""

from __future__ import annotations

import numpy as np
import torch

import amsgrad_optimizer_step_gb300 as fa
import oracle
from synthetic.configs import BF16, F16, F32, Workload

U = 2.0 ** -24
TORCH_DT = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}
ORACLE_DT = {F32: "f32", F16: "f16", BF16: "bf16"}


def widen_host(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F32:
        return bits.astype(np.float64)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def grad_bits_from_device(g: torch.Tensor) -> np.ndarray:
    if g.dtype == torch.float32:
        return g.cpu().numpy()
    return g.view(torch.int16).cpu().numpy().view(np.uint16)


def gate(dev, ref, tol, what):
    dev = np.asarray(dev, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(dev - ref)
    lim = tol * np.maximum(1.0, np.abs(ref))
    bad = ~(err <= lim)
    if bad.any():
        i = int(np.argmax(np.where(bad, err, -1)))
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond {tol:g}*max(1,|x|); "
                             f"worst at {i}: dev={dev[i]!r} ref={ref[i]!r} err={err[i]:.3e}")


def tight_bound(before, x, gmul, opts, t, ref):
    """Per-element bound on |device - oracle| for one update from identical state.

    Derived from FP32 rounding: each FP32 operation contributes at most one
    unit roundoff U of its result; host coefficients carry one cast each; the
    oracle output carries one final rounding.  A factor of 2 covers the
    counting slack.
    """
    p0, m0, v0, vm0 = before
    b1, b2, lr = opts["beta1"], opts["beta2"], opts["lr"]
    g = x * gmul
    bc1 = 1 - b1 ** t
    bc2 = 1 - b2 ** t
    p1, m1, v1, vm1 = ref
    bm = 6 * U * (np.abs(b1 * m0) + np.abs((1 - b1) * g)) + U * np.abs(m1)
    bv = 8 * U * (b2 * v0 + (1 - b2) * g * g) + U * np.abs(v1)
    v_used = vm1 if opts["amsgrad"] else v1
    denom = np.sqrt(v_used / bc2) + opts["eps"]
    upd = lr / bc1 * np.abs(m1) / denom
    with np.errstate(divide="ignore", invalid="ignore"):
        dv_rel = np.where(v_used > 0, bv / v_used, 0.0)
    bupd = 6 * U * upd + lr / bc1 * bm / denom + 0.5 * dv_rel * upd
    bp = 3 * U * np.abs(p0) + U * np.abs(p1) + bupd
    return 2 * bp, 2 * bm, 2 * bv, 2 * bv


def check_tight(dev, ref, bound, what):
    dev = np.asarray(dev, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(dev - ref)
    bad = ~(err <= bound + 1e-45)
    if bad.any():
        i = int(np.argmax(np.where(bad, err / (bound + 1e-45), -1)))
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the FP32 error bound; "
                             f"worst at {i}: dev={dev[i]!r} ref={ref[i]!r} err={err[i]:.3e} "
                             f"bound={bound[i]:.3e}")


def oracle_one_step(x_bits, dtype, opts, scale, coef, t, before, lib):
    p0, m0, v0, vm0 = (np.array(a, dtype=np.float64) for a in before)
    lib.update(x_bits, ORACLE_DT[dtype], opts, scale, coef, t, t > 1, True, p0, m0, v0, vm0)
    return p0, m0, v0, vm0


class DeviceState:
    """Device buffers of one workload (in place or out of place)."""

    def __init__(self, w: Workload, n: int, device, guard: int = 0):
        self.w, self.n, self.device, self.guard = w, n, device, guard
        self.ams = w.amsgrad
        self.t = 0

        def buf(dtype):
            full = torch.empty(n + 2 * guard, dtype=dtype, device=device)
            if guard:
                full.view(torch.uint8).fill_(0x7F)  # NaN-pattern sentinels
            return full, full[guard:guard + n]

        self._p_full, self.p = buf(torch.float32)
        w.fill_params_device(self.p)
        self._g_full, self.g = buf(TORCH_DT[w.grad_dtype])
        self.m = self.v = self.vmax = None
        self._full = {"p": self._p_full, "g": self._g_full}
        if w.inplace:
            self._m_full, self.m = buf(torch.float32)
            self._v_full, self.v = buf(torch.float32)
            self._full.update(m=self._m_full, v=self._v_full)
            if self.ams:
                self._vm_full, self.vmax = buf(torch.float32)
                self._full["vmax"] = self._vm_full

    def guards_intact(self) -> bool:
        if not self.guard:
            return True
        for full in self._full.values():
            b = full.view(torch.uint8)
            eb = full.element_size() * self.guard
            if not (bool((b[:eb] == 0x7F).all()) and bool((b[-eb:] == 0x7F).all())):
                return False
        return True

    def snapshot(self, idx_t):
        def take(x):
            return None if x is None else x[idx_t].double().cpu().numpy()
        return take(self.p), take(self.m), take(self.v), take(self.vmax)


def ulp16(x, dtype):
    """Spacing of the 16-bit format at |x| (subnormal spacing below the normal range)."""
    sig, emin = (8, -126) if dtype == BF16 else (11, -14)
    a = np.abs(np.asarray(x, np.float64))
    e = np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))), emin)
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (sig - 1)).astype(np.int64))


def check_model_copy(model_bits, p_dev_f32, p_oracle_f32, dtype, lib, what):
    """The device's low-precision copy is the round-to-nearest-even encoding of the
    device's own FP32 parameters (bit-exact: the same decision in the same
    precision), and a correct rounding of the oracle's own parameters up to the
    trajectory tolerance: |copy - p| <= ulp/2 + 1e-5 * max(1, |p|)."""
    want = lib.model_copy(p_dev_f32, dtype)
    if not np.array_equal(model_bits, want):
        i = int(np.argmax(model_bits != want))
        raise AssertionError(f"{what}: model copy differs from the encoding of the device "
                             f"parameter at {i}: {model_bits[i]:#06x} vs {want[i]:#06x}")
    widened = widen_host(model_bits, dtype)
    ref = p_oracle_f32.astype(np.float64)
    lim = 0.5 * ulp16(ref, dtype) + 1e-5 * np.maximum(1.0, np.abs(ref))
    err = np.abs(widened - ref)
    if not np.all(err <= lim):
        i = int(np.argmax(err - lim))
        raise AssertionError(f"{what}: copy {widened[i]!r} is not a rounding of the oracle's "
                             f"{ref[i]!r} (err {err[i]:.3e} > {lim[i]:.3e})")


def run_workload(w: Workload, n: int, api: str, device, idx: np.ndarray | None = None,
                 guard: int = 0, segments=None, row_len: int = 0, lib=None,
                 full_grad_on_host: bool = True, step_check=True, model_dtype=None,
                 grad_mult: float = 1.0):
    """Runs every call of ``w`` (at size n) and checks each one.  Returns a summary.

    ``api``: "oop", "inplace", "bucket", "clipped", "gated" (the clipped step with the
    update deciding on the device from the report, which the last merge also posts to a
    pinned mailbox) or "staged" (the 4/5-kernel comparison, on in-place storage).  ``grad_mult`` is a fixed factor on the
    unscaled gradient for "inplace" and "staged" (the oracle's clip coefficient)."""
    import dataclasses
    lib = lib or oracle.lib()
    ws = w if n == w.n else w.scaled(n)
    if segments is not None and n != w.n:
        ws = dataclasses.replace(ws, segments=tuple(segments))
    if api == "staged" and not ws.inplace:
        ws = dataclasses.replace(ws, inplace=True)
    assert grad_mult == 1.0 or api in ("inplace", "staged")
    segs = list(ws.segments) if ws.segments is not None else None
    st = DeviceState(ws, n, device, guard=guard)
    opts = ws.options()
    fopts = fa.options(**opts)
    idx = np.arange(n) if idx is None else np.asarray(idx)
    idx_t = torch.as_tensor(idx, device=device)
    traj = oracle.OracleAdamW(ws.params_host(idx), opts, storage="f32", lib_=lib)
    p_host0 = ws.params_host(idx)
    assert np.array_equal(st.p[idx_t].cpu().numpy(), p_host0), "device/host inputs differ"

    p_model = None
    if model_dtype is not None:
        full = torch.empty(n + 2 * guard, dtype=TORCH_DT[model_dtype], device=device)
        full.view(torch.int16).fill_(0x7F7F)
        p_model = full[guard:guard + n]
        st._full["model"] = full
    if api == "staged":
        delta = torch.empty(n, dtype=torch.float32, device=device)
    if api in ("clipped", "gated"):
        mailbox = fa.report_mailbox()
        rows = fa.fa_stats_rows(n, row_len, segs)
        rows_buf = fa.stats_buffer(rows, device)
        scratch = fa.scratch_buffer(rows, device)
        report = fa.stats_buffer(1, device)
    summary = {"updates": 0, "skips": 0, "reports": []}
    for call in range(1, ws.calls + 1):
        ws.fill_grad_device(call, st.g)
        gh = ws.grad_host(call, idx)
        assert np.array_equal(grad_bits_from_device(st.g[idx_t]), gh), "device/host grads differ"
        skip = call in ws.skip_calls
        ctl = fa.control(ws.gradient_scale, skip)
        before = st.snapshot(idx_t)
        model_before = None if p_model is None else grad_bits_from_device(p_model[idx_t])
        t_before = st.t
        coef_dev = grad_mult
        expect_skip = skip
        coef_or = grad_mult
        if api in ("clipped", "gated"):
            full_bits = (ws.grad_host(call, np.arange(n)) if full_grad_on_host
                         else grad_bits_from_device(st.g))
            s_or, c_or = lib.gradient_stats(full_bits, ORACLE_DT[ws.grad_dtype], ws.gradient_scale)
            skip_or, norm_or, coef_or = lib.clip_decision(s_or, c_or, ws.max_grad_norm)
            step = fa.fa_bucket_step_clipped if api == "clipped" else \
                (lambda *a: fa.fa_bucket_step_clipped_gated(*a, mailbox))
            t_new, rep = step(segs, st.p, st.g, st.m, st.v, st.vmax, st.t, fopts, ctl,
                              ws.max_grad_norm, row_len, rows_buf, scratch, report)
            torch.cuda.synchronize()
            if not skip:
                assert rep.nonfinite == c_or, (call, rep.nonfinite, c_or)
                assert bool(rep.skipped_nonfinite) == skip_or
                if not skip_or:
                    assert abs(rep.grad_norm - norm_or) <= 1e-5 * norm_or, (rep.grad_norm, norm_or)
                    assert abs(rep.clip_coef - coef_or) <= 1e-5 * coef_or
                summary["reports"].append((rep.grad_norm, norm_or, rep.nonfinite, c_or))
            expect_skip = skip or skip_or
            coef_dev = rep.clip_coef
            updated = bool(rep.updated)
        elif api == "oop":
            p2, m2, v2, vm2, t_new, updated = fa.fa_adamw_step(st.p, st.g, st.m, st.v, st.vmax,
                                                               st.t, fopts, ctl)
            st.p, st.m, st.v, st.vmax = p2, m2, v2, vm2
        elif api == "inplace":
            t_new, updated = fa.fa_adamw_step_inplace(st.p, st.g, st.m, st.v, st.vmax, st.t,
                                                      fopts, ctl, grad_mult=grad_mult)
        elif api == "staged":
            t_new, updated = fa.fa_adamw_step_staged(st.p, st.g, st.m, st.v, st.vmax, st.t,
                                                     fopts, ctl, delta, grad_mult=grad_mult)
        elif api == "bucket" and p_model is not None:
            updated = fa.fa_bucket_update(segs, st.p, st.g, st.m, st.v, st.vmax, st.t, fopts,
                                          ctl, p_model=p_model)
            t_new = st.t + int(updated)
        elif api == "bucket":
            t_new, updated = fa.fa_bucket_step(segs, st.p, st.g, st.m, st.v, st.vmax, st.t,
                                               fopts, ctl)
        else:
            raise ValueError(api)
        torch.cuda.synchronize()
        assert updated == (not expect_skip), (call, updated, expect_skip)
        assert t_new == t_before + (0 if expect_skip else 1)
        st.t = t_new
        after = st.snapshot(idx_t)
        assert st.guards_intact(), f"guard band overwritten at call {call}"

        if expect_skip:
            for a, b in zip(before, after):
                if a is not None:
                    assert np.array_equal(a, b), "skipped call changed state"
            if p_model is not None:
                assert np.array_equal(grad_bits_from_device(p_model[idx_t]), model_before), \
                    "skipped call wrote the model copy"
            summary["skips"] += 1
            traj.step(gh, ORACLE_DT[ws.grad_dtype], ws.gradient_scale, skip_update=True)
            continue
        summary["updates"] += 1
        x = widen_host(gh, ws.grad_dtype)
        # one step from identical state
        if step_check:
            zero = np.zeros(len(idx))
            # before the first update the moment buffers hold no state (never read)
            b4 = (before[0], zero, zero, zero) if t_before == 0 else \
                tuple(z if z is not None else zero for z in before)
            ref = oracle_one_step(gh, ws.grad_dtype, opts, ws.gradient_scale, coef_dev, st.t,
                                  b4, lib)
            gmul = (-1.0 if opts["maximize"] else 1.0) * coef_dev / ws.gradient_scale
            bounds = tight_bound(b4, x, gmul, opts, st.t, ref)
            names = ("p", "m", "v", "vmax")
            for k in range(4 if ws.amsgrad else 3):
                gate(after[k], ref[k], 1e-6, f"call {call} one-step {names[k]}")
                check_tight(after[k], ref[k], bounds[k], f"call {call} one-step {names[k]}")
        # trajectory
        traj.step(gh, ORACLE_DT[ws.grad_dtype], ws.gradient_scale, clip_coef=coef_or)
        assert traj.state.t == st.t
        gate(after[0], traj.p, 1e-5, f"call {call} trajectory p")
        gate(after[1], traj.state.m, 1e-5, f"call {call} trajectory m")
        gate(after[2], traj.state.v, 1e-5, f"call {call} trajectory v")
        if ws.amsgrad:
            gate(after[3], traj.state.vmax, 1e-5, f"call {call} trajectory vmax")
        if p_model is not None:
            check_model_copy(grad_bits_from_device(p_model[idx_t]),
                             after[0].astype(np.float32), traj.p.astype(np.float32),
                             model_dtype, lib, f"call {call} model copy")
    summary["t"] = st.t
    summary["state"] = st
    return summary
