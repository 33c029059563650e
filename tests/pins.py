"""Pins for the oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes an ``oracle.OracleLib`` and raises ``AssertionError`` when
the library disagrees with a closed form, an invariant, an independent library
routine (torch's CPU AdamW in float64, numpy's float16 decoding, ``math.fsum``)
or a number printed on the pages.  ``tests/test_oracle_pins.py`` runs them on
the real oracle; ``tests/test_oracle_mutants.py`` runs them on copies of the
oracle with one planted mistake each and expects every copy to be caught.
"""

from __future__ import annotations

import math

import numpy as np

from oracle import OracleAdamW, FAN_IN, MAX_ROWS

BASE = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2,
            amsgrad=False, maximize=False)


def _rng(seed):
    return np.random.default_rng(seed)


def _grads(rng, n, lo=1e-3, hi=1e-1):
    """Random FP32 gradients with magnitudes in [lo, hi] and random signs."""
    mag = np.exp(rng.uniform(np.log(lo), np.log(hi), n))
    return (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    bad = err > atol + rtol * np.abs(b)
    assert not bad.any(), f"{what}: max err {err.max():.3e} at {np.argmax(err)}"


def _run(L, p0, grads, opts, dtype="f32", scale=1.0, storage="f64", skips=()):
    o = OracleAdamW(p0, opts, storage=storage, lib_=L)
    traj = []
    for k, g in enumerate(grads, start=1):
        o.step(g, dtype, gradient_scale=scale, skip_update=k in skips)
        traj.append((o.p.copy(), o.state.t,
                     None if o.state.m is None else o.state.m.copy(),
                     None if o.state.v is None else o.state.v.copy(),
                     None if o.state.vmax is None else o.state.vmax.copy()))
    return o, traj


# ---------------------------------------------------------------------------
# Update: closed forms
# ---------------------------------------------------------------------------

def pin_first_step_closed_form(L):
    """t = 1: m/bc1 = g and v/bc2 = g^2, so the step is lr*g/(|g|+eps) plus decay."""
    rng = _rng(11)
    n = 512
    p0 = rng.normal(0, 0.02, n)
    g = _grads(rng, n)
    for ams in (False, True):
        opts = dict(BASE, amsgrad=ams)
        o, _ = _run(L, p0, [g], opts)
        gd = g.astype(np.float64)
        expect = p0 * (1 - opts["lr"] * opts["weight_decay"]) - opts["lr"] * gd / (np.abs(gd) + opts["eps"])
        _close(o.p, expect, 1e-13, what="p after step 1")
        _close(o.state.m / (1 - opts["beta1"]), gd, 1e-14, what="m/bc1")
        _close(o.state.v / (1 - opts["beta2"]), gd * gd, 1e-14, what="v/bc2")
        if ams:
            assert np.array_equal(o.state.vmax, o.state.v)
        assert o.state.t == 1


def pin_eps_zero_is_signed_lr(L):
    """t = 1 with eps -> 0: the step is lr*sign(g) plus decay, for every gradient dtype."""
    rng = _rng(12)
    n = 300
    p0 = rng.normal(0, 0.02, n)
    g32 = _grads(rng, n, 1e-2, 1.0)
    opts = dict(BASE, eps=0.0)
    cases = [("f32", g32),
             ("f16", g32.astype(np.float16).view(np.uint16)),
             ("bf16", (g32.view(np.uint32) >> 16).astype(np.uint16))]
    for dtype, g in cases:
        for scale in (1.0, 64.0, 3.0):
            o, _ = _run(L, p0, [g], opts, dtype=dtype, scale=scale)
            decayed = p0 * (1 - opts["lr"] * opts["weight_decay"])
            _close(o.p - decayed, -opts["lr"] * np.sign(g32.astype(np.float64)), 1e-12, 1e-18,
                   what=f"signed step {dtype} scale {scale}")


def pin_constant_gradient(L):
    """Constant g: m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, so every step is lr*g/(|g|+eps)."""
    rng = _rng(13)
    n = 200
    p0 = rng.normal(0, 0.02, n)
    g = _grads(rng, n)
    gd = g.astype(np.float64)
    for ams in (False, True):
        opts = dict(BASE, amsgrad=ams, beta1=0.8, beta2=0.95)
        o, traj = _run(L, p0, [g] * 25, opts)
        p = p0.copy()
        for t, (pt, tt, m, v, vmax) in enumerate(traj, start=1):
            p = p * (1 - opts["lr"] * opts["weight_decay"]) - opts["lr"] * gd / (np.abs(gd) + opts["eps"])
            assert tt == t
            _close(pt, p, 1e-12, 1e-15, what=f"p at t={t}")
            _close(m, (1 - opts["beta1"] ** t) * gd, 1e-13, what=f"m at t={t}")
            _close(v, (1 - opts["beta2"] ** t) * gd * gd, 1e-13, what=f"v at t={t}")
            if ams:
                _close(vmax, v, 0.0, what="vmax = v when v grows")


def pin_weight_decay_only(L):
    """g = 0: the moments stay 0, the step term is 0/(0+eps), p_t = p0 (1 - lr wd)^t."""
    rng = _rng(14)
    n = 100
    p0 = rng.normal(0, 0.02, n)
    for ams in (False, True):
        opts = dict(BASE, amsgrad=ams, weight_decay=0.3, lr=0.01)
        o, traj = _run(L, p0, [np.zeros(n, np.float32)] * 12, opts)
        for t, (pt, _, m, v, _) in enumerate(traj, start=1):
            _close(pt, p0 * (1 - 0.01 * 0.3) ** t, 1e-14, what=f"decay t={t}")
            assert not m.any() and not v.any()


def pin_lr_zero_moment_sums(L):
    """lr = 0: p is unchanged; m and v equal their unrolled exponential sums."""
    rng = _rng(15)
    n, T = 64, 9
    p0 = rng.normal(0, 0.02, n)
    gs = [_grads(rng, n) for _ in range(T)]
    opts = dict(BASE, lr=0.0, beta1=0.7, beta2=0.9)
    o, _ = _run(L, p0, gs, opts)
    assert np.array_equal(o.p, p0)
    G = np.stack([g.astype(np.float64) for g in gs])
    w1 = np.array([(1 - 0.7) * 0.7 ** (T - k) for k in range(1, T + 1)])
    w2 = np.array([(1 - 0.9) * 0.9 ** (T - k) for k in range(1, T + 1)])
    _close(o.state.m, w1 @ G, 1e-13, 1e-18, what="m sum")
    _close(o.state.v, w2 @ (G * G), 1e-13, 1e-22, what="v sum")


def pin_bias_correction_power(L):
    """The host power is an integer power: beta^t for t up to 1000."""
    for beta in (0.9, 0.999, 0.5):
        for t in (0, 1, 2, 3, 10, 1000):
            got = L.int_pow(beta, t)
            want = math.prod([beta] * t) if t else 1.0
            assert abs(got - want) <= 1e-15 * abs(want), (beta, t, got, want)
            assert abs(got - beta ** t) <= 1e-12 * beta ** t


# ---------------------------------------------------------------------------
# Update: the library special case (torch CPU AdamW, float64)
# ---------------------------------------------------------------------------

def _widen_independent(g, dtype):
    if dtype == "f32":
        return g.astype(np.float64)
    if dtype == "f16":
        return g.view(np.float16).astype(np.float64)
    return (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_torch_adamw(L):
    """12 cases (3 gradient dtypes x AMSGrad x maximize), 5 steps each, vs torch.optim.AdamW."""
    import torch
    rng = _rng(16)
    n = 257
    for dtype in ("f32", "f16", "bf16"):
        for ams in (False, True):
            for maxi in (False, True):
                opts = dict(lr=2e-3, beta1=0.85, beta2=0.99, eps=1e-6, weight_decay=0.05,
                            amsgrad=ams, maximize=maxi)
                p0 = rng.normal(0, 0.05, n)
                scale = 8.0
                # gradients that shrink then grow so that AMSGrad's max matters
                gs = []
                for k in range(5):
                    x = (_grads(rng, n) * (4.0 if k == 0 else 0.5 ** k) * scale).astype(np.float32)
                    if dtype == "f16":
                        gs.append(x.astype(np.float16).view(np.uint16))
                    elif dtype == "bf16":
                        gs.append((x.view(np.uint32) >> 16).astype(np.uint16))
                    else:
                        gs.append(x)
                o, traj = _run(L, p0, gs, opts, dtype=dtype, scale=scale)
                tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
                topt = torch.optim.AdamW([tp], lr=opts["lr"], betas=(opts["beta1"], opts["beta2"]),
                                         eps=opts["eps"], weight_decay=opts["weight_decay"],
                                         amsgrad=ams, maximize=maxi, foreach=False)
                for k, g in enumerate(gs):
                    tp.grad = torch.tensor(_widen_independent(g, dtype) / scale)
                    topt.step()
                    st = topt.state[tp]
                    pt, t, m, v, vmax = traj[k]
                    tag = f"{dtype} ams={ams} max={maxi} step {k + 1}"
                    scale_p = np.abs(pt).max()
                    _close(pt, tp.detach().numpy(), 1e-11, 1e-13 * scale_p, what="p " + tag)
                    _close(m, st["exp_avg"].numpy(), 1e-10, 1e-13 * np.abs(m).max(), what="m " + tag)
                    _close(v, st["exp_avg_sq"].numpy(), 1e-10, 1e-13 * np.abs(v).max(), what="v " + tag)
                    if ams:
                        _close(vmax, st["max_exp_avg_sq"].numpy(), 1e-10, 1e-13 * np.abs(vmax).max(),
                               what="vmax " + tag)


def _same_with_nan(a, b, rtol, what):
    """Equal NaN positions, and the other values within rtol (``_close`` alone lets
    a NaN on either side pass, because every comparison with NaN is false)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb), \
        f"{what}: NaN at {np.flatnonzero(na ^ nb)[:5]} on one side only"
    ok = ~nb
    _close(a[ok], b[ok], rtol, 1e-13 * max(1e-300, np.abs(b[ok]).max(initial=0.0)), what=what)


def pin_amsgrad_max_propagates_nan_like_torch(L):
    """A NaN gradient under AMSGrad: the running max of v takes the NaN and keeps it, as
    torch.maximum does in torch.optim.AdamW(amsgrad=True) (float64 CPU), for FP32 and
    BF16 storage; the other elements follow torch as usual.  A max that drops a NaN
    operand (C's fmax) keeps the old maximum there instead and fails."""
    import torch
    rng = _rng(31)
    n = 96
    nan_at = np.array([3, 17, 40, 95])
    for dtype in ("f32", "bf16"):
        opts = dict(BASE, amsgrad=True, beta2=0.99)
        p0 = rng.normal(0, 0.02, n)
        xs = [_grads(rng, n) * np.float32(2.0 if k == 0 else 0.5) for k in range(4)]
        xs[1] = xs[1].copy()
        xs[1][nan_at] = np.float32(np.nan)
        if dtype == "bf16":
            gs = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in xs]
            assert np.isnan(_widen_independent(gs[1], "bf16")[nan_at]).all()
        else:
            gs = xs
        _, traj = _run(L, p0, gs, opts, dtype=dtype)
        tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
        topt = torch.optim.AdamW([tp], lr=opts["lr"], betas=(opts["beta1"], opts["beta2"]),
                                 eps=opts["eps"], weight_decay=opts["weight_decay"],
                                 amsgrad=True, foreach=False)
        for k, g in enumerate(gs):
            tp.grad = torch.tensor(_widen_independent(g, dtype))
            topt.step()
            st = topt.state[tp]
            pt, _, m, v, vmax = traj[k]
            tag = f"{dtype} step {k + 1}"
            _same_with_nan(vmax, st["max_exp_avg_sq"].numpy(), 1e-10, "vmax " + tag)
            _same_with_nan(v, st["exp_avg_sq"].numpy(), 1e-10, "v " + tag)
            _same_with_nan(m, st["exp_avg"].numpy(), 1e-10, "m " + tag)
            _same_with_nan(pt, tp.detach().numpy(), 1e-11, "p " + tag)
            if k >= 1:
                assert np.isnan(vmax[nan_at]).all(), f"NaN dropped from the max, {tag}"
                assert not np.isnan(np.delete(vmax, nan_at)).any()


# ---------------------------------------------------------------------------
# Update: invariants
# ---------------------------------------------------------------------------

def pin_amsgrad_invariants(L):
    """vmax is non-decreasing and >= v; with shrinking gradients AMSGrad differs from AdamW."""
    rng = _rng(17)
    n = 400
    p0 = rng.normal(0, 0.02, n)
    gs = [_grads(rng, n) * np.float32(0.6 ** k) for k in range(8)]
    o_ams, tr = _run(L, p0, gs, dict(BASE, amsgrad=True))
    o_plain, _ = _run(L, p0, gs, dict(BASE, amsgrad=False))
    prev = np.zeros(n)
    for _, _, _, v, vmax in tr:
        assert (vmax >= prev).all() and (vmax >= v).all()
        prev = vmax
    assert (tr[-1][4] > tr[-1][3]).mean() > 0.5, "max never above v: shrink not seen"
    assert np.abs(o_ams.p - o_plain.p).max() > 1e-6
    # the stored max is uncorrected: it equals the largest v seen so far
    vs = np.stack([x[3] for x in tr])
    _close(tr[-1][4], vs.max(axis=0), 0.0, what="uncorrected max")


def pin_maximize_is_negated_gradient(L):
    rng = _rng(18)
    n = 300
    p0 = rng.normal(0, 0.02, n)
    gs = [_grads(rng, n) for _ in range(4)]
    for ams in (False, True):
        a, _ = _run(L, p0, gs, dict(BASE, amsgrad=ams, maximize=True))
        b, _ = _run(L, p0, [-g for g in gs], dict(BASE, amsgrad=ams, maximize=False))
        assert np.array_equal(a.p, b.p) and np.array_equal(a.state.m, b.state.m)
        assert np.array_equal(a.state.v, b.state.v)
        c, _ = _run(L, p0, gs, dict(BASE, amsgrad=ams, maximize=False))
        assert np.abs(a.p - c.p).max() > 1e-5, "maximize changed nothing"


def pin_skip_and_empty(L):
    """skip_update and an empty tensor change nothing and do not advance t."""
    rng = _rng(19)
    n = 100
    p0 = rng.normal(0, 0.02, n)
    gs = [_grads(rng, n) for _ in range(5)]
    for storage in ("f32", "f64"):
        a, tr = _run(L, p0, gs, dict(BASE, amsgrad=True), storage=storage, skips=(1, 3))
        assert [x[1] for x in tr] == [0, 1, 1, 2, 3]
        assert tr[0][2] is None and np.array_equal(tr[0][0], p0.astype(tr[0][0].dtype))
        for k in (2,):
            for j in (0, 2, 3, 4):
                assert np.array_equal(tr[k][j], tr[k - 1][j])
        b, _ = _run(L, p0, [gs[1], gs[3], gs[4]], dict(BASE, amsgrad=True), storage=storage)
        assert np.array_equal(a.p, b.p) and np.array_equal(a.state.vmax, b.state.vmax)
    e = OracleAdamW(np.zeros(0), BASE, lib_=L)
    assert e.step(np.zeros(0, np.float32), "f32") is False and e.state.t == 0


def pin_power_of_two_scale(L):
    """A gradient stored x 2^k with gradient_scale 2^k gives the identical update."""
    rng = _rng(20)
    n = 256
    p0 = rng.normal(0, 0.02, n)
    g = _grads(rng, n)
    for dtype in ("f32", "bf16"):
        if dtype == "f32":
            g1, g2 = g, (g * np.float32(128)).astype(np.float32)
        else:
            g1 = (g.view(np.uint32) >> 16).astype(np.uint16)
            g2 = ((g * np.float32(128)).view(np.uint32) >> 16).astype(np.uint16)
        a, _ = _run(L, p0, [g1], BASE, dtype=dtype, scale=1.0)
        b, _ = _run(L, p0, [g2], BASE, dtype=dtype, scale=128.0)
        assert np.array_equal(a.p, b.p)
        c, _ = _run(L, p0, [g2], BASE, dtype=dtype, scale=1.0)
        assert not np.array_equal(a.p, c.p)


def pin_clip_coefficient_scales_gradient(L):
    """clip_coef c is exactly a factor on the unscaled gradient (power-of-two c is exact)."""
    rng = _rng(21)
    n = 128
    p0 = rng.normal(0, 0.02, n)
    g = _grads(rng, n)
    a = OracleAdamW(p0, BASE, storage="f64", lib_=L)
    a.step(g, "f32", clip_coef=0.25)
    b = OracleAdamW(p0, BASE, storage="f64", lib_=L)
    b.step((g * np.float32(0.25)).astype(np.float32), "f32")
    assert np.array_equal(a.p, b.p) and np.array_equal(a.state.v, b.state.v)


def pin_fp32_storage_rounds(L):
    """FP32 storage keeps every stored value FP32-representable and within 1 ulp of FP64."""
    rng = _rng(22)
    n = 500
    p0 = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [_grads(rng, n)]
    a, _ = _run(L, p0, gs, dict(BASE, amsgrad=True), storage="f32")
    b, _ = _run(L, p0.astype(np.float64), gs, dict(BASE, amsgrad=True), storage="f64")
    for x, y in ((a.p, b.p), (a.state.m, b.state.m), (a.state.v, b.state.v)):
        assert x.dtype == np.float32
        _close(x, y, 2.0 ** -24, what="fp32 rounding")


# ---------------------------------------------------------------------------
# Widening of the stored gradient
# ---------------------------------------------------------------------------

def pin_widening(L):
    allbits = np.arange(65536, dtype=np.uint16)
    got = L.widen(allbits, "f16")
    want = allbits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    got = L.widen(allbits, "bf16")
    with np.errstate(invalid="ignore"):
        want = (allbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    rng = _rng(23)
    f = rng.integers(0, 2 ** 32, 4096, dtype=np.uint64).astype(np.uint32).view(np.float32)
    got = L.widen(f, "f32")
    ok = ~np.isnan(f)
    assert np.array_equal(got[ok], f[ok].astype(np.float64))


# ---------------------------------------------------------------------------
# Low-precision model copy (round to nearest, ties to even)
# ---------------------------------------------------------------------------

def _tie_structured_f32():
    """Every sign/exponent/high-mantissa pattern with low bits at and around the
    BF16 and FP16 rounding points (exact ties, one below, one above)."""
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x7FFF, 0x8000, 0x8001, 0xEFFF,
                     0xF000, 0xFFFF], dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).ravel()
    return bits.view(np.float32)


def pin_model_copy_rounding(L):
    import torch
    x = _tie_structured_f32()
    ok = ~np.isnan(x)
    got = L.model_copy(x, "bf16")
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got[ok], want[ok]), "bf16 rounding differs from torch"
    assert np.all((got[~ok] & 0x7F80) == 0x7F80) and np.all((got[~ok] & 0x7F) != 0)
    rng = _rng(27)
    y = np.concatenate([x[ok], (rng.standard_normal(200_000) * 10.0 ** rng.integers(-9, 6, 200_000)),
                        np.array([65504, 65519.996, 65520, 65536, 6.1e-5, 6.0e-5, 2.98e-8,
                                  2.9802322e-8, 5.96e-8, 1e-30, -0.0, 0.0, np.inf, -np.inf])
                        ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want16 = y.astype(np.float16).view(np.uint16)
    got16 = L.model_copy(y, "f16")
    assert np.array_equal(got16, want16), "f16 rounding differs from numpy"
    assert L.model_copy(np.array([np.nan], np.float32), "f16")[0] & 0x7C00 == 0x7C00


# ---------------------------------------------------------------------------
# Statistics and the decision
# ---------------------------------------------------------------------------

def _planted(rng, n, dtype, n_bad):
    x = _grads(rng, n, 1e-4, 10.0)
    bad = rng.choice(n, size=min(n_bad, n), replace=False) if n else np.zeros(0, int)
    vals = [np.inf, -np.inf, np.nan]
    for j, i in enumerate(bad):
        x[i] = vals[j % 3]
    if dtype == "f32":
        return x, bad
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16), bad
    return (x.view(np.uint32) >> 16).astype(np.uint16), bad


def pin_gradient_stats_brute_force(L):
    rng = _rng(24)
    for dtype in ("f32", "f16", "bf16"):
        for n in (0, 1, 3, 255, 256, 257, 1000, 4099):
            for n_bad in (0, 1, 5):
                for scale in (1.0, 128.0, 3.0):
                    g, bad = _planted(rng, n, dtype, n_bad)
                    w = _widen_independent(g, dtype)
                    fin = np.isfinite(w)
                    want_s = math.fsum(float(x / scale) ** 2 for x in w[fin])
                    s, c = L.gradient_stats(g, dtype, scale)
                    assert c == int((~fin).sum()) == len(set(bad.tolist()))
                    assert abs(s - want_s) <= 1e-13 * want_s, (dtype, n, s, want_s)


def _rows_brute(w, row_len, segments):
    seg = [0, len(w)] if segments is None else list(segments)
    out = []
    for a, b in zip(seg[:-1], seg[1:]):
        i = a
        while i < b:
            chunk = w[i:min(i + row_len, b)]
            fin = np.isfinite(chunk)
            out.append((math.fsum(float(x) ** 2 for x in chunk[fin]), int((~fin).sum())))
            i += row_len
    return out


def pin_row_stats_brute_force(L):
    rng = _rng(25)
    for dtype in ("f32", "bf16", "f16"):
        for n, row_len, segments in ((1000, 256, None), (257, 256, None), (7, 3, None),
                                     (2000, 128, [0, 5, 5, 700, 1300, 2000]),
                                     (4100, 256, [0, 1, 2049, 4100])):
            g, _ = _planted(rng, n, dtype, 6)
            w = _widen_independent(g, dtype)
            s, c = L.row_stats(g, dtype, row_len, segments)
            want = _rows_brute(w, row_len, segments)
            assert len(s) == len(want), (n, row_len, segments, len(s), len(want))
            for (ws, wc), gs_, gc in zip(want, s, c):
                assert gc == wc
                assert abs(gs_ - ws) <= 1e-13 * ws
    try:
        L.row_stats(np.zeros(10, np.float32), "f32", 4, [0, 6, 5, 10])
    except ValueError:
        pass
    else:
        raise AssertionError("decreasing segment table accepted")


def pin_stats_plan_golden(L, golden):
    fan = golden["fan_in"]
    lo, hi = golden["min_rows"], golden["max_rows"]
    assert fan == FAN_IN and hi == MAX_ROWS
    assert L.stats_plan(lo - 1) is None and L.stats_plan(hi + 1) is None
    worst_scratch, worst_extra = 0, 0
    probe = sorted(set([1, 2, 3, 1023, 1024, 1025, 2048, 4096, 1048575, 1048576, 1048577,
                        2 ** 21, 4194303, 4194304] + list(np.random.default_rng(26).integers(1, hi + 1, 300))))
    for rows in probe:
        k, e, levels = L.stats_plan(int(rows))
        extra = k - 1
        worst_scratch = max(worst_scratch, 4 * e)
        worst_extra = max(worst_extra, extra)
        assert levels[-1] == 1
        if rows <= golden["no_extra_merge_at_or_below_rows"]:
            assert extra == 0 and e == 0
        else:
            assert extra >= 1
        # each level holds ceil(previous / fan) records of 12 bytes (3 FP32 words)
        assert 4 * e == golden["report_bytes"] * sum(levels[:-1])
    assert worst_extra == golden["max_extra_merge_kernels"]
    assert worst_scratch == golden["max_extra_scratch_bytes"]
    k, e, _ = L.stats_plan(1048576)
    assert (k, 4 * e) == (2, 12288)


def pin_clip_decision(L):
    assert L.clip_decision(4.0, 0, 1.0) == (False, 2.0, 0.5)
    assert L.clip_decision(0.25, 0, 1.0) == (False, 0.5, 1.0)
    assert L.clip_decision(4.0, 0, 0.0) == (False, 2.0, 1.0)
    assert L.clip_decision(4.0, 3, 1.0)[0] is True
    s, n, c = L.clip_decision(1e6, 0, 10.0)
    assert not s and n == 1000.0 and abs(c - 0.01) < 1e-18


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
