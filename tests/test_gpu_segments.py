"""Per-parameter statistics and clipping (chunk merge, segment multipliers) vs the oracle.

The oracle needs nothing new here: a segment's statistics and its clip decision
are the pinned whole-gradient functions applied to that segment's slice, and a
segment's update is the pinned update with that segment's coefficient.
"""

import dataclasses
import math

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
import oracle
from gpu_harness import gate, grad_bits_from_device, oracle_one_step, TORCH_DT
from synthetic.configs import CONFIG4, decoder_bucket_shapes

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


def _segments(seed, count, max_len, empty_every=0):
    rng = np.random.default_rng(seed)
    sizes = rng.integers(1, max_len, count)
    if empty_every:
        sizes[::empty_every] = 0
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def _slice_stats(lib, bits, dtype, seg, scale=1.0):
    out = []
    for a, b in zip(seg[:-1], seg[1:]):
        out.append(lib.gradient_stats(bits[a:b], dtype, scale))
    return out


@pytest.mark.parametrize("gdt", ["bf16", "f32"])
@pytest.mark.parametrize("row_len", [256, 100])
def test_chunk_reports_match_oracle_per_segment(gdt, row_len, oracle_lib):
    seg = _segments(31, 300, 5000, empty_every=37)   # > 240 segments: several launches
    n = int(seg[-1])
    w = dataclasses.replace(CONFIG4, grad_dtype=gdt, segments=None).scaled(n)
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    w.fill_grad_device(1, g)
    bad = [int(seg[5]) + 1, int(seg[200])]   # NaN/Inf planted in two segments
    g[bad[0]] = float("inf")
    g[bad[1]] = float("nan")
    bits = grad_bits_from_device(g)
    crow = fa.segment_rows(list(seg), row_len)
    rows_buf = fa.stats_buffer(crow[-1], DEV)
    fa.fa_analyze_gradient(g, row_len, rows_buf, list(seg))
    scratch = torch.empty(max(1, fa.fa_stats_chunk_scratch(crow)), device=DEV)
    reports = fa.stats_buffer(len(seg) - 1, DEV)
    fa.fa_merge_gradient_stats_chunks(rows_buf, crow, scratch, reports)
    torch.cuda.synchronize()
    host = reports.cpu()
    sums = host[:, 0].view(torch.float32).double().numpy() + host[:, 2].view(torch.float32).double().numpy()
    counts = host[:, 1].numpy().astype(np.int64)
    want = _slice_stats(oracle_lib, bits, gdt, seg)
    for k, (s, c) in enumerate(want):
        assert counts[k] == c, (k, counts[k], c)
        if c == 0:
            assert abs(sums[k] - s) <= 1e-5 * s + 1e-30, (k, sums[k], s)
    assert counts.sum() == 2


def _bucket(n, gdt, seed):
    w = dataclasses.replace(CONFIG4, grad_dtype=gdt, amsgrad=True, seed=seed, segments=None).scaled(n)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    return w, p


def test_uniform_multipliers_equal_the_bucket_step_bitwise():
    seg = _segments(32, 50, 300_000)
    n = int(seg[-1])
    w, p0 = _bucket(n, "f16", 33)
    o = fa.options(**w.options())
    g = torch.empty(n, dtype=torch.float16, device=DEV)
    pa, pb = p0.clone(), p0.clone()
    sa = [torch.zeros(n, device=DEV) for _ in range(3)]
    sb = [torch.zeros(n, device=DEV) for _ in range(3)]
    ta = tb = 0
    for call in range(1, 4):
        w.fill_grad_device(call, g)
        ta, _ = fa.fa_bucket_step(list(seg), pa, g, *sa, ta, o, fa.control(2.0), 0.75)
        assert fa.fa_bucket_update(list(seg), pb, g, *sb, tb, o, fa.control(2.0),
                                   seg_grad_mult=[0.75] * (len(seg) - 1))
        tb += 1
    torch.cuda.synchronize()
    assert ta == tb == 3
    assert torch.equal(pa, pb) and all(torch.equal(x, y) for x, y in zip(sa, sb))


@pytest.mark.parametrize("gdt", ["bf16", "f32"])
def test_segment_multipliers_vs_oracle(gdt, oracle_lib):
    seg = _segments(34, 260, 3000, empty_every=50)
    n = int(seg[-1])
    w, p = _bucket(n, gdt, 35)
    opts = w.options()
    o = fa.options(**opts)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    rng = np.random.default_rng(36)
    refs = [oracle.OracleAdamW(w.params_host(np.arange(a, b)), opts, lib_=oracle_lib)
            for a, b in zip(seg[:-1], seg[1:])]
    t = 0
    for call in range(1, 4):
        mult = rng.uniform(0.1, 1.0, len(seg) - 1)
        w.fill_grad_device(call, g)
        assert fa.fa_bucket_update(list(seg), p, g, m, v, vm, t, o, fa.control(),
                                   seg_grad_mult=mult)
        t += 1
        bits = grad_bits_from_device(g)
        for k, (a, b) in enumerate(zip(seg[:-1], seg[1:])):
            refs[k].step(bits[a:b], gdt, clip_coef=float(mult[k]))
    torch.cuda.synchronize()
    ph = p.cpu().numpy()
    vh = vm.cpu().numpy()
    for k, (a, b) in enumerate(zip(seg[:-1], seg[1:])):
        gate(ph[a:b], refs[k].p, 1e-5, f"segment {k} p")
        gate(vh[a:b], refs[k].state.vmax, 1e-5, f"segment {k} vmax")


@pytest.mark.parametrize("gdt,maximize", [("f16", False), ("bf16", False), ("f32", True)])
def test_segment_multipliers_mixed_sizes_vs_oracle(gdt, maximize, oracle_lib):
    """Large segments between runs of tiny and empty ones, several million elements:
    steady steps take the shared-memory pipeline, whose tiles span up to dozens of
    segments and whose per-CTA segment index has to skip whole runs between tiles."""
    rng = np.random.default_rng(37)
    sizes = rng.integers(0, 3000, 230)
    sizes[::11] = rng.integers(150_000, 450_000, len(sizes[::11]))
    sizes[3::17] = 0
    seg = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    n = int(seg[-1])
    assert n > 2 * 152 * 4096
    w, p = _bucket(n, gdt, 38)
    w = dataclasses.replace(w, maximize=maximize)
    opts = w.options()
    o = fa.options(**opts)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    refs = [oracle.OracleAdamW(w.params_host(np.arange(a, b)), opts, lib_=oracle_lib)
            for a, b in zip(seg[:-1], seg[1:])]
    t = 0
    for call in range(1, 4):
        mult = rng.uniform(0.1, 1.0, len(seg) - 1)
        w.fill_grad_device(call, g)
        assert fa.fa_bucket_update(list(seg), p, g, m, v, vm, t, o, fa.control(),
                                   seg_grad_mult=mult)
        t += 1
        bits = grad_bits_from_device(g)
        for k, (a, b) in enumerate(zip(seg[:-1], seg[1:])):
            refs[k].step(bits[a:b], gdt, clip_coef=float(mult[k]))
    torch.cuda.synchronize()
    assert t == 3
    ph, mh, vh = p.cpu().numpy(), m.cpu().numpy(), vm.cpu().numpy()
    for k, (a, b) in enumerate(zip(seg[:-1], seg[1:])):
        gate(ph[a:b], refs[k].p, 1e-5, f"segment {k} p")
        gate(mh[a:b], refs[k].state.m, 1e-5, f"segment {k} m")
        gate(vh[a:b], refs[k].state.vmax, 1e-5, f"segment {k} vmax")


def _scaled_decoder_offsets(scale=32, layers=3):
    sizes = [int(np.prod([max(1, d // scale) for d in shape]))
             for _, shape in decoder_bucket_shapes()[:1 + 9 * layers]]
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def test_per_segment_clipped_step_vs_oracle(oracle_lib):
    seg = _scaled_decoder_offsets()
    n = int(seg[-1])
    w = dataclasses.replace(CONFIG4, segments=None, calls=4, inf_call=3, grad_sigma=1e-2).scaled(n)
    opts = w.options()
    o = fa.options(**opts)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype=torch.float16, device=DEV)
    row_len = 256
    crow = fa.segment_rows(list(seg), row_len)
    rows_buf = fa.stats_buffer(crow[-1], DEV)
    scratch = torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV)
    reports = fa.stats_buffer(len(seg) - 1, DEV)
    refs = [oracle.OracleAdamW(w.params_host(np.arange(a, b)), opts, lib_=oracle_lib)
            for a, b in zip(seg[:-1], seg[1:])]
    max_norm = 0.05
    t = 0
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        before = p.clone()
        t, rep, norms, coefs = fa.fa_bucket_step_clipped_per_segment(
            list(seg), p, g, m, v, vm, t, o, fa.control(), max_norm, row_len, rows_buf, scratch,
            reports)
        bits = grad_bits_from_device(g)
        stats = _slice_stats(oracle_lib, bits, "f16", seg)
        any_bad = any(c > 0 for _, c in stats)
        assert bool(rep.skipped_nonfinite) == any_bad == (call == 3)
        if any_bad:
            torch.cuda.synchronize()
            assert torch.equal(p, before) and rep.updated == 0
            for r in refs:
                r.step(np.zeros(0, np.uint16), "f16", skip_update=True)
            continue
        for k, ((s, c), (a, b)) in enumerate(zip(stats, zip(seg[:-1], seg[1:]))):
            _, norm, coef = oracle_lib.clip_decision(s, c, max_norm)
            assert abs(norms[k] - norm) <= 1e-5 * norm + 1e-30
            assert abs(coefs[k] - coef) <= 1e-5 * coef
            refs[k].step(bits[a:b], "f16", clip_coef=coef)
        assert min(coefs) < 1.0 and max(coefs) <= 1.0
    torch.cuda.synchronize()
    assert t == 3
    ph = p.cpu().numpy()
    for k, (a, b) in enumerate(zip(seg[:-1], seg[1:])):
        gate(ph[a:b], refs[k].p, 1e-5, f"segment {k}")


def _gated_layout(kind):
    if kind == "mixed":  # steady steps on the shared-memory pipeline
        rng = np.random.default_rng(41)
        sizes = rng.integers(0, 3000, 230)
        sizes[::11] = rng.integers(150_000, 450_000, len(sizes[::11]))
        sizes[3::17] = 0
        return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    if kind == "many":  # 300 segments: two launches, the skip vote over all of them
        return _segments(42, 300, 4000, empty_every=7)
    if kind == "sparse":  # 110 of 120 segments empty: the scratch (3 words per group of
        # rows) is too small for the decided table, so every launch decides itself
        rng = np.random.default_rng(43)
        sizes = np.zeros(120, np.int64)
        sizes[::12] = rng.integers(150_000, 250_000, 10)
        return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    return _scaled_decoder_offsets()  # "small" and "offset": register and scalar kernels


@pytest.mark.parametrize("kind,gdt,maximize,scale", [
    ("mixed", "f16", False, 1.0), ("mixed", "bf16", True, 1.0), ("many", "f32", False, 1.0),
    ("small", "f16", False, 1.0), ("offset", "bf16", False, 1.0),
    # powers of two decide on the full grid; other scales keep the pipeline and the
    # persistent kernel, whose few CTAs take the FP64 divisions
    ("mixed", "f16", False, 3.0), ("many", "bf16", False, 0.1), ("small", "f16", True, 2.0 ** -4),
    ("sparse", "bf16", False, 1.0), ("sparse", "f16", True, 3.0)])
def test_per_segment_gated_equals_host_decision_bitwise(kind, gdt, maximize, scale):
    """The per-segment step decided on the device (every segment's coefficient and the
    skip taken on the device from the device-resident reports: once for the bucket in
    the scratch when it has room, else in each update launch) against the host-decided
    per-segment step, over four calls with a +Inf in the third: reports, parameters and
    every moment bit for bit, the +Inf call skipped by both.  Two layouts read the
    bucket's record through a mailbox (with the decision table, and without: the
    scratch too small): when the call returns, the record holds the exact total count
    and the total sum of squares within 1e-12 of the exact sum of the segments'."""
    seg = _gated_layout(kind)
    n = int(seg[-1])
    w = dataclasses.replace(CONFIG4, segments=None, calls=4, inf_call=3, grad_sigma=1e-2,
                            grad_dtype=gdt, maximize=maximize, gradient_scale=scale,
                            grad_premul=scale).scaled(n)
    o = fa.options(**w.options())
    off = 1 if kind == "offset" else 0  # state views 4 bytes off the gradient's alignment

    def state():
        full = [torch.zeros(n + off, device=DEV) for _ in range(4)]
        w.fill_params_device(full[0][off:])
        return full, [x[off:] for x in full]

    _, (pa, ma, va, vma) = state()
    _, (pb, mb, vb, vmb) = state()
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    row_len = 256
    crow = fa.segment_rows(list(seg), row_len)
    bufs = [(fa.stats_buffer(crow[-1], DEV), torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV),
             fa.stats_buffer(len(seg) - 1, DEV)) for _ in range(2)]
    max_norm = 0.05
    mailbox = fa.report_mailbox() if kind in ("mixed", "sparse") else None
    ta = tb = 0
    for call in range(1, 5):
        w.fill_grad_device(call, g)
        ta, rep, _, coefs = fa.fa_bucket_step_clipped_per_segment(
            list(seg), pa, g, ma, va, vma, ta, o, fa.control(scale), max_norm, row_len, *bufs[0])
        fa.fa_bucket_step_clipped_per_segment_gated(
            list(seg), pb, g, mb, vb, vmb, tb, o, fa.control(scale), max_norm, row_len, *bufs[1],
            mailbox=mailbox)
        if mailbox is not None:  # posted before the call returned
            words = mailbox.numpy().view(np.uint32)[:3].copy()
            floats = words.view(np.float32)
            posted = fa.FaStats(float(floats[0]), int(words[1]), float(floats[2]))
        rb = bufs[1][2].cpu()
        if not bool((rb[:, 1] != 0).any()):
            tb += 1
        torch.cuda.synchronize()
        if mailbox is not None:
            recs = [fa.FaStats(*x) for x in zip(rb[:, 0].view(torch.float32).tolist(),
                                                 rb[:, 1].tolist(),
                                                 rb[:, 2].view(torch.float32).tolist())]
            assert posted.nonfinite == sum(r.nonfinite for r in recs)
            if posted.nonfinite == 0:
                exact = math.fsum(fa.fa_stats_sum_sq(r) for r in recs)
                assert abs(fa.fa_stats_sum_sq(posted) - exact) <= 1e-12 * exact
        assert torch.equal(bufs[0][2], bufs[1][2]), f"call {call}: reports differ"
        assert bool(rep.skipped_nonfinite) == (call == 3) and ta == tb
        if call != 3:
            assert min(coefs) < 1.0
        for x, y, name in ((pa, pb, "p"), (ma, mb, "m"), (va, vb, "v"), (vma, vmb, "vmax")):
            assert torch.equal(x, y), f"call {call}: {name} differs"
    assert ta == tb == 3


@pytest.mark.parametrize("kind,gdt", [("mixed", "f16"), ("many", "bf16")])
def test_composed_step_with_decided_table_equals_host_decision_bitwise(kind, gdt):
    """The per-segment step composed from the public calls: the segment-aligned analysis,
    the chunk merges, then fa_bucket_update with seg_reports and seg_decided, the merge
    scratch reused as the decision table.  Against the host-decided one-call step over
    four calls with a +Inf in the third: reports, p, m, v and vmax bit for bit."""
    seg = _gated_layout(kind)
    n = int(seg[-1])
    w = dataclasses.replace(CONFIG4, segments=None, calls=4, inf_call=3, grad_sigma=1e-2,
                            grad_dtype=gdt).scaled(n)
    o = fa.options(**w.options())
    sa = [torch.zeros(n, device=DEV) for _ in range(4)]
    sb = [torch.zeros(n, device=DEV) for _ in range(4)]
    w.fill_params_device(sa[0])
    w.fill_params_device(sb[0])
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    crow = fa.segment_rows(list(seg), 256)
    nseg = len(seg) - 1
    bufs = [(fa.stats_buffer(crow[-1], DEV), torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV),
             fa.stats_buffer(nseg, DEV)) for _ in range(2)]
    assert bufs[1][1].numel() >= nseg + 1
    ta = tb = 0
    for call in range(1, 5):
        w.fill_grad_device(call, g)
        ta, rep, _, _ = fa.fa_bucket_step_clipped_per_segment(
            list(seg), sa[0], g, sa[1], sa[2], sa[3], ta, o, fa.control(), 0.05, 256, *bufs[0])
        rows_b, scr_b, rep_b = bufs[1]
        fa.fa_analyze_gradient(g, 256, rows_b, list(seg))
        fa.fa_merge_gradient_stats_chunks(rows_b, crow, scr_b, rep_b)
        fa.fa_bucket_update(list(seg), sb[0], g, sb[1], sb[2], sb[3], tb, o, fa.control(),
                            seg_reports=rep_b, max_grad_norm=0.05, seg_decided=scr_b)
        if not bool((rep_b.cpu()[:, 1] != 0).any()):
            tb += 1
        torch.cuda.synchronize()
        assert torch.equal(bufs[0][2], rep_b), f"call {call}: reports differ"
        assert bool(rep.skipped_nonfinite) == (call == 3) and ta == tb
        for x, y, name in zip(sa, sb, ("p", "m", "v", "vmax")):
            assert torch.equal(x, y), f"call {call}: {name} differs"
    assert ta == tb == 3


def test_per_segment_gated_mailbox_rules():
    """The one-call per-segment step's optional mailbox: pageable host memory and device
    memory are rejected (FA_ERR_POINTER) before anything is enqueued, with every buffer
    untouched; NULL runs the call without waiting."""
    import ctypes
    from amsgrad_optimizer_step_gb300 import _lib
    seg = _segments(44, 20, 3000)
    n = int(seg[-1])
    w = dataclasses.replace(CONFIG4, segments=None).scaled(n)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype=torch.float16, device=DEV)
    w.fill_grad_device(1, g)
    crow = fa.segment_rows(list(seg), 256)
    rows = fa.stats_buffer(crow[-1], DEV)
    scr = torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV)
    rep = fa.stats_buffer(len(seg) - 1, DEV)
    rep.fill_(7)
    o = fa.options(**w.options())
    lib = _lib.load()
    table = (ctypes.c_int64 * len(seg))(*[int(x) for x in seg])
    snap = [x.clone() for x in (p, m, v, vm, rep)]

    def raw(mailbox_ptr):
        return lib.fa_bucket_step_clipped_per_segment_gated(
            table, len(seg) - 1, n, p.data_ptr(), g.data_ptr(), 1, m.data_ptr(), v.data_ptr(),
            vm.data_ptr(), 0, ctypes.byref(o), fa.control(), 0.05, 256, rows.data_ptr(),
            rows.shape[0], scr.data_ptr(), scr.numel(), rep.data_ptr(), mailbox_ptr, None)

    pageable = np.zeros(4, np.uint32)
    assert raw(pageable.ctypes.data) == 6
    on_device = torch.zeros(4, dtype=torch.int32, device=DEV)
    assert raw(on_device.data_ptr()) == 6
    torch.cuda.synchronize()
    for a, b in zip((p, m, v, vm, rep), snap):
        assert torch.equal(a, b)
    assert raw(None) == 0
    torch.cuda.synchronize()
    assert not torch.equal(p, snap[0])  # the update ran


def test_per_segment_clipped_full_size_sampled(oracle_lib):
    """The per-parameter clipped step on the whole 1,195,991,040-parameter decoder bucket
    (199 segments, FP16 gradients, AMSGrad, rows of 512), in the launch configuration the
    benchmark times. Every segment's report and clip coefficient is checked against the
    oracle over that segment's full gradient. Sampled elements are checked one step from
    identical state and along the trajectory. Call 3 carries +Inf and is skipped.  The
    same step decided on the device runs beside it on a copy of the state and must match
    it bit for bit over every element after every call."""
    w = dataclasses.replace(CONFIG4, calls=4, inf_call=3)
    seg = np.asarray(w.segments, dtype=np.int64)
    n = w.n
    opts = w.options()
    o = fa.options(**opts)
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v, vm = (torch.zeros(n, device=DEV) for _ in range(3))
    g = torch.empty(n, dtype=torch.float16, device=DEV)
    row_len = 512
    crow = fa.segment_rows(list(seg), row_len)
    rows_buf = fa.stats_buffer(crow[-1], DEV)
    scratch = torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV)
    reports = fa.stats_buffer(len(seg) - 1, DEV)
    dev_state = [x.clone() for x in (p, m, v, vm)]
    dev_bufs = (fa.stats_buffer(crow[-1], DEV), torch.empty_like(scratch),
                fa.stats_buffer(len(seg) - 1, DEV))
    t_dev = 0
    rng = np.random.default_rng(40)
    ends = np.concatenate([seg[1:-1], seg[1:-1] - 1, [0, n - 1, w.inf_index()]])
    idx = np.unique(np.concatenate([rng.integers(0, n, 40000), ends]))
    idx_t = torch.as_tensor(idx, device=DEV)
    kseg = np.searchsorted(seg, idx, side="right") - 1
    groups = [np.nonzero(kseg == k)[0] for k in range(len(seg) - 1)]
    assert all(len(gk) >= 2 for gk in groups)
    refs = [oracle.OracleAdamW(w.params_host(idx[gk]), opts, lib_=oracle_lib) for gk in groups]
    max_norm = 0.01
    t = 0
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        before = [x[idx_t].double().cpu().numpy() for x in (p, m, v, vm)]
        t_before = t
        t, rep, norms, coefs = fa.fa_bucket_step_clipped_per_segment(
            list(seg), p, g, m, v, vm, t, o, fa.control(), max_norm, row_len, rows_buf,
            scratch, reports)
        pd, md, vd, vmd = dev_state
        fa.fa_bucket_step_clipped_per_segment_gated(list(seg), pd, g, md, vd, vmd, t_dev, o,
                                                    fa.control(), max_norm, row_len, *dev_bufs)
        if not bool((dev_bufs[2][:, 1] != 0).any()):
            t_dev += 1
        torch.cuda.synchronize()
        assert t_dev == t and torch.equal(dev_bufs[2], reports)
        for x, y, name in zip((p, m, v, vm), dev_state, ("p", "m", "v", "vmax")):
            assert torch.equal(x, y), f"call {call}: decided on the device, {name} differs"
        bits = grad_bits_from_device(g)
        assert np.array_equal(bits[idx], w.grad_host(call, idx)), "device/host grads differ"
        stats = _slice_stats(oracle_lib, bits, "f16", seg)
        del bits
        after = [x[idx_t].double().cpu().numpy() for x in (p, m, v, vm)]
        bad = call == w.inf_call
        assert bool(rep.skipped_nonfinite) == bad == any(c > 0 for _, c in stats)
        if bad:
            assert t == t_before and rep.updated == 0
            for a, b in zip(before, after):
                assert np.array_equal(a, b), "skipped call changed state"
            for r in refs:
                r.step(np.zeros(0, np.uint16), "f16", skip_update=True)
            continue
        assert t == t_before + 1 and rep.updated == 1
        gh = w.grad_host(call, idx)
        for k, ((s_k, c_k), gk) in enumerate(zip(stats, groups)):
            _, norm, coef = oracle_lib.clip_decision(s_k, c_k, max_norm)
            assert abs(norms[k] - norm) <= 1e-5 * norm + 1e-30, (call, k, norms[k], norm)
            assert abs(coefs[k] - coef) <= 1e-5 * coef, (call, k, coefs[k], coef)
            zero = np.zeros(len(gk))
            b4 = (before[0][gk], zero, zero, zero) if t_before == 0 else \
                tuple(b[gk] for b in before)
            one = oracle_one_step(gh[gk], "f16", opts, 1.0, float(coefs[k]), t, b4, oracle_lib)
            for j, name in enumerate(("p", "m", "v", "vmax")):
                gate(after[j][gk], one[j], 1e-6, f"call {call} segment {k} one-step {name}")
            refs[k].step(gh[gk], "f16", clip_coef=coef)
            gate(after[0][gk], refs[k].p, 1e-5, f"call {call} segment {k} trajectory p")
            gate(after[3][gk], refs[k].state.vmax, 1e-5, f"call {call} segment {k} trajectory vmax")
        assert min(coefs) < 1.0
    assert t == 3
