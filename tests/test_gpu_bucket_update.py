"""fa_bucket_update in seeded random variants against the oracle.

Every variant of the bucket update is one call with a descriptor: the multiplier from
a host factor, one host factor per segment, one device report or one device report
per segment, and optionally the low-precision model copy.  Each case draws a variant,
(one device report per segment, half of the time with the decisions taken once in a
table first), a size (1 to 2.5 million), a segment table with empty segments, the
gradient dtype,
AMSGrad, maximize, a loss scale (a power of two in two cases of three, which a gated
launch runs on the full grid; else 3, 0.3 or 1000, which it runs on the pipeline), a
clip threshold (or none) and a skipped call, and runs three calls.  Each segment is compared with its own oracle run
(trajectory within 1e-5 x max(1,|x|)), whose coefficient is the host factor, or the
oracle's own decision from its FP64 statistics over the whole gradient or over the
segment.  The model copy must be the encoding of the device's own parameters and a
rounding of the oracle's.
"""

import dataclasses

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
import oracle
from gpu_harness import TORCH_DT, check_model_copy, gate
from synthetic.configs import CONFIG2

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
MODEL_DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


def _case(k):
    rng = np.random.default_rng(9000 + k)
    n = int(rng.choice([1, 17, 4097, 100_003, 1_000_003, 2_500_001]))
    nseg = int(rng.integers(1, 40))
    cuts = np.sort(rng.integers(0, n + 1, nseg - 1))
    seg = [0] + [int(c) for c in cuts] + [n]
    # every source, and both model copies with each single-factor source, by case index
    source = ("host", "seg_host", "report", "seg_reports")[k % 4]
    model = ("none", "bf16", "f16")[(k // 4) % 3] if source in ("host", "report") else "none"
    # powers of two (the gated full grid) and other scales (the gated pipeline)
    scale = float(2.0 ** rng.integers(-2, 7)) if rng.integers(3) else float(
        rng.choice([3.0, 0.3, 1000.0]))
    w = dataclasses.replace(
        CONFIG2, name=f"bucket_update{k}", seed=int(rng.integers(1, 10_000)),
        grad_dtype=str(rng.choice(["f32", "f16", "bf16"])), amsgrad=bool(rng.integers(2)),
        maximize=bool(rng.integers(2)), gradient_scale=scale, grad_premul=scale, calls=3,
        skip_calls=(2,) if rng.integers(2) else (), weight_decay=float(rng.choice([0.0, 0.01])),
        max_grad_norm=float(rng.choice([0.0, 1e-3, 0.05, 10.0]))).scaled(n)
    return w, seg, source, model, rng


@pytest.mark.parametrize("k", range(16))
def test_bucket_update_random_variant_vs_oracle(k, oracle_lib):
    w, seg, source, model, rng = _case(k)
    n, gdt, opts = w.n, w.grad_dtype, w.options()
    o = fa.options(**opts)
    nseg = len(seg) - 1
    p = torch.empty(n, device=DEV)
    w.fill_params_device(p)
    m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    vmax = torch.zeros(n, device=DEV) if w.amsgrad else None
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    p_model = torch.zeros(n, dtype=MODEL_DT[model], device=DEV) if model != "none" else None
    refs = [oracle.OracleAdamW(w.params_host(np.arange(a, b)), opts, storage="f32",
                               lib_=oracle_lib) for a, b in zip(seg[:-1], seg[1:])]
    if source == "report":
        rows = fa.fa_stats_rows(n, 256, seg)
        rows_buf, scratch = fa.stats_buffer(rows, DEV), fa.scratch_buffer(rows, DEV)
        report = fa.stats_buffer(1, DEV)
    elif source == "seg_reports":
        crow = fa.segment_rows(seg, 256)
        rows_buf = fa.stats_buffer(crow[-1], DEV)
        scratch = torch.empty(max(1, fa.fa_stats_chunk_scratch(crow)), device=DEV)
        report = fa.stats_buffer(nseg, DEV)
    # half of the per-segment device decisions take them once in a table first
    decided = (torch.full((nseg + 1,), float("nan"), device=DEV)
               if source == "seg_reports" and (k // 4) % 2 else None)
    t = 0
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        bits = w.grad_host(call, np.arange(n))
        skip = call in w.skip_calls
        ctl = fa.control(w.gradient_scale, skip)
        kw = {}
        if source == "host":
            c = float(rng.uniform(0.1, 1.0))
            coefs = [c] * nseg
            kw = dict(grad_mult=c)
        elif source == "seg_host":
            coefs = [float(x) for x in rng.uniform(0.1, 1.0, nseg)]
            kw = dict(seg_grad_mult=coefs)
        elif source == "report":
            s, cnt = oracle_lib.gradient_stats(bits, gdt, w.gradient_scale)
            coefs = [oracle_lib.clip_decision(s, cnt, w.max_grad_norm)[2]] * nseg
            if not skip:
                fa.fa_analyze_gradient(g, 256, rows_buf, seg)
                fa.fa_merge_gradient_stats(rows_buf, rows, scratch, report)
            kw = dict(report=report, max_grad_norm=w.max_grad_norm)
        else:
            coefs = []
            for a, b in zip(seg[:-1], seg[1:]):
                s, cnt = oracle_lib.gradient_stats(bits[a:b], gdt, w.gradient_scale)
                coefs.append(oracle_lib.clip_decision(s, cnt, w.max_grad_norm)[2])
            if not skip:
                fa.fa_analyze_gradient(g, 256, rows_buf, seg)
                fa.fa_merge_gradient_stats_chunks(rows_buf, crow, scratch, report)
            kw = dict(seg_reports=report, max_grad_norm=w.max_grad_norm, seg_decided=decided)
        enq = fa.fa_bucket_update(seg, p, g, m, v, vmax, t, o, ctl, p_model=p_model, **kw)
        assert enq == (not skip and n > 0)
        t += int(enq)  # no gradient here is non-finite: a device decision never skips
        for ref, (a, b), c in zip(refs, zip(seg[:-1], seg[1:]), coefs):
            ref.step(bits[a:b], gdt, w.gradient_scale, skip_update=skip, clip_coef=c)
    torch.cuda.synchronize()
    assert t == w.calls - len(w.skip_calls)
    host = {"p": p.cpu().numpy(), "m": m.cpu().numpy(), "v": v.cpu().numpy()}
    if vmax is not None:
        host["vmax"] = vmax.cpu().numpy()
    for j, (ref, (a, b)) in enumerate(zip(refs, zip(seg[:-1], seg[1:]))):
        if b == a:
            continue
        assert ref.state.t == t
        gate(host["p"][a:b], ref.p, 1e-5, f"case {k} ({source}) segment {j} p")
        gate(host["m"][a:b], ref.state.m, 1e-5, f"case {k} segment {j} m")
        gate(host["v"][a:b], ref.state.v, 1e-5, f"case {k} segment {j} v")
        if vmax is not None:
            gate(host["vmax"][a:b], ref.state.vmax, 1e-5, f"case {k} segment {j} vmax")
    if p_model is not None and n > 0:
        ref_p = np.concatenate([r.p for r, (a, b) in zip(refs, zip(seg[:-1], seg[1:])) if b > a])
        bits_model = p_model.view(torch.int16).cpu().numpy().view(np.uint16)
        check_model_copy(bits_model, host["p"], ref_p.astype(np.float32), model, oracle_lib,
                         f"case {k} model copy")


def test_bucket_update_rejections_leave_everything_untouched():
    """Reports or a model copy overlapping the state or the gradient, a model copy with a
    per-segment source, two sources at once, a host factor beside a device report, a
    decision table without per-segment reports, too small or inside the state: each
    rejected before anything is enqueued, every buffer bit-identical afterwards."""
    n = 1 << 20
    p, m, v = (torch.randn(n, device=DEV) for _ in range(3))
    g = torch.randn(n, device=DEV).to(torch.bfloat16)
    report = fa.stats_buffer(4, DEV)
    report.zero_()
    model = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    snap = [x.clone() for x in (p, m, v, g, report, model)]
    o, ctl = fa.options(), fa.control()
    seg = [0, n // 2, n]
    cases = [
        (5, dict(report=m.view(torch.int32)[:3].view(1, 3))),               # report inside m
        (5, dict(seg_reports=v.view(torch.int32)[:6].view(2, 3), max_grad_norm=1.0)),
        (5, dict(p_model=g)),                                                # copy over g
        (5, dict(p_model=p.view(torch.bfloat16)[:n])),                       # copy over p
        (4, dict(seg_grad_mult=[1.0, 1.0], p_model=model)),                  # no such kernel
        (4, dict(report=report[:1], seg_reports=report[:2])),                # two sources
        (4, dict(report=report[:1], grad_mult=0.5)),                         # factor + report
        (4, dict(report=report[:1], seg_decided=torch.empty(3, device=DEV))),  # table, no seg
        (3, dict(seg_reports=report[:2], max_grad_norm=1.0,
                 seg_decided=torch.empty(2, device=DEV))),                   # table too small
        (5, dict(seg_reports=report[:2], max_grad_norm=1.0, seg_decided=m[:3])),  # table in m
    ]
    for status, kw in cases:
        with pytest.raises(fa.FusedAdamWError) as e:
            fa.fa_bucket_update(seg, p, g, m, v, None, 3, o, ctl, **kw)
        assert e.value.status == status, (kw.keys(), e.value.status)
    torch.cuda.synchronize()
    for a, b in zip((p, m, v, g, report, model), snap):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
