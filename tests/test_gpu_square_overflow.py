"""Finite gradient values whose squares leave FP32's range, against the oracle.

A finite value above about 1.8e19 (possible in FP32 and BF16 storage) squares
past FP32's largest value, so a row's FP32 sum of squares overflows although
the row holds no NaN or +-Inf.  Such a row is summed again with its values
scaled by 2^-96 and its record carries the scaled sum (negated, so that the
sign marks the form); merges move to the scaled domain when they meet one or
when a partial sum reaches 2^126.  The step must then behave as the oracle's
FP64 sum says ("训练与状态保存", section "在 ruda:0 上进行原生 PyTorch 训练": only
non-finite values skip the step, and the global L2 clip uses the norm of the
unscaled gradient): no skip, the true norm within 1e-5, the oracle's clip
coefficient and update.  Sums are decoded with the library's fa_stats_sum_sq.
"""

import math

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
from gpu_harness import run_workload
from synthetic.configs import CONFIG5

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()
    torch.cuda.init()


def _grad(n, gdt, seed, planted):
    """N(0, 1e-2) values with ``planted`` {index: value} written over them."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    for i, val in planted.items():
        x[i] = np.float32(val)
    t = torch.from_numpy(x).to(TORCH_DT[gdt])
    bits = t.numpy() if gdt == "f32" else t.view(torch.int16).numpy().view(np.uint16)
    return t.to(DEV), bits


def _record(hi, count, lo):
    r = fa.FaStats()
    r.sum_sq, r.nonfinite, r.sum_sq_lo = float(hi), int(count), float(lo)
    return r


def _decoded(host):
    """Sums of squares of an (rows, 3) int32 record array: plain records added here,
    scaled ones (negative first word) decoded by the library."""
    hi = host[:, 0].view(torch.float32).double().numpy()
    lo = host[:, 2].view(torch.float32).double().numpy()
    cnt = host[:, 1].numpy().astype(np.int64)
    out = hi + lo
    for r in np.flatnonzero(hi < 0):
        out[r] = fa.fa_stats_sum_sq(_record(hi[r], cnt[r], lo[r]))
    return out, cnt, int((hi < 0).sum())


def _report_sum(report):
    h = fa.fa_read_report(report)
    return fa.fa_stats_sum_sq(h), int(h.nonfinite), h.sum_sq < 0


# (n, row_len, segments): the fast kernel with whole rows, with short rows at segment
# ends, and the generic kernel (rows not a whole number of 512-byte chunks)
LAYOUTS = [(256 * 600, 256, None),
           (256 * 600 + 77, 256, [0, 5000, 5000, 70_001, 256 * 600 + 77]),
           (100_003, 300, None)]


@pytest.mark.parametrize("gdt", ["f32", "bf16"])
@pytest.mark.parametrize("n,row_len,segs", LAYOUTS)
def test_rows_and_report_with_squares_beyond_fp32(gdt, n, row_len, segs, oracle_lib):
    big = 3.0e38 if gdt == "f32" else 3.3e38
    planted = {0: 1e20, 777: -big, n - 1: 2.5e19, n // 2: 4e19, 4999: 1e25}
    # one whole row of 1.5e19 values: each square is finite, their sum is not
    r0 = (n // row_len // 3) * row_len
    for i in range(r0, r0 + row_len):
        planted[i] = 1.5e19
    g, bits = _grad(n, gdt, 31, planted)
    rows = fa.fa_stats_rows(n, row_len, segs)
    buf = fa.stats_buffer(rows, DEV)
    assert fa.fa_analyze_gradient(g, row_len, buf, segs) == rows
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    fa.fa_merge_gradient_stats(buf, rows, scratch, report)
    torch.cuda.synchronize()
    got, cnt, rescued = _decoded(buf.cpu())
    rs, rc = oracle_lib.row_stats(bits, gdt, row_len, segs)
    assert np.array_equal(cnt, rc.astype(np.int64)) and not rc.any()
    assert rescued >= 5, rescued  # the rows above took the scaled form
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - rs) <= 2e-6 * rs + 1e-30)
    s, c, scaled = _report_sum(report)
    s_or, c_or = oracle_lib.gradient_stats(bits, gdt)
    assert c == c_or == 0 and scaled
    assert abs(s - math.fsum(got.tolist())) <= 1e-12 * s
    assert abs(s - s_or) <= 2e-6 * s_or
    # the decision: finite norm, tiny positive coefficient, no skip
    skip, norm, coef = fa.fa_clip_decision(s, c, 1.0, 1.0)
    o_skip, o_norm, o_coef = oracle_lib.clip_decision(s_or, c_or, 1.0)
    assert not skip and not o_skip
    assert abs(norm - o_norm) <= 1e-5 * o_norm
    assert 0 < o_coef < 1e-19 and abs(coef - o_coef) <= 1e-5 * o_coef


@pytest.mark.parametrize("gdt", ["f32", "bf16"])
def test_non_finite_rows_still_counted_beside_overflowing_ones(gdt, oracle_lib):
    """Rows holding a huge finite value and a NaN or +Inf: counts exact (the step is
    skipped), no rescue (their sums are not used), other rows as the oracle's."""
    n = 256 * 64
    g, bits = _grad(n, gdt, 32, {5: 1e30, 9: float("nan"), 300: 2e30, 301: float("inf")})
    rows = fa.fa_stats_rows(n, 256)
    buf = fa.stats_buffer(rows, DEV)
    fa.fa_analyze_gradient(g, 256, buf)
    torch.cuda.synchronize()
    host = buf.cpu()
    rs, rc = oracle_lib.row_stats(bits, gdt, 256)
    cnt = host[:, 1].numpy().astype(np.int64)
    assert np.array_equal(cnt, rc.astype(np.int64)) and cnt[0] == 1 and cnt[1] == 1
    got, _, rescued = _decoded(host)
    assert rescued == 0  # rows with a non-finite value keep their (unused) plain sum
    ok = rc == 0
    assert np.all(np.abs(got - rs)[ok] <= 2e-6 * rs[ok] + 1e-30)


@pytest.mark.parametrize("value,rows", [(5e37, 3000), (2e38, 3000), (5e37, 1_048_577)])
def test_merge_moves_to_the_scaled_domain(value, rows):
    """Plain records whose total passes FP32's range (each below 2^126, so the switch
    comes from the partial sum; each above it; and over three merge levels), mixed
    with small records and a few scaled ones: the report is the exact sum of the
    decoded records within 1e-12."""
    rng = np.random.default_rng(rows)
    hi = (value * (0.5 + rng.random(rows))).astype(np.float32)
    small = rng.random(rows) < 0.5
    hi[small] = (rng.random(int(small.sum())) * 10).astype(np.float32)
    lo = np.zeros(rows, np.float32)
    scaled = rng.choice(rows, 3, replace=False)
    # scaled records standing for sums near 1e41, comparable to the plain total
    hi[scaled] = -np.float32(1e-17) * (1 + rng.random(3)).astype(np.float32)
    host = torch.zeros((rows, 3), dtype=torch.int32)
    host[:, 0] = torch.from_numpy(hi).view(torch.int32)
    host[:, 2] = torch.from_numpy(lo).view(torch.int32)
    want, _, nscaled = _decoded(host)
    assert nscaled == 3
    recs = host.to(DEV)
    scratch = fa.scratch_buffer(rows, DEV)
    report = fa.stats_buffer(1, DEV)
    fa.fa_merge_gradient_stats(recs, rows, scratch, report)
    s, c, is_scaled = _report_sum(report)
    exact = math.fsum(want.tolist())
    assert c == 0 and is_scaled and math.isfinite(s)
    assert abs(s - exact) <= 1e-12 * exact


@pytest.mark.parametrize("gdt,value", [("bf16", 1e20), ("f32", 1e30)])
def test_clipped_step_with_an_overflowing_finite_value_vs_oracle(gdt, value):
    """The statistics-guarded step with one finite value whose square overflows FP32
    planted in the second of three calls: nothing skipped, the reported norm and clip
    coefficient within 1e-5 of the oracle's, every element of every call against the
    oracle (one step from identical state and the trajectory)."""
    w = CONFIG5.scaled(256 * 5000 + 77, calls=3, inf_call=2, inf_value=value,
                       grad_dtype=gdt)
    s = run_workload(w, w.n, "clipped", DEV, row_len=256)
    assert s["skips"] == 0 and s["updates"] == 3 and s["t"] == 3
    norm_dev, norm_or, nonfinite, _ = s["reports"][1]
    assert nonfinite == 0 and norm_or > value / 2
    assert abs(norm_dev - norm_or) <= 1e-5 * norm_or


def test_gated_steps_equal_host_decided_with_an_overflowing_value():
    """The update deciding on the device from a scaled report is bit-identical to the
    host's decision: whole-bucket clip and per-segment clip, with the huge finite
    value in the second of three calls."""
    n = 256 * 5000 + 77
    w = CONFIG5.scaled(n, calls=3, inf_call=2, inf_value=1e20)
    k = w.inf_index()
    seg = sorted([0, 7, 400_000, 400_000, k + 1, n])  # the huge value ends a segment
    assert seg[-2] == k + 1 < n
    crow = fa.segment_rows(seg, 256)
    mailbox = fa.report_mailbox()
    states = []
    for mode in ("host", "gated", "seg_host", "seg_gated"):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        m, v = torch.empty_like(p), torch.empty_like(p)
        g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        per_seg = mode.startswith("seg")
        rows = crow[-1] if per_seg else fa.fa_stats_rows(n, 256)
        rb = fa.stats_buffer(rows, DEV)
        sc = (torch.empty(fa.fa_stats_chunk_scratch(crow), device=DEV) if per_seg
              else fa.scratch_buffer(rows, DEV))
        rep = fa.stats_buffer(len(seg) - 1 if per_seg else 1, DEV)
        o = fa.options(**w.options())
        t, out = 0, []
        for call in range(1, w.calls + 1):
            w.fill_grad_device(call, g)
            if mode == "host":
                t, r = fa.fa_bucket_step_clipped(None, p, g, m, v, None, t, o, fa.control(),
                                                 1.0, 256, rb, sc, rep)
                out.append((r.skipped_nonfinite, repr(r.grad_norm), repr(r.clip_coef)))
            elif mode == "gated":
                t, r = fa.fa_bucket_step_clipped_gated(None, p, g, m, v, None, t, o,
                                                       fa.control(), 1.0, 256, rb, sc, rep,
                                                       mailbox)
                out.append((r.skipped_nonfinite, repr(r.grad_norm), repr(r.clip_coef)))
            elif mode == "seg_host":
                t, r, norms, coefs = fa.fa_bucket_step_clipped_per_segment(
                    seg, p, g, m, v, None, t, o, fa.control(), 1.0, 256, rb, sc, rep)
                out.append(tuple(repr(c) for c in coefs))
            else:
                fa.fa_bucket_step_clipped_per_segment_gated(seg, p, g, m, v, None, t, o,
                                                            fa.control(), 1.0, 256, rb, sc,
                                                            rep)
                torch.cuda.synchronize()
                host = rep.cpu()
                t += 0 if bool(host[:, 1].any()) else 1
                coefs = []
                for k in range(len(seg) - 1):
                    rec = _record(host[k, 0:1].view(torch.float32).item(), int(host[k, 1]),
                                  host[k, 2:3].view(torch.float32).item())
                    coefs.append(fa.fa_clip_decision(fa.fa_stats_sum_sq(rec), 0, 1.0, 1.0)[2])
                out.append(tuple(repr(c) for c in coefs))
            torch.cuda.synchronize()
        states.append((t, out, p.clone(), m.clone(), v.clone()))
    for a, b in ((0, 1), (2, 3)):
        ta, oa, *xa = states[a]
        tb, ob, *xb = states[b]
        assert ta == tb == 3 and oa == ob, (oa, ob)
        for x, y in zip(xa, xb):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    # the whole-bucket clip saw the huge value: coefficient far below 1 on call 2
    assert float(states[0][1][1][2]) < 1e-19
