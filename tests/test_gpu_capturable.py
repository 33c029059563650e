"""The step with a device-resident count (fa_device_step) against the host-decided path.

The decision kernel repeats the host's FP64 operations in the host's order, so the
two paths must agree bit for bit: parameters, moments, the step count, the skip
flag, the norm and the clip coefficient.  The host path itself is checked against
the oracle elsewhere; here every comparison is exact.  The same step is captured
once into a CUDA graph and replayed for every step.
"""

import dataclasses

import numpy as np
import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
from gpu_harness import TORCH_DT
from synthetic.configs import CONFIG2, CONFIG5

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


class Run:
    """One optimizer state (p, m, v[, vmax]) with its statistics buffers."""

    def __init__(self, w, n, row_len):
        self.p = torch.empty(n, device=DEV)
        w.fill_params_device(self.p)
        self.m = torch.zeros(n, device=DEV)
        self.v = torch.zeros(n, device=DEV)
        self.vmax = torch.zeros(n, device=DEV) if w.amsgrad else None
        self.rows = fa.stats_buffer(fa.fa_stats_rows(n, row_len), DEV)
        self.scratch = fa.scratch_buffer(self.rows.shape[0], DEV)
        self.report = fa.stats_buffer(1, DEV)
        self.dstep = fa.device_step_buffer(DEV)
        self.t = 0

    def state(self):
        return [x for x in (self.p, self.m, self.v, self.vmax) if x is not None]


def _workload(gdt, ams, maximize, n, scale):
    return dataclasses.replace(CONFIG5, grad_dtype=gdt, amsgrad=ams, maximize=maximize,
                               gradient_scale=scale, grad_premul=scale, calls=6,
                               inf_call=4).scaled(n)


def _same(a, b):
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(a, b))


@pytest.mark.parametrize("n", [100_003, 3_000_001])
@pytest.mark.parametrize("gdt,ams,maximize,scale", [
    ("bf16", False, False, 1.0), ("f16", True, False, 128.0), ("f32", True, True, 4.0),
    ("f32", False, False, 1.0)])
def test_clipped_capturable_equals_clipped_bitwise(n, gdt, ams, maximize, scale):
    w = _workload(gdt, ams, maximize, n, scale)
    row_len = 256
    host, dev = Run(w, n, row_len), Run(w, n, row_len)
    g = torch.empty(n, dtype=TORCH_DT[gdt], device=DEV)
    o = fa.options(**w.options())
    ctl = fa.control(scale)
    max_norm = 0.05
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        host.t, rep = fa.fa_bucket_step_clipped(None, host.p, g, host.m, host.v, host.vmax,
                                                host.t, o, ctl, max_norm, row_len, host.rows,
                                                host.scratch, host.report)
        fa.fa_bucket_step_clipped_capturable(None, dev.p, g, dev.m, dev.v, dev.vmax, dev.dstep,
                                             o, ctl, max_norm, row_len, dev.rows, dev.scratch,
                                             dev.report)
        torch.cuda.synchronize()
        d = fa.read_device_step(dev.dstep)
        assert d.t == host.t, (call, d.t, host.t)
        assert d.skipped == rep.skipped_nonfinite == (call == w.inf_call)
        assert d.nonfinite == rep.nonfinite
        assert d.grad_norm == rep.grad_norm or (np.isnan(d.grad_norm) and np.isnan(rep.grad_norm))
        assert d.clip_coef == rep.clip_coef
        if call != w.inf_call:
            assert rep.clip_coef < 1.0
        assert _same(host.state(), dev.state()), f"call {call}: states differ"
    assert host.t == w.calls - 1


@pytest.mark.parametrize("n", [1, 9, 4097, 2_000_000])
def test_capturable_without_report_equals_bucket_step_bitwise(n):
    w = dataclasses.replace(CONFIG2, calls=5, skip_calls=()).scaled(n)
    host, dev = Run(w, n, 256), Run(w, n, 256)
    g = torch.empty(n, dtype=TORCH_DT[w.grad_dtype], device=DEV)
    o = fa.options(**w.options())
    ctl = fa.control(w.gradient_scale)
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        host.t, _ = fa.fa_bucket_step(None, host.p, g, host.m, host.v, host.vmax, host.t, o, ctl)
        fa.fa_bucket_step_capturable(None, dev.p, g, dev.m, dev.v, dev.vmax, dev.dstep, o, ctl)
        torch.cuda.synchronize()
        d = fa.read_device_step(dev.dstep)
        assert d.t == host.t == call and d.skipped == 0 and d.clip_coef == 1.0
        assert _same(host.state(), dev.state()), f"call {call}"


def test_skip_update_enqueues_nothing():
    n = 4097
    w = CONFIG2.scaled(n)
    r = Run(w, n, 256)
    g = torch.ones(n, dtype=torch.bfloat16, device=DEV)
    o = fa.options(**w.options())
    before = [x.clone() for x in r.state()]
    rec = r.dstep.clone()
    fa.fa_bucket_step_capturable(None, r.p, g, r.m, r.v, r.vmax, r.dstep, o,
                                 fa.control(128.0, skip_update=True))
    torch.cuda.synchronize()
    assert _same(before, r.state()) and torch.equal(rec, r.dstep)


def test_cuda_graph_replay_equals_host_path_bitwise():
    """One capture of the whole statistics-guarded step, replayed for every step with a
    fresh gradient copied into the captured buffer; the first step and a non-finite skip
    happen inside replays."""
    n = 1_500_007
    w = _workload("bf16", True, False, n, 1.0)
    row_len = 256
    host, dev = Run(w, n, row_len), Run(w, n, row_len)
    o = fa.options(**w.options())
    ctl = fa.control(1.0)
    max_norm = 0.05
    g_static = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    grads = []
    for call in range(1, w.calls + 1):
        gk = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        w.fill_grad_device(call, gk)
        grads.append(gk)

    # warm-up on other buffers of the same shape (kernel attributes, occupancy caches)
    warm = Run(w, n, row_len)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g_static.copy_(grads[0])
        for _ in range(2):
            fa.fa_bucket_step_clipped_capturable(None, warm.p, g_static, warm.m, warm.v,
                                                 warm.vmax, warm.dstep, o, ctl, max_norm,
                                                 row_len, warm.rows, warm.scratch, warm.report)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_bucket_step_clipped_capturable(None, dev.p, g_static, dev.m, dev.v, dev.vmax,
                                             dev.dstep, o, ctl, max_norm, row_len, dev.rows,
                                             dev.scratch, dev.report)
    torch.cuda.synchronize()
    d = fa.read_device_step(dev.dstep)
    assert d.t == 0, "capture must not execute"

    for call in range(1, w.calls + 1):
        g_static.copy_(grads[call - 1])
        graph.replay()
        host.t, rep = fa.fa_bucket_step_clipped(None, host.p, grads[call - 1], host.m, host.v,
                                                host.vmax, host.t, o, ctl, max_norm, row_len,
                                                host.rows, host.scratch, host.report)
        torch.cuda.synchronize()
        d = fa.read_device_step(dev.dstep)
        assert d.t == host.t and d.skipped == rep.skipped_nonfinite
        assert d.clip_coef == rep.clip_coef
        assert _same(host.state(), dev.state()), f"replay {call}: states differ"
    assert host.t == w.calls - 1


def test_full_size_stats_clip_workload_bitwise():
    """The 1,073,741,824-parameter BF16 workload with its +Inf call, through the
    capturable step and through the host-decided step: identical at every call."""
    w = CONFIG5
    n = w.n
    row_len = w.row_len
    host, dev = Run(w, n, row_len), Run(w, n, row_len)
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    o = fa.options(**w.options())
    ctl = fa.control(w.gradient_scale)
    for call in range(1, w.calls + 1):
        w.fill_grad_device(call, g)
        host.t, rep = fa.fa_bucket_step_clipped(None, host.p, g, host.m, host.v, None, host.t,
                                                o, ctl, w.max_grad_norm, row_len, host.rows,
                                                host.scratch, host.report)
        fa.fa_bucket_step_clipped_capturable(None, dev.p, g, dev.m, dev.v, None, dev.dstep, o,
                                             ctl, w.max_grad_norm, row_len, dev.rows,
                                             dev.scratch, dev.report)
        torch.cuda.synchronize()
        d = fa.read_device_step(dev.dstep)
        assert d.t == host.t and d.skipped == rep.skipped_nonfinite == (call == w.inf_call)
        assert d.grad_norm == rep.grad_norm or call == w.inf_call
        assert torch.equal(host.p, dev.p) and torch.equal(host.m, dev.m)
        assert torch.equal(host.v, dev.v)
    assert host.t == 4


def test_capturable_rejections_leave_everything_untouched():
    n = 4097
    w = CONFIG2.scaled(n)
    r = Run(w, n, 256)
    g = torch.ones(n, dtype=torch.bfloat16, device=DEV)
    o = fa.options(**w.options())
    ctl = fa.control(128.0)
    before = [x.clone() for x in r.state()]
    host_rec = torch.zeros(80, dtype=torch.uint8)
    with pytest.raises(fa.FusedAdamWError, match="FA_ERR_POINTER"):
        fa.fa_bucket_step_capturable(None, r.p, g, r.m, r.v, r.vmax, host_rec, o, ctl)
    big = torch.zeros(96, dtype=torch.uint8, device=DEV)
    with pytest.raises(fa.FusedAdamWError, match="FA_ERR_ALIGN"):
        fa.fa_bucket_step_capturable(None, r.p, g, r.m, r.v, r.vmax, big[4:84], o, ctl)
    with pytest.raises(fa.FusedAdamWError, match="FA_ERR_ALIAS"):
        fa.fa_bucket_step_capturable(None, r.p, g, r.m, r.v, r.vmax,
                                     r.m.view(torch.uint8)[:80], o, ctl)
    with pytest.raises(fa.FusedAdamWError, match="FA_ERR_ALIAS"):
        fa.fa_bucket_step_capturable(None, r.p, g, r.m, r.v, r.vmax, r.dstep, o, ctl,
                                     report=r.p.view(torch.int32)[:3].view(1, 3))
    torch.cuda.synchronize()
    assert _same(before, r.state())
    assert int(r.dstep.sum()) == 0
