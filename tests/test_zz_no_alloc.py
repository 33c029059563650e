"""The allocation-free merge entry point, checked against the caller-scratch merge.

``fa_merge_gradient_stats_static`` is for callers that cannot allocate device
memory themselves -- a plugin whose host framework owns every device
allocation, or a latency-critical path where cudaMalloc/cudaFree (which may
synchronise the device) are not allowed.  It keeps its intermediate records
in one fixed array inside the library instead of a scratch buffer from the
caller.  These tests call it through the C ABI twice in a row, with
different plans, and require the same report as ``fa_merge_gradient_stats``
with caller-owned scratch.

This file is collected last so that a run stopping at the first failure has
run every other test first; it also passes on its own in a fresh process.
"""

import ctypes
import gc

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def fa():
    from amsgrad_optimizer_step_gb300 import build
    build.build()
    import amsgrad_optimizer_step_gb300 as fa_mod
    return fa_mod


def _records(rows, seed):
    rng = np.random.default_rng(seed)
    host = torch.zeros((rows, 3), dtype=torch.int32)
    host[:, 0] = torch.from_numpy((rng.random(rows) * 10).astype(np.float32)).view(torch.int32)
    bad = (rng.random(rows) < 1e-3) * rng.integers(1, 4, rows)
    host[:, 1] = torch.from_numpy(bad.astype(np.int32))
    host[:, 2] = torch.from_numpy((rng.random(rows) * 1e-7).astype(np.float32)).view(torch.int32)
    return host.to(DEV)


def _report(fa, report):
    h = fa.fa_read_report(report)
    return float(h.sum_sq) + float(h.sum_sq_lo), int(h.nonfinite)


def test_static_scratch_merge_matches_caller_scratch_merge(fa):
    lib = fa._lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    # largest plan first (fills the whole fixed scratch), then a smaller one on
    # top of the leftovers
    for rows, seed in ((4_194_304, 1), (1_048_577, 2)):
        recs = _records(rows, seed)
        scratch = fa.scratch_buffer(rows, DEV)
        want = fa.stats_buffer(1, DEV)
        fa.fa_merge_gradient_stats(recs, rows, scratch, want)
        got = fa.stats_buffer(1, DEV)
        gc.collect()  # so that no earlier garbage is freed during the call
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated()
        st = lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                                ctypes.c_void_p(got.data_ptr()),
                                                ctypes.c_void_p(stream))
        assert st == 0, fa._lib.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() <= allocated  # nothing allocated
        s_want, c_want = _report(fa, want)
        s_got, c_got = _report(fa, got)
        assert c_got == c_want
        assert abs(s_got - s_want) <= 1e-12 * s_want


def test_static_scratch_merge_rejects_too_many_rows(fa):
    lib = fa._lib.load()
    recs = fa.stats_buffer(16, DEV)
    report = fa.stats_buffer(1, DEV)
    report.fill_(7)
    for rows in (0, 4_194_305):
        st = lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                                ctypes.c_void_p(report.data_ptr()), None)
        assert st == 8  # FA_ERR_PLAN: rows outside 1..4,194,304, nothing enqueued
    torch.cuda.synchronize()
    assert bool((report == 7).all())
