"""The allocation-free merge entry point, checked against exact host sums and the
caller-scratch merge.

``fa_merge_gradient_stats_static`` is for callers that cannot allocate device
memory themselves -- a plugin whose host framework owns every device
allocation, or a latency-critical path where cudaMalloc/cudaFree (which may
synchronise the device) are not allowed.  It keeps its intermediate records
in one fixed array inside the library instead of a scratch buffer from the
caller.  These tests call it through the C ABI, several times in a row with
plans of different sizes (smaller after larger and larger after smaller, so
that whatever the previous call left in the shared array is overwritten in
both directions), and require:

* the non-finite count equal to the exact integer sum of the records' counts,
  and the sum within 1e-12 of ``math.fsum`` over every record's (sum_sq,
  sum_sq_lo) pair;
* the same 12 bytes as ``fa_merge_gradient_stats`` with caller-owned scratch
  (the same kernels in the same order);
* no change in the device's free memory (``cudaMemGetInfo``) across a call, once
  a first call has looked up the array's address.

This file is collected last so that a run stopping at the first failure has
run every other test first; it also passes on its own in a fresh process.
"""

import ctypes
import gc
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    from amsgrad_optimizer_step_gb300 import build
    build.build()
    import amsgrad_optimizer_step_gb300 as fa_mod
    return fa_mod


def _records(rows, seed):
    """Row records on the host: sums in [0, 10), residuals in [0, 1e-7), about one
    row in a thousand with 1 to 3 non-finite values."""
    rng = np.random.default_rng(seed)
    hi = (rng.random(rows) * 10).astype(np.float32)
    lo = (rng.random(rows) * 1e-7).astype(np.float32)
    cnt = ((rng.random(rows) < 1e-3) * rng.integers(1, 4, rows)).astype(np.uint32)
    host = np.zeros((rows, 3), dtype=np.uint32)
    host[:, 0] = hi.view(np.uint32)
    host[:, 1] = cnt
    host[:, 2] = lo.view(np.uint32)
    return host, math.fsum(np.concatenate([hi, lo]).astype(np.float64).tolist()), int(cnt.sum())


def _to_device(host):
    return torch.from_numpy(host.view(np.int32)).to(DEV)


def _call_static(fa, recs, rows, report, stream):
    lib = fa._lib.load()
    return lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                              ctypes.c_void_p(report.data_ptr()),
                                              ctypes.c_void_p(stream))


def _report(fa, report):
    h = fa.fa_read_report(report)
    return float(h.sum_sq) + float(h.sum_sq_lo), int(h.nonfinite)


def test_static_scratch_merge_exact_sums_and_caller_scratch_bits(fa):
    stream = torch.cuda.current_stream().cuda_stream
    # a first call: looks up the array's address (and may load the module)
    host, want_sum, want_cnt = _records(3000, 0)
    recs = _to_device(host)
    report = fa.stats_buffer(1, DEV)
    assert _call_static(fa, recs, 3000, report, stream) == 0
    torch.cuda.synchronize()
    s, c = _report(fa, report)
    assert c == want_cnt and abs(s - want_sum) <= 1e-12 * want_sum
    # plans of 1, 2 and 3 merge kernels, small after large and large after small
    for rows, seed in ((1_000, 1), (1_048_577, 2), (4_194_304, 3), (5_000, 4), (1_048_576, 5),
                       (4_194_304, 6)):
        host, want_sum, want_cnt = _records(rows, seed)
        recs = _to_device(host)
        scratch = fa.scratch_buffer(rows, DEV)
        want = fa.stats_buffer(1, DEV)
        fa.fa_merge_gradient_stats(recs, rows, scratch, want)
        got = fa.stats_buffer(1, DEV)
        got.fill_(-1)
        gc.collect()  # so that no earlier garbage is freed during the call
        torch.cuda.synchronize()
        free_before, _ = torch.cuda.mem_get_info(DEV)
        assert _call_static(fa, recs, rows, got, stream) == 0
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info(DEV)
        assert free_after == free_before, f"{rows} rows: device memory allocated by the call"
        s, c = _report(fa, got)
        assert c == want_cnt, (rows, c, want_cnt)
        assert abs(s - want_sum) <= 1e-12 * want_sum, (rows, s, want_sum)
        assert torch.equal(got, want), f"{rows} rows: differs from the caller-scratch merge"


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


_FRESH_CAPTURE = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import amsgrad_optimizer_step_gb300 as fa
dev = torch.device("cuda", 0)
lib = fa._lib.load()
rows = 5000
recs = torch.from_numpy(np.ones((rows, 3), dtype=np.float32).view(np.int32)).to(dev)
recs[:, 1] = 0
recs[:, 2] = 0
report = fa.stats_buffer(1, dev)
report.fill_(7)
s = torch.cuda.Stream(dev)
torch.cuda.synchronize()
graph = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    graph.capture_begin()
    st_capture = lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                                    ctypes.c_void_p(report.data_ptr()),
                                                    ctypes.c_void_p(s.cuda_stream))
    graph.capture_end()
torch.cuda.synchronize()
untouched = bool((report == 7).all())
# outside a capture the first call looks the address up; then a capture may use it
st_plain = lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                              ctypes.c_void_p(report.data_ptr()),
                                              ctypes.c_void_p(s.cuda_stream))
s.synchronize()
plain = fa.fa_read_report(report).sum_sq
report.fill_(7)
graph2 = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    graph2.capture_begin()
    st_capture2 = lib.fa_merge_gradient_stats_static(ctypes.c_void_p(recs.data_ptr()), rows,
                                                     ctypes.c_void_p(report.data_ptr()),
                                                     ctypes.c_void_p(s.cuda_stream))
    graph2.capture_end()
graph2.replay()
torch.cuda.synchronize()
print(st_capture, int(untouched), st_plain, plain, st_capture2, fa.fa_read_report(report).sum_sq)
"""


def test_static_scratch_merge_first_call_inside_a_capture_is_refused(fa):
    """In a fresh process (no earlier call has looked up the array's address), a
    first call on a stream being captured returns FA_ERR_CUDA, enqueues nothing and
    leaves the capture usable; after one call outside a capture, a captured call
    replays to the right report."""
    out = subprocess.run([sys.executable, "-c", _FRESH_CAPTURE, ROOT], capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    st_capture, untouched, st_plain, plain, st_capture2, replayed = out.stdout.split()[-6:]
    assert int(st_capture) == 9 and int(untouched) == 1
    assert int(st_plain) == 0 and float(plain) == 5000.0
    assert int(st_capture2) == 0 and float(replayed) == 5000.0
