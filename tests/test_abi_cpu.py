"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
its host-only logic (plan, row count, coefficients, clip decision, validation,
skip/empty) agrees with the pinned oracle and the pages.  No kernel is launched."""

import ctypes
import math
import os
import re

import numpy as np
import pytest

from conftest import ROOT, read_golden

import amsgrad_optimizer_step_gb300 as fa
from amsgrad_optimizer_step_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} missing from the Python binding"


def test_binding_names_match_header():
    assert sorted(_lib.SIGNATURES) == declared_functions()
    for name in declared_functions():
        if name != "fa_status_string":
            assert hasattr(fa, name), name


def test_abi_version_and_defaults(lib):
    assert fa.fa_abi_version() == 2
    d = fa.fa_options_default()
    assert (d.beta1, d.beta2, d.eps, d.weight_decay, d.amsgrad, d.maximize) == \
        (0.9, 0.999, 1e-5, 1e-4, 0, 0)
    for s in range(11):
        assert lib.fa_status_string(s)


def test_stats_plan_matches_oracle_and_pages(oracle_lib):
    gold = read_golden("stats_plan.txt")
    rows_list = [1, 2, 1023, 1024, 1025, 4096, 1048575, 1048576, 1048577, 3_000_000,
                 4_194_303, 4_194_304] + list(np.random.default_rng(5).integers(1, 4_194_305, 200))
    for rows in rows_list:
        k, e = fa.fa_stats_plan(int(rows))
        ok, oe, _ = oracle_lib.stats_plan(int(rows))
        assert (k, e) == (ok, oe)
        assert 4 * e <= gold["max_extra_scratch_bytes"]
        assert k - 1 <= gold["max_extra_merge_kernels"]
    assert fa.fa_stats_plan(4_194_304) == (3, 12_300)
    for bad in (0, -1, gold["max_rows"] + 1):
        with pytest.raises(fa.FusedAdamWError) as e:
            fa.fa_stats_plan(bad)
        assert e.value.status == 8


def test_stats_rows_matches_oracle(oracle_lib):
    from synthetic.configs import CONFIG4
    cases = [(1000, 256, None), (257, 256, None), (1, 7, None), (2000, 128, [0, 5, 5, 700, 1300, 2000]),
             (CONFIG4.n, 256, list(CONFIG4.segments)), (CONFIG4.n, 512, list(CONFIG4.segments))]
    for n, row_len, seg in cases:
        want = None
        if n < 100000:
            want = len(oracle_lib.row_stats(np.zeros(n, np.float32), "f32", row_len, seg)[0])
        else:  # count rows per segment by the same rule, without materialising the gradient
            want = sum(-(-(b - a) // row_len) for a, b in zip(seg[:-1], seg[1:]))
        assert fa.fa_stats_rows(n, row_len, seg) == want
    # the decoder bucket at 256-element rows exceeds the plan; 512 fits
    assert fa.fa_stats_rows(CONFIG4.n, 256, list(CONFIG4.segments)) > 4_194_304
    assert fa.fa_stats_rows(CONFIG4.n, 512, list(CONFIG4.segments)) <= 4_194_304
    with pytest.raises(fa.FusedAdamWError):
        fa.fa_stats_rows(10, 4, [0, 6, 5, 10])


def test_clip_decision_matches_oracle(oracle_lib):
    rng = np.random.default_rng(6)
    for _ in range(200):
        s = float(rng.uniform(0, 10) ** 4)
        cnt = int(rng.integers(0, 3))
        scale = float(2.0 ** rng.integers(0, 10))
        mx = float(rng.choice([0.0, 1.0, 5.0, 100.0]))
        skip, norm, coef = fa.fa_clip_decision(s, cnt, scale, mx)
        o_skip, o_norm, o_coef = oracle_lib.clip_decision(s / scale ** 2, cnt, mx)
        assert skip == o_skip
        assert math.isclose(norm, o_norm, rel_tol=1e-15)
        assert math.isclose(coef, o_coef, rel_tol=1e-15)


def test_stats_sum_sq_decodes_both_record_forms(lib):
    """A plain record is hi + lo; a record whose sum left FP32's range is stored
    negated at 2^-192 (its values scaled by 2^-96 before squaring): -(hi + lo) * 2^192.
    Checked against exact rational arithmetic on the record's two floats."""
    from fractions import Fraction
    rng = np.random.default_rng(9)
    for _ in range(200):
        hi = np.float32(rng.uniform(0, 1e30))
        lo = np.float32(rng.uniform(-1, 1) * float(np.spacing(hi)) / 2)
        for scaled in (False, True):
            rec = fa.FaStats()
            rec.nonfinite = 0
            rec.sum_sq = float(-hi if scaled else hi)
            rec.sum_sq_lo = float(-lo if scaled else lo)
            want = Fraction(float(hi)) + Fraction(float(lo))
            if scaled:
                want *= Fraction(2) ** 192
            assert fa.fa_stats_sum_sq(rec) == float(want)
    # the largest square of an FP32 value, scaled: finite in FP64
    big = np.float32(3.4028235e38)
    rec = fa.FaStats()
    rec.sum_sq = -float(np.float32(float(big) * 2.0 ** -96) ** 2)
    assert math.isclose(fa.fa_stats_sum_sq(rec), float(big) ** 2, rel_tol=1e-7)
    assert lib.fa_stats_sum_sq(None, ctypes.byref(ctypes.c_double())) == 1  # FA_ERR_NULL


def test_step_coefficients_are_fp64_then_fp32():
    o = fa.options(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-5, weight_decay=0.01,
                   maximize=True)
    for t in (1, 2, 7, 1000):
        c = fa.fa_step_coefficients(o, t, gradient_scale=128.0, grad_mult=0.5)
        bc1 = 1 - 0.9 ** t
        bc2 = 1 - 0.999 ** t
        want = [0.9, 1 - 0.9, 0.999, 1 - 0.999, 1e-3 / bc1, 1 / bc2, 1e-5, 1 - 1e-3 * 0.01,
                -0.5 / 128.0]
        for got, w in zip(c, want):
            assert got == float(np.float32(w)) or abs(got - w) <= 2 ** -24 * abs(w)
    # (1 - beta2) formed in FP64 then cast, not fp32(1) - fp32(beta2)
    c = fa.fa_step_coefficients(o, 1)
    assert c[3] == float(np.float32(1 - 0.999))
    assert c[3] != float(np.float32(1) - np.float32(0.999))


def _call_step(lib, n, opts, ctl, t_in=0, p=None, g=None):
    tout = ctypes.c_uint64(12345)
    upd = ctypes.c_int32(7)
    st = lib.fa_adamw_step(n, p, g, 0, None, None, None, t_in, ctypes.byref(opts), ctl,
                           None, None, None, None, ctypes.byref(tout), ctypes.byref(upd), None)
    return st, tout.value, upd.value


def test_skip_and_empty_touch_nothing(lib):
    o = fa.options()
    # empty tensor: OK, t unchanged, nothing launched (NULL pointers accepted)
    assert _call_step(lib, 0, o, fa.control(), t_in=3, p=None) == (0, 3, 0)
    # skip_update: OK, t unchanged, outputs not needed
    assert _call_step(lib, 1000, o, fa.control(skip_update=True), t_in=5) == (0, 5, 0)
    t = ctypes.c_uint64(9)
    upd = ctypes.c_int32(3)
    st = lib.fa_adamw_step_inplace(10, None, None, 0, None, None, None, ctypes.byref(t),
                                   ctypes.byref(o), fa.control(skip_update=True), 1.0,
                                   ctypes.byref(upd), None)
    assert (st, t.value, upd.value) == (0, 9, 0)


@pytest.mark.parametrize("field,value", [("lr", -1.0), ("lr", float("nan")), ("beta1", 1.0),
                                         ("beta2", -0.1), ("eps", -1e-8),
                                         ("weight_decay", float("inf")), ("amsgrad", 2)])
def test_bad_options_rejected_before_anything(lib, field, value):
    o = fa.options()
    setattr(o, field, value)
    st, tout, upd = _call_step(lib, 0, o, fa.control())
    assert st == 4 and tout == 12345 and upd == 7  # outputs untouched


@pytest.mark.parametrize("scale", [0.0, -1.0, float("inf"), float("nan")])
def test_bad_scale_rejected(lib, scale):
    st, tout, upd = _call_step(lib, 0, fa.options(), fa.control(gradient_scale=scale))
    assert st == 4 and tout == 12345 and upd == 7


def test_state_pointers_must_match_t(lib):
    o = fa.options()
    tout = ctypes.c_uint64(0)
    upd = ctypes.c_int32(0)
    fake = ctypes.c_void_p(0x1000)
    # t_in == 0 (no state) but a moment pointer given
    st = lib.fa_adamw_step(4, fake, fake, 0, fake, None, None, 0, ctypes.byref(o), fa.control(),
                           None, None, None, None, ctypes.byref(tout), ctypes.byref(upd), None)
    assert st == 1
    # t_in > 0 but moments missing
    st = lib.fa_adamw_step(4, fake, fake, 0, None, None, None, 3, ctypes.byref(o), fa.control(),
                           None, None, None, None, ctypes.byref(tout), ctypes.byref(upd), None)
    assert st == 1
    # bad dtype
    st = lib.fa_adamw_step(4, fake, fake, 9, None, None, None, 0, ctypes.byref(o), fa.control(),
                           None, None, None, None, ctypes.byref(tout), ctypes.byref(upd), None)
    assert st == 2


def test_segment_table_validation(lib):
    for seg, n in (([0, 5, 3, 10], 10), ([1, 10], 10), ([0, 9], 10)):
        arr = (ctypes.c_int64 * len(seg))(*seg)
        r = ctypes.c_int64()
        assert lib.fa_stats_rows(n, 4, arr, len(seg) - 1, ctypes.byref(r)) == 10


def test_binding_rejects_bad_layouts():
    import torch
    p = torch.zeros(16)
    g = torch.zeros(32)[::2]  # strided view
    with pytest.raises(ValueError):
        fa.fa_adamw_step(p, g, None, None, None, 0, fa.options(), fa.control())
    with pytest.raises(TypeError):
        fa.fa_adamw_step(p, torch.zeros(16, dtype=torch.int32), None, None, None, 0,
                         fa.options(), fa.control())
    with pytest.raises(ValueError):
        fa.fa_adamw_step(p, torch.zeros(15), None, None, None, 0, fa.options(), fa.control())
    with pytest.raises(ValueError):
        fa.fa_adamw_step(p, torch.zeros(1).expand(16), None, None, None, 0, fa.options(),
                         fa.control())


def test_host_memory_is_rejected_not_computed():
    """CPU tensors reach the library and are refused: there is no CPU fallback."""
    import torch
    p = torch.zeros(64)
    g = torch.zeros(64)
    with pytest.raises(fa.FusedAdamWError) as e:
        fa.fa_adamw_step(p, g, None, None, None, 0, fa.options(), fa.control(), stream=0)
    assert e.value.status in (6, 9)  # not device memory / no CUDA device here
    assert not p.any()


def test_byte_model_matches_pages():
    gold = read_golden("byte_model.txt")
    assert fa.bytes_per_param(4, False, False) == gold["fused_adamw_f32grad_steady"]
    assert fa.bytes_per_param(4, True, False) == gold["fused_amsgrad_f32grad_steady"]
    assert fa.bytes_per_param(2, False, False) == 26
    assert fa.bytes_per_param(2, True, False) == 34
    assert fa.bytes_per_param(4, False, True) == 20
    assert fa.bytes_per_param(2, False, True) == 18
    assert fa.bytes_per_param(2, True, True) == 22


def _update_record(**kw):
    """A fa_bucket_update record with placeholder (never dereferenced) device pointers."""
    from amsgrad_optimizer_step_gb300._lib import FaBucketUpdate
    fake = 0x1000
    base = dict(seg_offsets=None, nseg=0, n_total=16, p=fake, g=fake, gdt=0, m=fake, v=fake,
                vmax=None, t=3, grad_mult=1.0, seg_grad_mult=None, report=None,
                seg_reports=None, max_grad_norm=1.0, p_model=None, model_dtype=2,
                seg_decided=None, seg_decided_elements=0)
    base.update(kw)
    return FaBucketUpdate(**base)


def _update(lib, ctl=None, opts=None, **kw):
    """Status and *enqueued of one fa_bucket_update call (no GPU: only host checks run)."""
    u = _update_record(**kw)
    enq = ctypes.c_int32(9)
    st = lib.fa_bucket_update(ctypes.byref(u), ctypes.byref(opts or fa.options()),
                              ctl or fa.control(), ctypes.byref(enq), None)
    return st, enq.value


def test_writeback_validation_without_gpu(lib):
    # model dtype must be FP16 or BF16: rejected before any pointer is looked at
    assert _update(lib, p_model=0x2000, model_dtype=0) == (2, 9)
    # skip: nothing launched or written
    assert _update(lib, p_model=0x2000, ctl=fa.control(skip_update=True)) == (0, 0)
    assert fa.bytes_per_param(2, False, False) + 2 == 28  # write-back adds one 16-bit store


def test_bucket_update_takes_one_multiplier_source(lib):
    """fa_bucket_update: at most one of the per-segment factors, one report and the
    per-segment reports; a host factor other than 1 only on its own; no model copy with
    a per-segment source; a finite, non-negative host factor.  All checked on the host
    before any pointer is looked at."""
    seg = (ctypes.c_int64 * 3)(0, 8, 16)
    mult = (ctypes.c_double * 2)(0.5, 1.0)
    fake = 0x3000
    assert _update(lib, report=fake, seg_reports=fake, seg_offsets=seg, nseg=2)[0] == 4
    assert _update(lib, report=fake, seg_grad_mult=mult, seg_offsets=seg, nseg=2)[0] == 4
    assert _update(lib, report=fake, grad_mult=0.5)[0] == 4
    assert _update(lib, seg_grad_mult=mult, seg_offsets=seg, nseg=2, p_model=fake)[0] == 4
    assert _update(lib, grad_mult=float("nan"))[0] == 4
    assert _update(lib, grad_mult=-1.0)[0] == 4
    bad = (ctypes.c_double * 2)(0.5, float("inf"))
    assert _update(lib, seg_grad_mult=bad, seg_offsets=seg, nseg=2)[0] == 4
    assert _update(lib, seg_grad_mult=mult)[0] == 10  # per segment needs a segment table
    assert _update(lib, t=2 ** 64 - 1)[0] == 4          # the step count would overflow
    assert _update(lib, ctl=fa.control(skip_update=True), report=fake) == (0, 0)


def test_bucket_update_decided_table_rules(lib):
    """seg_decided, the scratch where every segment's decision is taken once: only with
    seg_reports, and holding at least nseg + 1 elements; both checked on the host
    before any pointer is looked at."""
    seg = (ctypes.c_int64 * 3)(0, 8, 16)
    mult = (ctypes.c_double * 2)(0.5, 1.0)
    fake = 0x3000
    assert _update(lib, seg_decided=fake, seg_decided_elements=3)[0] == 4
    assert _update(lib, report=fake, seg_decided=fake, seg_decided_elements=3)[0] == 4
    assert _update(lib, seg_grad_mult=mult, seg_offsets=seg, nseg=2, seg_decided=fake,
                   seg_decided_elements=3)[0] == 4
    assert _update(lib, seg_reports=fake, seg_offsets=seg, nseg=2, seg_decided=fake,
                   seg_decided_elements=2)[0] == 3  # nseg + 1 = 3 needed
    # skip: nothing launched, the table never looked at
    assert _update(lib, seg_reports=fake, seg_offsets=seg, nseg=2, seg_decided=fake,
                   seg_decided_elements=3, ctl=fa.control(skip_update=True)) == (0, 0)


def test_chunk_scratch_plan():
    assert fa.fa_stats_chunk_scratch([0, 1024, 1025, 5000]) == 3 * (1 + 1 + 4)
    assert fa.fa_stats_chunk_scratch([0, 0, 7, 7]) == 3
    assert fa.segment_rows([0, 5, 5, 700, 1300], 256) == [0, 1, 1, 4, 7]
    for bad, code in (([0, 5, 3], 10), ([1, 5], 10), ([0, 0], 8), ([0, 4_194_305], 8)):
        with pytest.raises(fa.FusedAdamWError) as e:
            fa.fa_stats_chunk_scratch(bad)
        assert e.value.status == code


def test_device_decided_calls_validate_on_the_host(lib):
    """The device-decided updates (one report, one per segment, with or without the model
    copy) check options, control, dtype, the segment table and max_grad_norm on the host,
    before any pointer is looked at, and launch nothing for skip_update or an empty
    bucket."""
    o = fa.options()
    seg = (ctypes.c_int64 * 3)(0, 8, 16)
    fake = ctypes.c_void_p(0x1000)
    variants = (dict(report=0x1000), dict(report=0x1000, p_model=0x2000),
                dict(seg_reports=0x1000))

    def one(v, *, ctl=None, nseg=2, table=seg, n=16, dtype=0, max_norm=1.0, opts=o):
        return _update(lib, ctl=ctl, opts=opts, seg_offsets=table, nseg=nseg, n_total=n,
                       gdt=dtype, max_grad_norm=max_norm, **v)[0]

    bad_opts = fa.options(lr=-1.0)
    for v in variants:
        assert one(v, opts=bad_opts) == 4
        assert one(v, ctl=fa.control(gradient_scale=0.0)) == 4
        assert one(v, dtype=7) == 2
        assert one(v, max_norm=float("nan")) == 4
        assert one(v, table=(ctypes.c_int64 * 3)(0, 9, 8), n=8) == 10  # FA_ERR_SEGMENTS
        assert one(v, ctl=fa.control(skip_update=True)) == 0  # nothing launched
        assert one(v, table=(ctypes.c_int64 * 3)(0, 0, 0), n=0) == 0
    assert one(variants[2], nseg=0, table=None) == 10  # a segment table is required

    # the one-call per-segment form: row length and scratch checked first as well
    def clipped(row_len=256, scratch=1 << 20, ctl=None, nseg=2, table=seg):
        return lib.fa_bucket_step_clipped_per_segment_gated(
            table, nseg, 16, fake, fake, 0, fake, fake, None, 0, ctypes.byref(o),
            ctl or fa.control(), 1.0, row_len, fake, 1 << 20, fake, scratch, fake, None, None)
    assert clipped(row_len=0) == 3
    assert clipped(nseg=0, table=None) == 10
    assert clipped(scratch=0) == 3
    assert clipped(ctl=fa.control(skip_update=True)) == 0


def test_library_allocates_nothing():
    """The library never allocates (device memory, pinned or managed host memory) and
    creates no stream or event: none of the CUDA runtime or driver calls that do is
    among the symbols it imports (it links the runtime as a shared library, so every
    runtime call it makes is an undefined dynamic symbol).  Both builds."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm (binutils) not available")
    forbidden = re.compile(r"^(cuda(Malloc\w*|HostAlloc|HostRegister|Free\w*|EventCreate\w*|"
                           r"StreamCreate\w*|MemPool\w*|GraphCreate)|cuMem(Alloc|Create|Map)\w*|"
                           r"cu(Event|Stream)Create\w*)$")
    for variant in ("normal", "checked"):
        path = build.build(variant=variant)
        out = subprocess.run([nm, "-D", "--undefined-only", path], capture_output=True,
                             text=True, check=True).stdout
        names = [line.split()[-1].split("@")[0] for line in out.splitlines() if line.strip()]
        assert any(n.startswith("cudaLaunchKernel") for n in names)  # the runtime is dynamic
        bad = sorted(n for n in names if forbidden.match(n))
        assert not bad, f"{variant} build imports allocating calls: {bad}"


def test_every_entry_point_cites_its_passage():
    """Each declaration in include/*.h is preceded by a comment that cites the page
    passage defining the operation, or says that the pages have no counterpart."""
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        prev = 0
        for m in re.finditer(r"^\w[\w \*]*?\b(fa_[a-z0-9_]+)\s*\(", text, flags=re.M):
            comments = re.findall(r"/\*.*?\*/", text[prev:m.start()], flags=re.S)
            last = comments[-1] if comments else ""
            assert re.search(r"\[(FA-ja|FA-zh|TR-zh)\]|no counterpart", last), m.group(1)
            prev = m.start()


def test_a_missing_library_fails_loudly(tmp_path):
    """Without the built library nothing runs: loading raises and names the build step
    (there is no CPU or library fallback to fall through to)."""
    with pytest.raises(RuntimeError, match="is not built"):
        _lib.open_library(str(tmp_path / "libfused_adamw.so"))
