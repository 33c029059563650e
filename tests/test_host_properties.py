"""Randomised properties of the library's host logic, against the oracle (no GPU).

The row count and reduction plan for arbitrary segment tables and sizes, the skip /
clip decision over the whole input range, and the shard split used by several ranks.
"""

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import amsgrad_optimizer_step_gb300 as fa  # noqa: E402
from amsgrad_optimizer_step_gb300 import sharded  # noqa: E402

MAX_ROWS = 4_194_304
SETTINGS = settings(max_examples=150, deadline=None)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from amsgrad_optimizer_step_gb300 import build
    build.build()


@SETTINGS
@given(sizes=st.lists(st.integers(0, 4000), min_size=1, max_size=40),
       row_len=st.integers(1, 700))
def test_rows_and_plan_match_the_oracle(sizes, row_len, oracle_lib):
    seg = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    n = int(seg[-1])
    rows = fa.fa_stats_rows(n, row_len, [int(x) for x in seg])
    want_rows = oracle_lib.row_stats(np.zeros(n, np.float32), "f32", row_len, seg)[0].shape[0] \
        if n else 0
    assert rows == want_rows
    if rows >= 1:
        assert fa.fa_stats_plan(rows) == oracle_lib.stats_plan(rows)[:2]


@SETTINGS
@given(rows=st.one_of(st.integers(-5, 5000), st.integers(1_000_000, MAX_ROWS + 5)))
def test_plan_matches_the_oracle_or_both_reject(rows, oracle_lib):
    want = oracle_lib.stats_plan(rows)
    if want is None:
        with pytest.raises(fa.FusedAdamWError, match="FA_ERR_PLAN"):
            fa.fa_stats_plan(rows)
    else:
        assert fa.fa_stats_plan(rows) == want[:2]


@SETTINGS
# (normal-range sums: the oracle is handed sum / scale^2, which a subnormal sum underflows)
@given(sum_sq=st.one_of(st.just(0.0), st.floats(1e-250, 1e30)),
       count=st.integers(0, 3),
       scale=st.sampled_from([1.0, 2.0, 128.0, 65536.0, 0.5, 3.0]),
       max_norm=st.one_of(st.just(0.0), st.floats(1e-6, 1e6)))
def test_clip_decision_matches_the_oracle(sum_sq, count, scale, max_norm, oracle_lib):
    skip, norm, coef = fa.fa_clip_decision(sum_sq, count, scale, max_norm)
    o_skip, o_norm, o_coef = oracle_lib.clip_decision(sum_sq / (scale * scale), count, max_norm)
    assert skip == o_skip == (count > 0)
    assert norm == pytest.approx(o_norm, rel=1e-14, abs=1e-300)
    if not skip:
        assert coef == pytest.approx(o_coef, rel=1e-14)
        assert 0.0 < coef <= 1.0


@SETTINGS
@given(n=st.integers(0, 10 ** 10), world=st.integers(1, 64))
def test_shards_are_contiguous_aligned_and_balanced(n, world):
    bounds = [sharded.shard_range(n, r, world) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == n
    for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
        assert a1 == b0
    for lo, hi in bounds:
        assert lo <= hi and lo % 8 == 0 and (hi % 8 == 0 or hi == n)
    lens = [hi - lo for lo, hi in bounds]
    # shards hold floor or ceil of ceil(n/8)/world 8-element units; the last may be short
    assert max(lens) - min(lens) <= 16


@SETTINGS
@given(n=st.integers(0, 10 ** 10), world=st.integers(1, 64))
def test_zero1_shards_cover_the_bucket_aligned_and_minimal(n, world):
    """The ZeRO-1 shard length: world equal shards of S elements cover the n-element
    bucket, S is a multiple of 8 (every shard starts 16-byte aligned in an aligned FP32
    buffer), and S is the smallest such length, so the padding is under 8 * world."""
    s = sharded.zero1_shard_len(n, world)
    assert s % 8 == 0 and s * world >= n
    assert s == 0 or (s - 8) * world < n
    assert s * world - n < 8 * world or n == 0


@SETTINGS
@given(data=st.lists(st.tuples(st.booleans(), st.integers(0, 3), st.integers(0, 40)),
                     min_size=1, max_size=30))
def test_active_runs_cover_exactly_the_active_parameters(data):
    from amsgrad_optimizer_step_gb300.optim import active_runs
    active = [a for a, _, _ in data]
    steps = [s for _, s, _ in data]
    offsets, pos = [], 0
    for _, _, size in data:
        offsets.append(pos)
        pos += (size + 7) // 8 * 8
    runs = active_runs(active, steps, offsets, pos)
    covered = [i for i, j, _, _ in runs for i in range(i, j)]
    assert covered == [i for i, a in enumerate(active) if a]
    for i, j, lo, hi in runs:
        assert len({steps[k] for k in range(i, j)}) == 1
        assert lo == offsets[i] and hi == (offsets[j] if j < len(data) else pos)
        # maximal: the next parameter is inactive or has another step count
        assert j == len(data) or not active[j] or steps[j] != steps[i]
    if all(active) and len(set(steps)) == 1:
        assert runs == [(0, len(data), 0, pos)]


def _int_pow(beta, t):
    """beta^t by repeated squaring in FP64 (the host's integer power)."""
    r, b = 1.0, beta
    while t:
        if t & 1:
            r *= b
        b *= b
        t >>= 1
    return r


@SETTINGS
@given(lr=st.floats(0.0, 1.0), beta1=st.floats(0.0, 0.999999), beta2=st.floats(0.0, 0.999999),
       eps=st.floats(0.0, 1e-2), wd=st.floats(0.0, 1.0), t=st.integers(1, 10 ** 12),
       log2_scale=st.integers(-8, 16), mult=st.floats(0.0, 1.0), maximize=st.booleans())
def test_step_coefficients_are_the_fp64_formula_cast_once(lr, beta1, beta2, eps, wd, t,
                                                          log2_scale, mult, maximize):
    """Every coefficient is the FP64 expression rounded once to FP32: exactly for the
    ones without a power, and for the bias corrections to the FP32 rounding of the same
    repeated-squaring power."""
    scale = 2.0 ** log2_scale
    o = fa.options(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=wd,
                   maximize=maximize)
    c = fa.fa_step_coefficients(o, t, gradient_scale=scale, grad_mult=mult)
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    assert c[0] == f32(beta1) and c[1] == f32(1.0 - beta1)
    assert c[2] == f32(beta2) and c[3] == f32(1.0 - beta2)
    assert c[4] == f32(lr / (1.0 - _int_pow(beta1, t)))
    assert c[5] == f32(1.0 / (1.0 - _int_pow(beta2, t)))
    assert c[6] == f32(eps) and c[7] == f32(1.0 - lr * wd)
    assert c[8] == f32((-1.0 if maximize else 1.0) * mult / scale)


@SETTINGS
@given(sizes=st.lists(st.integers(0, 200_000), min_size=1, max_size=60),
       row_len=st.integers(1, 4096))
def test_segment_rows_and_chunk_scratch(sizes, row_len):
    """Per-segment rows (rows never span segments) and the per-segment merge scratch:
    three FP32 words per group of at most 1024 rows inside each segment."""
    seg = [0]
    for s in sizes:
        seg.append(seg[-1] + s)
    crow = fa.segment_rows(seg, row_len)
    assert crow == [0] + list(np.cumsum([-(-s // row_len) for s in sizes]))
    if crow[-1] == 0 or crow[-1] > MAX_ROWS:
        with pytest.raises(fa.FusedAdamWError):
            fa.fa_stats_chunk_scratch(crow)
        return
    groups = sum(-(-(b - a) // 1024) for a, b in zip(crow[:-1], crow[1:]))
    assert fa.fa_stats_chunk_scratch(crow) == 3 * groups
    assert fa.fa_stats_rows(seg[-1], row_len, seg) == crow[-1]
