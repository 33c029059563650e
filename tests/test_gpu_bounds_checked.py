"""The bounds-checked build of the library: the CUDA path's own cases, rerun through it.

In place of an external memory checker, the library has a test variant
(-DFA_BOUNDS_CHECK=1) in which every kernel checks the element range it is about to
touch against its array's length and counts, then skips, any access outside it.  The
cases below are the parity tests of the other modules (each against the oracle, with
guard bands where they have them), called with every binding call routed through the
checked build; afterwards the count of out-of-range accesses must be zero.  A checked
build also has to compute exactly what the normal one does.
"""

import contextlib
import dataclasses

import pytest
import torch

import amsgrad_optimizer_step_gb300 as fa
import test_gpu_bucket_update as U
import test_gpu_parity as P
import test_gpu_segments as S
import test_gpu_square_overflow as O
from amsgrad_optimizer_step_gb300 import _lib, build
from synthetic.configs import CONFIG3, CONFIG4

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def checked():
    build.build()
    lib = _lib.open_library(build.build(variant="checked"))
    with _lib.using(lib):
        enabled, _ = fa.fa_bounds_check_report(clear=True)
    assert enabled
    return lib


def test_normal_build_has_no_checks():
    build.build()
    assert fa.fa_bounds_check_report() == (False, 0)


CASES = [
    ("config1 out of place", lambda lib: P.test_config1_out_of_place_full()),
    ("config2 with skip", lambda lib: P.test_config2_bf16_scaled_amsgrad_with_skip_full()),
    ("config3 ragged, in place", lambda lib: P.test_config3_scaled_ragged("inplace")),
    ("config3 ragged out of place", lambda lib: P.test_config3_scaled_ragged("oop")),
    ("decoder bucket", lambda lib: P.test_config4_scaled_decoder_bucket(CONFIG4)),
    ("statistics, clip, +Inf skip, decided on the host and on the device",
     lambda lib: [P.test_config5_scaled_stats_clip_and_inf_skip(api) for api in ("clipped", "gated")]),
    ("edge sizes", lambda lib: [P.test_edge_sizes(gdt, ams, n) for gdt in ("f32", "bf16")
                                for ams in (False, True) for n in (1, 9, 4097, 65537)]),
    ("misaligned views", lambda lib: [P.test_misaligned_views(gdt, off) for gdt in ("f16",)
                                      for off in ((3, 3, 3, 3, 3), (0, 1, 2, 3, 5))]),
    ("analysis rows", lambda lib: [P.test_analyze_rows_match_oracle(
        "bf16", n, rl, segs, lib) for n, rl, segs in (
            (256 * 777 + 5, 256, None), (12_345, 100, None),
            (100_000, 256, [0, 1, 2049, 70_000, 70_000, 100_000]))]),
    ("merge at plan boundaries", lambda lib: [P.test_merge_matches_exact_sum(r)
                                              for r in (1, 1025, 1_048_577)]),
    ("staged comparison", lambda lib: P.test_staged_equals_fused_bitwise("bf16", True)),
    ("model copy", lambda lib: [P.test_writeback_edge_sizes(4097, "bf16"),
                                P.test_writeback_misaligned_model_view(lib)]),
    ("per-segment reports", lambda lib: S.test_chunk_reports_match_oracle_per_segment(
        "bf16", 100, lib)),
    ("per-segment multipliers, mixed sizes",
     lambda lib: S.test_segment_multipliers_mixed_sizes_vs_oracle("f16", False, lib)),
    ("per-segment decision on the device, full grid and pipeline",
     lambda lib: [S.test_per_segment_gated_equals_host_decision_bitwise(*k) for k in (
         ("mixed", "f16", False, 1.0), ("many", "f32", False, 1.0),
         ("offset", "bf16", False, 1.0), ("mixed", "f16", False, 3.0),
         ("small", "f16", True, 2.0 ** -4))]
                 + [S.test_composed_step_with_decided_table_equals_host_decision_bitwise(
                     "many", "bf16")]),
    ("full-grid stretch edges and scalar heads, decided on the host and on the device",
     lambda lib: [P.test_full_grid_stretch_edges_and_scalar_heads(n, off, lib)
                  for n in (1025, 3 * 1024 + 5) for off in (0, 3)]),
    ("gated step at scales with and without an exact inverse",
     lambda lib: [P.test_gated_step_equals_host_decided_step_bitwise_at_any_scale(sc, ams)
                  for sc in (128.0, 3.0) for ams in (False, True)]),
    ("staged comparison vs the oracle, scalar tail",
     lambda lib: P.test_staged_vs_oracle("f16", True, 70_001)),
    ("rows whose squares overflow FP32, rescued",
     lambda lib: [O.test_rows_and_report_with_squares_beyond_fp32(gdt, *layout, lib)
                  for gdt in ("f32", "bf16") for layout in O.LAYOUTS]),
    ("merges in the scaled domain",
     lambda lib: O.test_merge_moves_to_the_scaled_domain(5e37, 3000)),
    ("device-decided steps with an overflowing value, report through the mailbox",
     lambda lib: O.test_gated_steps_equal_host_decided_with_an_overflowing_value()),
    ("the descriptor call in random variants",
     lambda lib: [U.test_bucket_update_random_variant_vs_oracle(k, lib) for k in range(8)]),
]


@pytest.mark.parametrize("name,case", CASES, ids=[c[0] for c in CASES])
def test_case_touches_nothing_out_of_range(checked, oracle_lib, name, case):
    with _lib.using(checked):
        fa.fa_bounds_check_report(clear=True)
        case(oracle_lib)
        torch.cuda.synchronize()
        enabled, violations = fa.fa_bounds_check_report()
    assert enabled and violations == 0, f"{name}: {violations} out-of-range accesses"


def test_checked_build_computes_the_same_bits(checked):
    n = 1_000_003
    w = dataclasses.replace(CONFIG3, calls=4).scaled(n)
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    results = []
    for lib in (None, checked):
        p = torch.empty(n, device=DEV)
        w.fill_params_device(p)
        m, v = torch.zeros_like(p), torch.zeros_like(p)
        t = 0
        ctx = _lib.using(lib) if lib is not None else contextlib.nullcontext()
        with ctx:
            for call in range(1, w.calls + 1):
                w.fill_grad_device(call, g)
                t, _ = fa.fa_adamw_step_inplace(p, g, m, v, None, t, fa.options(**w.options()),
                                                fa.control())
        torch.cuda.synchronize()
        results.append((p, m, v))
    for a, b in zip(*results):
        assert torch.equal(a, b)

