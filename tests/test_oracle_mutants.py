"""Each plausible mistake planted in a copy of the oracle must be caught by a pin.

The mistakes are planted on the CPU, in a temporary copy of the oracle's C
sources; the committed oracle is never modified.  A mutant "survives" when
every pin in ``tests/pins.py`` still passes on it, which would mean the pins
cannot tell that mistake from the method.
"""

import inspect
import os
import shutil

import pytest

import oracle
import pins
from conftest import read_golden

MUTANTS = {
    "drop_bc1": ("adamw_oracle.c", "(m_new / bc1)", "(m_new)"),
    "drop_bc2": ("adamw_oracle.c", "sqrt(v_used / bc2)", "sqrt(v_used)"),
    "eps_inside_sqrt": ("adamw_oracle.c", "(sqrt(v_used / bc2) + o->eps)",
                        "sqrt(v_used / bc2 + o->eps)"),
    "beta1_in_v": ("adamw_oracle.c", "(1.0 - o->beta2) * grad * grad",
                   "(1.0 - o->beta1) * grad * grad"),
    "beta2_in_m": ("adamw_oracle.c", "o->beta1 * m_old + (1.0 - o->beta1)",
                   "o->beta2 * m_old + (1.0 - o->beta1)"),
    "g_not_squared": ("adamw_oracle.c", "(1.0 - o->beta2) * grad * grad",
                      "(1.0 - o->beta2) * grad"),
    "no_maximize": ("adamw_oracle.c", "grad = -grad;", "grad = grad;"),
    "no_decay": ("adamw_oracle.c", "p[i] * (1.0 - o->lr * o->weight_decay)", "p[i]"),
    "decay_not_scaled_by_lr": ("adamw_oracle.c", "(1.0 - o->lr * o->weight_decay)",
                               "(1.0 - o->weight_decay)"),
    "no_amsgrad_max": ("adamw_oracle.c", "max_propagate_nan(vmax_old, v_new)", "v_new"),
    "amsgrad_min": ("adamw_oracle.c", "return a > b ? a : b;", "return a < b ? a : b;"),
    "amsgrad_max_drops_nan": ("adamw_oracle.c", "if (isnan(a) || isnan(b))\n        return NAN;",
                              "if (isnan(a) || isnan(b))\n        return isnan(a) ? b : a;"),
    "vmax_ignored_in_update": ("adamw_oracle.c", "v_used = vmax_new;", "v_used = v_new;"),
    "store_corrected_max": ("adamw_oracle.c", "vmax[i] = store(vmax_new,",
                            "vmax[i] = store(vmax_new / bc2,"),
    "scale_multiplies": ("adamw_oracle.c", "oracle_widen(g, gdtype, i) / gradient_scale",
                         "oracle_widen(g, gdtype, i) * gradient_scale"),
    "clip_ignored": ("adamw_oracle.c", "grad = grad * clip_coef;", "grad = grad;"),
    "power_off_by_one": ("adamw_oracle.c", "k < t; ++k", "k <= t; ++k"),
    "step_uses_m_old": ("adamw_oracle.c", "o->lr * (m_new / bc1)", "o->lr * (m_old / bc1)"),
    "f16_exponent_bias": ("adamw_oracle.c", "expo - 25", "expo - 24"),
    "f16_subnormal_scale": ("adamw_oracle.c", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    "bf16_shift": ("adamw_oracle.c", "(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "model_copy_truncates": ("adamw_oracle.c", "double y = rint(x / q) * q;",
                             "double y = trunc(x / q) * q;"),
    "model_copy_ties_away": ("adamw_oracle.c", "double y = rint(x / q) * q;",
                             "double y = round(x / q) * q;"),
    "bf16_seven_bits": ("adamw_oracle.c", "round_to_format((double)x, 8, -126, 127)",
                        "round_to_format((double)x, 7, -126, 127)"),
    "f16_no_subnormal_floor": ("adamw_oracle.c", "int qexp = (e < emin ? emin : e) - (sig_bits - 1);",
                               "int qexp = e - (sig_bits - 1);"),
    "f16_no_overflow": ("adamw_oracle.c", "round_to_format((double)x, 11, -14, 15)",
                        "round_to_format((double)x, 11, -14, 16)"),
    "stats_sum_not_squared": ("stats_oracle.c", "s += u * u;", "s += u;"),
    "stats_scale_ignored": ("stats_oracle.c", "double u = x / gradient_scale;", "double u = x;"),
    "stats_count_dropped": ("stats_oracle.c", "++c;\n            continue;\n        }\n        double u",
                            "continue;\n        }\n        double u"),
    "rows_span_segments": ("stats_oracle.c",
                           "start + row_len < seg[k + 1] ? start + row_len : seg[k + 1]",
                           "start + row_len"),
    "rows_count_inf_only": ("stats_oracle.c", "return isnan(x) || isinf(x);", "return isinf(x);"),
    "plan_floor_division": ("stats_oracle.c", "(count + fan_in - 1) / fan_in", "count / fan_in + (count > 1 && count < fan_in)"),
    "plan_counts_report": ("stats_oracle.c", "if (count > 1)\n            scratch_records += count;",
                           "scratch_records += count;"),
    "clip_inverted": ("stats_oracle.c", "*coef = max_grad_norm / *norm;", "*coef = *norm / max_grad_norm;"),
    "clip_without_threshold": ("stats_oracle.c", "&& *norm > max_grad_norm", ""),
}


def _run_pins(lib):
    failures = []
    for pin in pins.ALL_PINS:
        try:
            if "golden" in inspect.signature(pin).parameters:
                pin(lib, read_golden("stats_plan.txt"))
            else:
                pin(lib)
        except Exception as e:  # any failure counts as "caught"
            failures.append(f"{pin.__name__}: {type(e).__name__}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    fname, old, new = MUTANTS[name]
    for f in oracle.SOURCES + ("oracle.h",):
        shutil.copy(os.path.join(oracle.HERE, f), tmp_path / f)
    src = (tmp_path / fname).read_text()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    (tmp_path / fname).write_text(src.replace(old, new))
    lib = oracle.OracleLib(oracle.build(src_dir=str(tmp_path), force=True))
    assert _run_pins(lib), f"mutant {name} survived every pin"
