"""The pins are strong enough: each plausible mistake, planted in a copy of the
oracle's source and compiled on the CPU, fails at least one pin."""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "adaln_oracle.cpp")

# (name, original text, planted text) -- each original must occur exactly once.
MUTANTS = [
    ("unbiased_variance", "const double var = ss / (double)D;", "const double var = ss / (double)(D - 1);"),
    ("eps_outside_sqrt", "1.0 / std::sqrt(var + eps)", "1.0 / (std::sqrt(var) + eps)"),
    ("mean_over_d_plus_1", "const double mu = sum / (double)D;", "const double mu = sum / (double)(D + 1);"),
    ("scale_without_one", "const double a = 1.0 + element(scale, dtype, m * D + d);",
     "const double a = element(scale, dtype, m * D + d);"),
    ("shift_scale_swapped", "const double b = element(shift, dtype, m * D + d);",
     "const double b = element(scale, dtype, m * D + d);"),
    ("segment_index_as_modulation_row",
     "const int64_t m = mod_idx[segment_of(cu_seqlens, nseg, r)];\n        const int64_t base = r * D;\n        double sum = 0.0;",
     "const int64_t m = segment_of(cu_seqlens, nseg, r);\n        const int64_t base = r * D;\n        double sum = 0.0;"),
    ("dx_sign", "rho * (g - mean_g - xhat * mean_gx)", "rho * (g - mean_g + xhat * mean_gx)"),
    ("dx_drops_mean_g", "rho * (g - mean_g - xhat * mean_gx)", "rho * (g - xhat * mean_gx)"),
    ("dx_without_rstd", "dx[o * D + d] = rho * (g - mean_g - xhat * mean_gx);",
     "dx[o * D + d] = (g - mean_g - xhat * mean_gx);"),
    ("dscale_uses_g", "dscale[m * D + d] += gy * xhat;", "dscale[m * D + d] += g * xhat;"),
    ("dshift_uses_g", "dshift[m * D + d] += gy;", "dshift[m * D + d] += g;"),
    ("bwd_scale_row_zero",
     "const double g = element(dy, dtype, base + d) * (1.0 + element(scale, dtype, m * D + d));",
     "const double g = element(dy, dtype, base + d) * (1.0 + element(scale, dtype, d));"),
    ("bf16_widen_shift", "<< 16;", "<< 15;"),
    ("round_ties_away", "std::nearbyint(units)", "std::floor(units + 0.5)"),
    ("round_truncates", "std::nearbyint(units)", "std::trunc(units)"),
    ("segment_end_inclusive", "cu[s] <= row && row < cu[s + 1]", "cu[s] <= row && row <= cu[s + 1]"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, planted):
    text = open(SRC).read()
    assert text.count(orig) == 1, "mutation anchor for %s must be unique" % name
    src = tmp_path / ("mutant_%s.cpp" % name)
    src.write_text(text.replace(orig, planted))
    lib = oracle.compile_library(str(src), str(tmp_path / ("mutant_%s.so" % name)))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, "planted mistake %s passed every pin" % name
