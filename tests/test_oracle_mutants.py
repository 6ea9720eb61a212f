"""Plant plausible mistakes in copies of the oracle and check that the pin
battery rejects every one of them (CPU only; the real oracle is untouched).

Each mutant is a textual edit of oracle.c compiled into a temporary
library. A mutant that survives every pin would mean the pins cannot tell
that mistake from the definition.
"""
import pytest

import _pins
import oracle

MUTANTS = {
    "tie_goes_to_last": ("return v > m;", "return v >= m;"),
    "nan_never_wins": ("return !isnan(m);", "return 0;"),
    "adaptive_end_floor": ("*end = ((i + 1) * I + O - 1) / O;", "*end = ((i + 1) * I) / O;"),
    "adaptive_start_ceil": ("*start = (i * I) / O;", "*start = (i * I + O - 1) / O;"),
    "fixed_size_off_by_one": ("return (I - K) / S + 1;", "return (I - K) / S;"),
    "fixed_window_short": ("*end = o * S + K;", "*end = o * S + K - 1;"),
    "offset_axes_swapped": ("int64_t off = (d * H + h) * W + w;",
                            "int64_t off = (d * W + h) * H + w;"),
    "scan_h_before_d": ("for (d = ds; d < de; d++)\n        for (h = hs; h < he; h++)",
                        "for (h = hs; h < he; h++)\n        for (d = ds; d < de; d++)"),
    "y_from_wrong_element": ("(p * vol + best) * es", "(p * vol + best - (best > 0)) * es"),
    "bwd_drops_earlier_terms": ("acc[target] = acc[target] + gv;", "acc[target] = gv;"),
    "bwd_subtracts": ("acc[target] = acc[target] + gv;", "acc[target] = acc[target] - gv;"),
    "bwd_rounds_every_add": (
        "acc[target] = acc[target] + gv;   /* binary32 add */",
        "{ store_rounded(dtype, gin, p * in_vol, acc[target] + gv);"
        " acc[target] = load_f32(dtype, gin, p * in_vol); }"),
    "bwd_empty_is_negative_zero": ("seen[j] ? acc[j] : 0.0f", "seen[j] ? acc[j] : -0.0f"),
    "bwd_sum_starts_at_positive_zero": ("acc[target] = gv;", "acc[target] = 0.0f + gv;"),
    "round_ties_away": ("r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "r = fl + 1.0;"),
    "f16_subnormal_scale": ("(float)frac * 0x1p-24f", "(float)frac * 0x1p-25f"),
    "f16_exponent_bias": ("((e - 15 + 127) << 23)", "((e - 14 + 127) << 23)"),
    "bf16_subnormal_limit": ("r = round_to_format(fabs((double)f), 7, -126);",
                             "r = round_to_format(fabs((double)f), 7, -125);"),
    # padding, dilation and ceil mode
    "ex_no_ceil_drop": ("if (ceil_mode && (O - 1) * S >= I + p)", "if (0)"),
    "ex_truncating_division": ("O = (num >= 0 ? num / S : -((-num + S - 1) / S)) + 1;",
                               "O = num / S + 1;"),
    "ex_padding_limit_loose": ("if (2 * p > K)", "if (2 * p > K + 1)"),
    "ex_padding_added": ("int64_t d = od * sd - pd + a * dd;", "int64_t d = od * sd + pd + a * dd;"),
    "ex_dilation_ignored_w": ("int64_t w = ow * sw - pw + c * dw;", "int64_t w = ow * sw - pw + c;"),
    "ex_y_from_wrong_element": ("es * (p * vol + best)", "es * (p * vol + best - (best > 0))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mutant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for check in _pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failures.append(check.__name__)
        except (RuntimeError, ValueError, IndexError):
            failures.append(check.__name__ + " (raised)")
    assert failures, f"mutant {name} survived every pin"
