"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each case patches one place of ``oracle/oracle.c`` in a temporary copy (a
dropped term, a reversed order, a wrong divisor, a wrong rounding rule, a
wrong index or sign), builds it with the same flags, and runs the pins of
``pins.py`` until one fails.  The unpatched oracle passes them all
(``test_oracle_pins``), so each failure here is caused by the planted
mistake.
"""
import pytest

import oracle
import pins

MUTANTS = {
    "dropped_last_rank": ("for (int r = 1; r < P; ++r)\n        acc = acc + load",
                          "for (int r = 1; r < P - 1; ++r)\n        acc = acc + load"),
    "reversed_rank_order": (
        "float acc = load(x[0], i, dtype);\n    for (int r = 1; r < P; ++r)\n"
        "        acc = acc + load(x[r], i, dtype);",
        "float acc = load(x[P - 1], i, dtype);\n    for (int r = P - 2; r >= 0; --r)\n"
        "        acc = acc + load(x[r], i, dtype);"),
    "seeded_with_plus_zero": (
        "float acc = load(x[0], i, dtype);\n    for (int r = 1; r < P; ++r)",
        "float acc = 0.0f;\n    for (int r = 0; r < P; ++r)"),
    "mean_by_reciprocal": ("acc = acc / (float)P;", "acc = acc * (1.0f / (float)P);"),
    "mean_missing": ("if (op == OR_MEAN)\n        acc = acc / (float)P;", "(void)op;"),
    "bf16_ties_away": ("return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);",
                       "return (uint16_t)((u + 0x8000u) >> 16);"),
    "bf16_truncate": ("return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);",
                      "return (uint16_t)(u >> 16);"),
    "bf16_widen_wrong_half": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h;"),
    "rs_strided_shard": ("(size_t)r * shard + j, dtype, op)", "(size_t)j * (size_t)P + r, dtype, op)"),
    "ag_wrong_offset": ("char *dst = (char *)recv[r] + (size_t)s * bytes;",
                        "char *dst = (char *)recv[r] + (size_t)r * bytes;"),
    "bc_from_rank0": ("memcpy(buf[r], buf[root], n * elem_size(dtype));",
                      "memcpy(buf[r], buf[0], n * elem_size(dtype));"),
    "sgd_wrong_sign": ("w[i] = w[i] - step;", "w[i] = w[i] + step;"),
    "sgd_step_uses_g": ("float step = lr * v[i];", "float step = lr * g;"),
    "sgd_no_momentum": ("float mv = momentum * v[i];", "float mv = 0.0f * v[i];"),
    "sgd_ignores_write_back": ("if (!sgd || write_back)", "if (!sgd)"),
    "plan_forward_order": ("for (int t = ntensors - 1; t >= 0; --t)",
                           "for (int t = 0; t < ntensors; ++t)"),
    "plan_closes_at_cap": ("fill + nbytes[t] > cap_bytes", "fill + nbytes[t] >= cap_bytes"),
    "accum_scale_ignored": ("float s = scale * load(g, i, dtype);", "float s = load(g, i, dtype);"),
    "accum_first_ignored": ("a[i] = first ? s : a[i] + s;", "a[i] = a[i] + s;"),
    "accum_final_drops_acc": ("total[r] = first ? s : a[r][i] + s;", "total[r] = s;"),
    "accum_final_scale_ignored": ("float s = scale * load(x[r], i, dtype);",
                                  "float s = load(x[r], i, dtype);"),
    "syncbn_var_no_mean_sq": ("double var = s2 / n - m * m;", "double var = s2 / n;"),
    "syncbn_eps_outside": ("double is = 1.0 / sqrt(var + (double)eps);",
                           "double is = 1.0 / sqrt(var) + (double)eps;"),
    "syncbn_rank0_count": ("n_total += count[r];", "n_total = count[r];"),
    "syncbn_drops_rank": ("s1 = s1 + (double)sum[r][c];", "s1 = s1 + 0.0 * (double)sum[r][c];"),
    "zero1_sgd_wrong_sign": ("w[j] = w[j] - step;", "w[j] = w[j] + step;"),
    "zero1_sgd_no_momentum": ("float mv = momentum * v[j];", "float mv = 0.0f * v[j];"),
    "zero1_strided_owner": ("size_t i = (size_t)r * s + j;", "size_t i = j * (size_t)P + (size_t)r;"),
    "zero1_gathers_gradient": ("store(params[q], i, dtype, w[j]);", "store(params[q], i, dtype, g);"),
    "zero1_skips_own_rank": ("for (int q = 0; q < P; ++q)\n                store(params[q]",
                             "for (int q = 0; q < P; ++q)\n                if (q != r) store(params[q]"),
}


def _cases():
    """(mutant name, occurrence): a target that appears in several functions
    is planted in each of them separately."""
    src = oracle.SRC.read_text()
    out = []
    for name in sorted(MUTANTS):
        n = src.count(MUTANTS[name][0])
        out += [(name, k) for k in range(max(n, 1))]
    return out


@pytest.mark.parametrize("name,occurrence", _cases())
def test_planted_mistake_fails_a_pin(name, occurrence, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.SRC.read_text()
    assert src.count(old) >= 1, f"mutation target of {name} not found"
    at = -1
    for _ in range(occurrence + 1):
        at = src.index(old, at + 1)
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src[:at] + new + src[at + len(old):])
    L = oracle.load(oracle.build(src=mutant, out=tmp_path / "liboracle_mutant.so"))
    for pin in pins.ALL_PINS:
        try:
            pin(L)
        except AssertionError:
            return
    pytest.fail(f"planted mistake {name} (occurrence {occurrence}) passed every pin")
