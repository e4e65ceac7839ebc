"""The pins are sharp enough: each plausible mistake, planted in a copy of the
oracle's C source and compiled on the CPU, must fail at least one pin.

The mutations are textual edits of a temporary copy; the oracle itself is
never modified.  CPU only (gcc).
"""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("entropy_sign", "if (p > 0.0) H -= p * log(p);",
     "if (p > 0.0) H += p * log(p);"),
    ("entropy_log2", "if (p > 0.0) H -= p * log(p);",
     "if (p > 0.0) H -= p * log2(p);"),
    ("sum_skips_first_term",
     "    double S = 0.0;\n    for (int64_t i = 0; i < C; ++i) {\n"
     "        S += exp(((double)l[i] - m) / T);\n    }\n    double H = 0.0;",
     "    double S = 0.0;\n    for (int64_t i = 1; i < C; ++i) {\n"
     "        S += exp(((double)l[i] - m) / T);\n    }\n    double H = 0.0;"),
    ("max_is_min", "if ((double)l[i] > m) m = (double)l[i];",
     "if ((double)l[i] < m) m = (double)l[i];"),
    ("softmax_ignores_T", "p[i] = exp(((double)l[i] - m) / T) / S;",
     "p[i] = exp(((double)l[i] - m)) / S;"),
    ("softmax_times_T", "p[i] = exp(((double)l[i] - m) / T) / S;",
     "p[i] = exp(((double)l[i] - m) * T) / S;"),
    ("branch_swapped", "if (Hmid > bound) {", "if (Hmid < bound) {"),
    ("search_up_to_t_max", "double hi = t_max < 1.0 ? t_max : 1.0;",
     "double hi = t_max;"),
    ("output_at_hi", "softmax_at(l, C, lo, p);\n    *T_out = lo;",
     "softmax_at(l, C, hi, p);\n    *T_out = hi;"),
    ("one_step_short", "for (int32_t k = 0; k < max_iter; ++k) {",
     "for (int32_t k = 1; k < max_iter; ++k) {"),
    ("midpoint_wrong", "double mid = (lo + hi) / 2.0;",
     "double mid = lo + hi / 2.0;"),
    ("first_check_at_t_min", "if (entropy_at(l, C, 1.0) <= bound) {",
     "if (entropy_at(l, C, t_min) <= bound) {"),
    ("overflow_flag_at_hi",
     "if (entropy_at(l, C, lo) > bound) return ORACLE_FLAG_ENTROPY_OVERFLOW;",
     "if (entropy_at(l, C, hi) > bound) return ORACLE_FLAG_ENTROPY_OVERFLOW;"),
    ("nan_inf_flags_swapped",
     "return has_nan ? ORACLE_FLAG_NAN_INPUT : ORACLE_FLAG_INF_INPUT;",
     "return has_nan ? ORACLE_FLAG_INF_INPUT : ORACLE_FLAG_NAN_INPUT;"),
    ("inf_not_detected", "else if (isinf(l[i])) has_inf = 1;",
     "else if (0) has_inf = 1;"),
    ("bound_strict", "if (entropy_at(l, C, 1.0) <= bound) {",
     "if (entropy_at(l, C, 1.0) < bound - 1e-3) {"),
    ("backward_without_inv_T", "out[k] = pb[k] * (gb[k] - dot) / T[b];",
     "out[k] = pb[k] * (gb[k] - dot);"),
    ("backward_times_T", "out[k] = pb[k] * (gb[k] - dot) / T[b];",
     "out[k] = pb[k] * (gb[k] - dot) * T[b];"),
    ("backward_dot_sign", "out[k] = pb[k] * (gb[k] - dot) / T[b];",
     "out[k] = pb[k] * (gb[k] + dot) / T[b];"),
    ("backward_no_p_factor", "out[k] = pb[k] * (gb[k] - dot) / T[b];",
     "out[k] = (gb[k] - dot) / T[b];"),
    ("backward_dot_skips_first",
     "for (int64_t i = 0; i < C; ++i) dot += gb[i] * pb[i];",
     "for (int64_t i = 1; i < C; ++i) dot += gb[i] * pb[i];"),
    ("backward_dot_of_p_with_itself", "dot += gb[i] * pb[i];",
     "dot += pb[i] * pb[i];"),
    ("backward_nan_rows_not_zeroed",
     "if (!(T[b] > 0.0) || isinf(T[b])) {", "if (0) {"),
    ("attention_causal_off_by_one",
     "const int64_t kept_end = causal ? i + 1 : S;",
     "const int64_t kept_end = causal ? i : S;"),
    ("attention_causal_keeps_diagonal_out",
     "const int64_t kept_end = causal ? i + 1 : S;",
     "const int64_t kept_end = causal ? i + 2 : S;"),
    ("attention_mask_of_batch_0", "const float* m = mask ? mask + b * S : 0;",
     "const float* m = mask ? mask : 0;"),
    ("attention_mask_ignored", "const float v = s[j] + m[j];",
     "const float v = s[j];"),
    ("attention_mask_added_in_fp64", "const float v = s[j] + m[j];",
     "const double v = (double)s[j] + (double)m[j];"),
    ("attention_no_max_subtraction",
     "p[j] = exp(masked_score(s, m, j) - vmax);",
     "p[j] = exp(masked_score(s, m, j));"),
    ("attention_mask_inf_not_error",
     "else if (isinf(m[j]) && m[j] > 0) has_inf = 1;",
     "else if (0) has_inf = 1;"),
    ("attention_row_index_is_head", "const int64_t i = r % S;",
     "const int64_t i = (r / S) % S;"),
    ("biencoder_scale_missing",
     "scores[(bh * Q + i) * K + j] = s * scale;",
     "scores[(bh * Q + i) * K + j] = s;"),
    ("biencoder_keys_transposed",
     "const float* kj = k + (bh * K + j) * D;",
     "const float* kj = k + (bh * K) * D + j;"),
    ("biencoder_dot_skips_last",
     "for (int64_t d = 0; d < D; ++d) s = fmaf(qi[d], kj[d], s);",
     "for (int64_t d = 0; d + 1 < D; ++d) s = fmaf(qi[d], kj[d], s);"),
    ("biencoder_dot_in_double",
     "for (int64_t d = 0; d < D; ++d) s = fmaf(qi[d], kj[d], s);",
     "double t = 0.0; for (int64_t d = 0; d < D; ++d) t += (double)qi[d] * kj[d]; s = (float)t;"),
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_fails_a_pin(name, old, new, mutant_dir):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(mutant_dir, f"{name}.c")
    so_path = os.path.join(mutant_dir, f"lib{name}.so")
    with open(c_path, "w") as f:
        f.write(mutated)
    subprocess.run(oracle.build_command(c_path, so_path), check=True)
    lib = oracle.load(so_path)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
