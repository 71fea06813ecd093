"""Plant plausible mistakes in copies of the C oracle and check that the pins
catch every one of them.

Each mutant is a text edit of oracle/diffattn_oracle.c, compiled into a
temporary library and loaded as a separate instance of the oracle package;
the pin tests of test_oracle_pins.py then run against it, and at least one
must fail.  Only the oracle is mutated, on the CPU.
"""
import importlib.util
import os

import pytest

import test_oracle_bwd_pins as bwd_pins
import test_oracle_paired_pins as paired_pins
import test_oracle_pins as pins
import test_oracle_prologue_pins as pro_pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")

MUTANTS = {
    "scale 1/sqrt(2d) in V1": ("const double scale = 1.0 / sqrt((double)d);",
                               "const double scale = 1.0 / sqrt((double)(2 * d));"),
    "lam_init of layer+1": ("return 0.8 - 0.6 * exp(-0.3 * (double)layer_index);",
                            "return 0.8 - 0.6 * exp(-0.3 * (double)(layer_index + 1));"),
    "lambda terms swapped": ("return exp(s1) - exp(s2) + lam_init;", "return exp(s2) - exp(s1) + lam_init;"),
    "(1 - lam_init) dropped": ("y[c] *= (1.0 - J->lam_init);", "y[c] *= 1.0;"),
    "eps outside the root": ("const double r = 1.0 / sqrt(ms + eps);", "const double r = 1.0 / (sqrt(ms) + eps);"),
    "V1 combine sign": ("x[c] = a1[c] - J->lam_full * a2[c];", "x[c] = a1[c] + J->lam_full * a2[c];"),
    "causal mask admits one future key": (
        "attend_row(q1, k1, qk_row, v, v_row, (int64_t)t + 1, d, dv, scale, scores, a1);",
        "attend_row(q1, k1, qk_row, v, v_row, (int64_t)(t + 1 < T ? t + 2 : t + 1), d, dv, scale, scores, a1);"),
    "V1 branch 2 reads k1": ("attend_row(q2, k2, qk_row,", "attend_row(q2, k1, qk_row,"),
    "RMS mean over half the channels": ("ms /= (double)n;", "ms /= (double)(n / 2);"),
    "V2 odd head kept": ("    const int he = 2 * i, ho = 2 * i + 1;\n    const int g = he / G;        /* == ho / G because G is even */",
                         "    const int he = 2 * i + 1, ho = 2 * i;\n    const int g = he / G;        /* == ho / G because G is even */"),
    "V2 kv head h % Hkv": ("const int g = he / G;        /* == ho / G because G is even */",
                           "const int g = he % Hkv;"),
    "V2 sigmoid sign": ("    const double lg = J->lam[((int64_t)b * T + t) * P + i];\n    const double sg = 1.0 / (1.0 + exp(-lg));",
                        "    const double lg = J->lam[((int64_t)b * T + t) * P + i];\n    const double sg = 1.0 / (1.0 + exp(lg));"),
    "decode lengths ignored": ("const int64_t L = J->lens ? J->lens[b] : Lc;   /* rows this sequence attends */",
                               "const int64_t L = Lc;"),
    "V2 decode cache stride from the length": ("const double *k = J->k1 + ((int64_t)b * Lc * Hkv + g) * D;",
                                               "const double *k = J->k1 + ((int64_t)b * L * Hkv + g) * D;"),
    "V1 decode branch 2 reads k1": ("attend_row(q2, k2, (int64_t)H * d,", "attend_row(q2, k1, (int64_t)H * d,"),
    "bwd: RMSNorm Jacobian without its r^3 term": (
        "dx[c] = r * dy - r * r * r * x[c] * xdy / (double)dvd;", "dx[c] = r * dy;"),
    "bwd: dlam sign": ("dlam -= xa2;", "dlam += xa2;"),
    "bwd: dq without the score scale": ("dq[c] += scale * ds * kj[c];", "dq[c] += ds * kj[c];"),
    "bwd: softmax Jacobian without its mean term": ("const double ds = p[j] * (dp[j] - pdp);",
                                                    "const double ds = p[j] * dp[j];"),
    "bwd: V2 odd-head gradient sign": ("go[c] = -sg * dout[c];", "go[c] = sg * dout[c];"),
    "bwd: V2 dlam without (1 - sigmoid)": ("J->dlam[tok * P + i] = -sg * (1.0 - sg) * da;",
                                           "J->dlam[tok * P + i] = -sg * da;"),
    "bwd: V1 branch-2 gradient not scaled by lam": ("g2[c] = -J->lam_full * dx[c];", "g2[c] = -dx[c];"),
    "bwd: dk from the key instead of the query": ("dkj[c] += scale * ds * q[c];", "dkj[c] += scale * ds * kj[c];"),
    "rope: sign of the sine in the first half": ("out[row + i] = x1 * c - x2 * s;", "out[row + i] = x1 * c + x2 * s;"),
    "rope: frequency exponent -i/D": ("pow(base, -2.0 * (double)i / (double)D)", "pow(base, -(double)i / (double)D)"),
    "rope: pairs i with i + 1": ("const double x1 = x[row + i], x2 = x[row + i + half];",
                                 "const double x1 = x[row + i], x2 = x[row + (i + 1) % D];"),
    "lambda projection reads w transposed": ("acc += x[n * C + c] * w[(int64_t)c * P + i];",
                                             "acc += x[n * C + c] * w[(int64_t)i * C + c];"),
    "paired: own position excluded": ("const int64_t n = 2 * (int64_t)t + e + 1;      /* interleaved positions 0 .. 2t+e */",
                                      "const int64_t n = 2 * (int64_t)t + e + (t > 0 ? 0 : 1);"),
    "paired: partner's key of the same token always visible": (
        "const int64_t n = 2 * (int64_t)t + e + 1;      /* interleaved positions 0 .. 2t+e */",
        "const int64_t n = 2 * (int64_t)t + 2;"),
    "paired: heads swapped in the interleave": ("const int64_t ts = s / 2, hs = 2 * i + (int)(s % 2);",
                                                "const int64_t ts = s / 2, hs = 2 * i + 1 - (int)(s % 2);"),
    "paired: pairs (i, i + H/2)": ("const int i = h / 2, e = h % 2;", "const int i = h % (H / 2), e = h / (H / 2);"),
    "lse: key head h % Hk": ("const double *kj = k + (((int64_t)b * T + j) * Hk + h / G) * d;",
                             "const double *kj = k + (((int64_t)b * T + j) * Hk + h % Hk) * d;"),
    "lse: one future key": ("const int n = t + 1;   /* causal: keys 0 .. t */",
                            "const int n = t + 1 < T ? t + 2 : t + 1;"),
    "decode drops the last cache row": ("attend_row(qe, k, kv_row, v, kv_row, L, D, D, scale, scores, a1);",
                                        "attend_row(qe, k, kv_row, v, kv_row, L - 1, D, D, scale, scores, a1);"),
}

# mutants whose text stands at more than one site (every site is mutated:
# the same mistake made in the prefill, decode and backward of one variant)
SITES = {"scale 1/sqrt(2d) in V1": 4, "V1 combine sign": 2, "paired: heads swapped in the interleave": 2}

# pin checks that take only the oracle (parametrised ones get one case each)
CHECKS = [
    pins.test_lambda_init_printed_value_and_shape,
    pins.test_lambda_full_closed_forms,
    pins.test_rmsnorm_matches_library_and_unit_rms,
    pins.test_v1_hand_worked_example,
    lambda o: pins.test_v1_matches_four_sdpa_formulation(o, 2, 37, 3, 8, 4),
    pins.test_v1_lambda_zero_reduces_to_plain_attention,
    pins.test_v1_identical_branches,
    pins.test_first_row_is_first_value_row,
    lambda o: pins.test_v2_matches_library_gqa(o, 2, 29, 8, 2, 8),
    pins.test_v2_sigmoid_zero_gives_even_head_attention,
    pins.test_decode_matches_library_and_last_prefill_row,
    pins.test_v1_decode_matches_library_and_last_prefill_row,
    pins.test_decode_lengths_read_only_each_sequence_rows,
    pins.test_causality_future_rows_do_not_matter,
    lambda o: bwd_pins.test_v1_bwd_matches_autograd_of_library_forward(o, 1, 17, 2, 16, 0),
    lambda o: bwd_pins.test_v2_bwd_matches_autograd_of_library_forward(o, 2, 19, 8, 2, 8),
    bwd_pins.test_v1_bwd_finite_differences_of_the_forward,
    bwd_pins.test_v2_bwd_finite_differences_of_the_forward,
    bwd_pins.test_bwd_closed_forms,
    pro_pins.test_rope_identity_norm_and_inverse,
    pro_pins.test_rope_scores_depend_on_distance_only,
    pro_pins.test_rope_complex_form_and_quarter_turn,
    pro_pins.test_lambda_proj_one_hot_and_library,
    paired_pins.test_paired_page_interleave_order,
    paired_pins.test_paired_page_visibility_example,
    paired_pins.test_paired_matches_library_sdpa_on_interleaved,
    paired_pins.test_paired_closed_forms,
    pins.test_lse_closed_forms,
    lambda o: pins.test_lse_matches_library_logsumexp(o, 8, 2),
]


def _load_mutant(name, old, new, tmp_path):
    src = open(os.path.join(ORACLE_DIR, "diffattn_oracle.c")).read()
    assert src.count(old) == SITES.get(name, 1), f"mutation site count changed: {name}"
    c_path = tmp_path / "oracle_mut.c"
    c_path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{abs(hash(name))}",
                                                  os.path.join(ORACLE_DIR, "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(c_path)
    mod._LIB = str(tmp_path / "liboracle_mut.so")
    mod._lib = None
    mod.build(force=True)
    return mod


def test_unmutated_copy_passes_every_check(tmp_path):
    mod = _load_mutant("none", "ms /= (double)n;", "ms /= (double)n;", tmp_path)
    for check in CHECKS:
        check(mod)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new, tmp_path)
    failed = []
    for check in CHECKS:
        try:
            check(mod)
        except (AssertionError, RuntimeError, FloatingPointError, ValueError):
            failed.append(getattr(check, "__name__", "lambda"))
    assert failed, f"no pin caught the mutant '{name}'"
