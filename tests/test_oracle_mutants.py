"""Plant plausible mistakes in copies of the C oracle and check that the pins catch each.

Every mutant is a textual edit of a temporary copy of oracle/diffattn_oracle.c,
compiled with gcc on the CPU; the real oracle is never modified.  A mutant that
passes every pin would show a hole in the pins.
"""
import os
import shutil

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "diffattn_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("plus_lambda", "w[j] = p1[j] - lam * p2[j];", "w[j] = p1[j] + lam * p2[j];"),
    ("no_scale", "const double scale = 1.0 / sqrt((double)d);", "const double scale = 1.0;"),
    ("scale_by_2d", "const double scale = 1.0 / sqrt((double)d);",
     "const double scale = 1.0 / sqrt((double)(2 * d));"),
    ("strict_mask", "return causal ? (j <= i) : 1;", "return causal ? (j < i || j == 0) : 1;"),
    ("reversed_mask", "return causal ? (j <= i) : 1;", "return causal ? (j >= i) : 1;"),
    ("causal_ignored", "return causal ? (j <= i) : 1;", "return 1;"),
    ("transposed_k", "s += q_row[c] * k[j * d + c];", "s += q_row[c] * k[c * N + j];"),
    ("map2_uses_q1", "softmax_row(i, N, d, q2_row, k2, causal, p2);",
     "softmax_row(i, N, d, q1_row, k2, causal, p2);"),
    ("unnormalised_map", "p[j] /= sum;", "p[j] /= 1.0;"),
    ("v_columns_reversed", "o[c] += wrow[j] * v[j * dv + c];",
     "o[c] += wrow[j] * v[j * dv + (dv - 1 - c)];"),
    ("norm_over_d", "ms /= (double)dv;", "ms /= (double)(dv / 2);"),
    ("eps_outside_sqrt", "const double r = 1.0 / sqrt(ms + eps);",
     "const double r = 1.0 / (sqrt(ms) + eps);"),
    ("no_lambda_init_scale", "o[c] = o[c] * r * g * (1.0 - lambda_init);",
     "o[c] = o[c] * r * g;"),
    ("lambda_init_not_one_based", "exp(-0.3 * (double)(layer - 1))", "exp(-0.3 * (double)(layer))"),
    ("lambda_init_sign", "0.8 - 0.6 * exp(", "0.8 + 0.6 * exp("),
    ("lambda_of_head0", "lam[h], causal, headnorm, w ? w + (int64_t)h * dv : NULL,\n"
     "                    eps, lambda_init, scratch, out + vo + i * dv);",
     "lam[0], causal, headnorm, w ? w + (int64_t)h * dv : NULL,\n"
     "                    eps, lambda_init, scratch, out + vo + i * dv);"),
    ("weight_of_head0", "lam[h], causal, headnorm, w ? w + (int64_t)h * dv : NULL,\n"
     "                    eps, lambda_init, scratch, out + vo + i * dv);",
     "lam[h], causal, headnorm, w ? w : NULL,\n"
     "                    eps, lambda_init, scratch, out + vo + i * dv);"),
    # key/value-cache form
    ("kv_top_left_mask", "const int64_t pos = Nkv - Nq + i;", "const int64_t pos = i;"),
    ("kv_position_off_by_one", "const int64_t pos = Nkv - Nq + i;",
     "const int64_t pos = Nkv - Nq + i - 1;"),
    ("kv_key_stride_of_queries", "ko = bh * Nkv * d,", "ko = bh * Nq * d,"),
    ("kv_value_stride_of_queries", "vo = bh * Nkv * dv;", "vo = bh * Nq * dv;"),
    ("kv_query_stride_of_keys", "qo = bh * Nq * d,", "qo = bh * Nkv * d,"),
    # backward
    ("bwd_ds2_sign", "const double ds2 = p2[j] * (-lam * dvj + lam * do_o2);",
     "const double ds2 = p2[j] * (lam * dvj - lam * do_o2);"),
    ("bwd_softmax_centre_dropped", "const double ds1 = p1[j] * (dvj - do_o1);",
     "const double ds1 = p1[j] * dvj;"),
    ("bwd_dk_unscaled", "dk1[j * d + c] += ds1 * q1i[c] * scale;",
     "dk1[j * d + c] += ds1 * q1i[c];"),
    ("bwd_dv_plus_lambda", "dv[j * dv_ + c] += (p1[j] - lam * p2[j]) * dout[c];",
     "dv[j * dv_ + c] += (p1[j] + lam * p2[j]) * dout[c];"),
    ("bwd_norm_term_halved",
     "dout[c] = r * g * dyi[c] - r * r * r / (double)dv_ * (o[c] - mu) * t;",
     "dout[c] = r * g * dyi[c] - r * r * r / (double)(2 * dv_) * (o[c] - mu) * t;"),
    ("bwd_dw_missing_lambda_init", "dw[c] += dyi[c] * (o[c] - mu) * r * (1.0 - lambda_init);",
     "dw[c] += dyi[c] * (o[c] - mu) * r;"),
    ("bwd_groupnorm_do_not_centred", "dout[c] -= md;", "dout[c] -= 0.0 * md;"),
    ("bwd_groupnorm_mean_dropped", "                    mu += o[c];\n",
     "                    mu += 0.0 * o[c];\n"),
    ("bwd_groupnorm_dw_uncentred", "dw[c] += dyi[c] * (o[c] - mu) * r * (1.0 - lambda_init);",
     "dw[c] += dyi[c] * o[c] * r * (1.0 - lambda_init);"),
    ("bwd_dlambda_of_map1", "*dlam -= do_o2;", "*dlam -= do_o1;"),
    ("groupnorm_variance_uncentred", "var += (o[c] - mu) * (o[c] - mu);", "var += o[c] * o[c];"),
    ("groupnorm_output_uncentred", "o[c] = (o[c] - mu) * rg * g * (1.0 - lambda_init);",
     "o[c] = o[c] * rg * g * (1.0 - lambda_init);"),
    ("groupnorm_mean_over_d", "    mu /= (double)dv;\n", "    mu /= (double)(dv / 2);\n"),
    ("bwd_dq2_uses_k1", "dq2[i * d + c] += ds2 * k2[j * d + c] * scale;",
     "dq2[i * d + c] += ds2 * k1[j * d + c] * scale;"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, mut):
    text = open(SRC).read()
    assert text.count(orig) >= 1, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(orig, mut))
    lib_path = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load(lib_path)
    res = pins.run_pins(lib)
    failed = [k for k, (ok, _) in res.items() if not ok]
    assert failed, f"mutant {name} passed every pin"
