"""The pins are sharp: every plausible mistake planted in a copy of the oracle's
source is caught by at least one pin (CPU only).

Each mutant replaces one exact snippet of ``oracle/qref.c`` (the test fails if
the snippet is not found, so the list stays in step with the source), compiles
the copy into a temporary library, and runs every pin against it through
``oracle.using``.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "qref.c")

MUTANTS = {
    "int4_zero_point_7": ("return (double)(code - 8);", "return (double)(code - 7);"),
    "int4_high_nibble_first": ("(row[i / 2] >> (4 * (i % 2)))", "(row[i / 2] >> (4 * (1 - i % 2)))"),
    "int2_zero_point_1": ("return (double)(code - 2);", "return (double)(code - 1);"),
    "int2_high_bits_first": ("(row[i / 4] >> (2 * (i % 4)))", "(row[i / 4] >> (2 * (3 - i % 4)))"),
    "int8_ones_complement": ("if (v >= 128) v -= 256;", "if (v >= 128) v -= 255;"),
    "int8_unsigned": ("if (v >= 128) v -= 256;", ";"),
    "f32_byte_offset": ("memcpy(&f, row + 4 * i, sizeof f);", "memcpy(&f, row + i, sizeof f);"),
    "scale_dropped": ("double sc = scales ? (double)scales[o] : 1.0;", "double sc = 1.0;"),
    "scale_squared": ("double sc = scales ? (double)scales[o] : 1.0;",
                      "double sc = scales ? (double)scales[o] * scales[o] : 1.0;"),
    "x_transposed": ("* (double)xs[i];", "* (double)x[i * S + s];"),
    "x_row_stride_O": ("const float *xs = x + s * I;", "const float *xs = x + s * O;"),
    "last_term_dropped": ("for (long i = 0; i < I; ++i) {\n            double t",
                          "for (long i = 0; i + 1 < I; ++i) {\n            double t"),
    "bound_signed": ("bnd += fabs(t);", "bnd += t;"),
    "bound_signed_scale": ("bound[so] = fabs(sc) * bnd;", "bound[so] = sc * bnd;"),
    "int4_row_bytes_floor": ("case QREF_I4:  return (I + 1) / 2;", "case QREF_I4:  return I / 2;"),
    "int2_row_bytes_floor": ("case QREF_I2:  return (I + 3) / 4;", "case QREF_I2:  return I / 4;"),
    "silu_sign": ("double v = z / (1.0 + exp(-z)) * (double)u[k];",
                  "double v = z / (1.0 + exp(z)) * (double)u[k];"),
    "silu_no_u": ("double v = z / (1.0 + exp(-z)) * (double)u[k];",
                  "double v = z / (1.0 + exp(-z));"),
    "bf16_ties_odd": ("return ((lo_bits >> 16) & 1u) ? hi : lo;", "return ((lo_bits >> 16) & 1u) ? lo : hi;"),
    "bf16_truncate": ("if (dlo < dhi) return lo;", "return lo;"),
    "gate_up_same_tensor": ("return qref_matmul(fmt, O, I, codes_u, scales_u, x, S, yu, NULL, bound_u);",
                            "return qref_matmul(fmt, O, I, codes_g, scales_g, x, S, yu, NULL, bound_u);"),
    "y_rounded_before_scale": ("y[so] = (float)(sc * acc);", "y[so] = (float)(sc * (float)acc);"),
    "gs_first_scale_only": ("double sc = (double)gscales[o * G + g];", "double sc = (double)gscales[o * G];"),
    "gs_bound_unscaled": ("bnd += fabs(sc) * gb;", "bnd += gb;"),
    "gs_short_group_dropped": ("long G = (I + gs - 1) / gs;", "long G = I / gs;"),
    "rms_sum_not_mean": ("double inv = 1.0 / sqrt(ss / (double)D + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    "rms_no_root": ("double inv = 1.0 / sqrt(ss / (double)D + eps);", "double inv = 1.0 / (ss / (double)D + eps);"),
    "rms_eps_outside_root": ("double inv = 1.0 / sqrt(ss / (double)D + eps);",
                             "double inv = 1.0 / (sqrt(ss / (double)D) + eps);"),
    "rms_abs_not_square": ("ss += (double)hv * (double)hv;", "ss += fabs((double)hv);"),
    "rms_weight_dropped": ("double v = (double)hv * (double)w[d] * inv;", "double v = (double)hv * inv;"),
    "mla_window_from_zero": ("long first = st0, last = T - S + s;", "long first = 0, last = T - S + s;"),
    "mla_window_short_by_one": ("long first = st0, last = T - S + s;", "long first = st0, last = T - S + s - 1;"),
    "mla_window_not_causal": ("long first = st0, last = T - S + s;", "long first = st0, last = T - 1;"),
    "mla_values_from_key_rows": ("long key0 = h * (Dn + Dv), val0 = key0 + Dn;",
                                 "long key0 = h * (Dn + Dv), val0 = key0;"),
    "mla_head_stride_dn": ("long key0 = h * (Dn + Dv), val0 = key0 + Dn;",
                           "long key0 = h * Dn, val0 = key0 + Dn;"),
    "mla_rope_dropped": ("                dot += t;\n", "                (void)t;\n"),
    "mla_scale_dropped": ("score[w] = dot * scale;", "score[w] = dot;"),
    "mla_softmax_unnormalized": ("double p = score[w] / z;", "double p = score[w];"),
    "mla_q_head_token_swapped": ("const float *qn = q_nope + (s * H + h) * Dn;",
                                 "const float *qn = q_nope + (h * S + s) * Dn;"),
    "mla_key_scale_dropped": ("double kw = mla_scale(scales, gs, G, key0 + d, i) *", "double kw = 1.0 *"),
    "mla_value_scale_dropped": ("double vw = mla_scale(scales, gs, G, val0 + v, i) *", "double vw = 1.0 *"),
    "mla_first_group_scale_only": ("return gs ? (double)scales[row * G + i / gs] : (double)scales[row];",
                                   "return gs ? (double)scales[row * G] : (double)scales[row];"),
    "mla_group_stride_one": ("return gs ? (double)scales[row * G + i / gs] : (double)scales[row];",
                             "return gs ? (double)scales[row + i / gs] : (double)scales[row];"),
    "mla_bound_without_softmax_term": ("bound[out] = (1.0 + amax) * b;", "bound[out] = b;"),
    "mla_latent_not_weighted": ("clat[i] += p * (double)lt[i];", "clat[i] += (double)lt[i] / (double)nwin;"),
    "rms_residual_dropped": ("float hv = r ? (float)((double)x[s * D + d] + (double)r[s * D + d]) : x[s * D + d];\n            if (h)",
                             "float hv = x[s * D + d];\n            if (h)"),
}


def _compile(text: str, out: str):
    with tempfile.NamedTemporaryFile("w", suffix=".c", delete=False) as f:
        f.write(text)
        c = f.name
    try:
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared", c,
                               "-o", out, "-lm"])
    finally:
        os.unlink(c)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found once: %r" % old
    so = str(tmp_path / ("qref_%s.so" % name))
    _compile(src.replace(old, new), so)
    failures = []
    with oracle.using(so):
        for check in P.ALL_CHECKS:
            try:
                check()
            except AssertionError:
                failures.append(check.__name__)
            except (ValueError, IndexError) as e:          # a broken layout may also raise
                failures.append("%s (%s)" % (check.__name__, type(e).__name__))
    assert failures, "planted mistake %s passed every pin" % name
