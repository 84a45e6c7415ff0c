"""CPU tier: the pins have teeth. Each case copies oracle/oracle.c, plants one
plausible mistake (a dropped term, a wrong sign, divisor or index, a
different rounding rule), builds the copy with gcc in a temporary directory
and requires at least one pin of tests/oracle_pins.py to fail on it.

Mistakes are planted only in throw-away copies on the CPU; the oracle itself
is never modified.
"""
import os
import shutil

import pytest

import oracle
from oracle import build as obuild
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, mutated text); the original must occur exactly once.
MUTANTS = [
    ("fwd_divisor_H_plus_1", "double ms = ss / (double)H;",
     "double ms = ss / (double)(H + 1);"),
    ("fwd_eps_dropped", "double r = 1.0 / sqrt(ms + eps);",
     "double r = 1.0 / sqrt(ms);"),
    ("fwd_eps_outside_sqrt", "double r = 1.0 / sqrt(ms + eps);",
     "double r = 1.0 / (sqrt(ms) + eps);"),
    ("fwd_no_sqrt", "double r = 1.0 / sqrt(ms + eps);",
     "double r = 1.0 / (ms + eps);"),
    ("fwd_weight_reversed",
     "y[i * H + j] = dec(w, dtype, j) * dec(x, dtype, i * H + j) * r;",
     "y[i * H + j] = dec(w, dtype, H - 1 - j) * dec(x, dtype, i * H + j) * r;"),
    ("fwd_store_transposed",
     "y[i * H + j] = dec(w, dtype, j)", "y[j * M + i] = dec(w, dtype, j)"),
    ("fwd_weight_dropped",
     "y[i * H + j] = dec(w, dtype, j) * dec(x, dtype, i * H + j) * r;",
     "y[i * H + j] = dec(x, dtype, i * H + j) * r;"),
    ("bwd_eps_dropped", "double r = 1.0 / sqrt(ss / (double)H + eps);",
     "double r = 1.0 / sqrt(ss / (double)H);"),
    ("bwd_divisor_wrong", "double r = 1.0 / sqrt(ss / (double)H + eps);",
     "double r = 1.0 / sqrt(ss / (double)(H + 1) + eps);"),
    ("bwd_dx_sign", "r * (wdy - xv * r * r * c)", "r * (wdy + xv * r * r * c)"),
    ("bwd_dx_term_dropped", "r * (wdy - xv * r * r * c)", "r * (wdy)"),
    ("bwd_dx_r_power", "r * (wdy - xv * r * r * c)", "r * (wdy - xv * r * c)"),
    ("bwd_dx_outer_r_dropped", "dx[i * H + j] = r * (wdy - xv * r * r * c);",
     "dx[i * H + j] = (wdy - xv * r * r * c);"),
    ("bwd_c_not_mean", "double c = csum / (double)H;", "double c = csum;"),
    ("bwd_c_without_w", "double wdy = dec(w, dtype, j) * dec(dy, dtype, i * H + j);",
     "double wdy = dec(dy, dtype, i * H + j);"),
    ("bwd_dx_without_w", "double wdy = dec(w, dtype, j) * dyv;",
     "double wdy = dyv;"),
    ("bwd_dw_no_r", "dw[j] += dyv * xv * r;", "dw[j] += dyv * xv;"),
    ("bwd_dw_with_w", "dw[j] += dyv * xv * r;", "dw[j] += wdy * xv * r;"),
    ("bwd_dw_last_row_only", "dw[j] += dyv * xv * r;", "dw[j] = dyv * xv * r;"),
    ("bwd_tdx_power", "fabs(xv) * r * r * r * (cabs / (double)H)",
     "fabs(xv) * r * (cabs / (double)H)"),
    ("bwd_tdw_signed", "tdw[j] += fabs(dyv * xv * r);", "tdw[j] += dyv * xv * r;"),
    ("bf16_ties_away", "double n = nearbyint(scaled);", "double n = round(scaled);"),
    ("bf16_truncate", "double n = nearbyint(scaled);", "double n = trunc(scaled);"),
    ("bf16_double_rounding", "(void)frexp(v, &e);",
     "v = (double)(float)v;\n    (void)frexp(v, &e);"),
    ("bf16_no_subnormal_clamp", "if (q < -133)\n        q = -133;", ""),
    ("bf16_decode_shift", "((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    ("f16_ties_away", "double r = ldexp(nearbyint(ldexp(a, -q)), q);",
     "double r = ldexp(round(ldexp(a, -q)), q);"),
    ("f16_truncate", "double r = ldexp(nearbyint(ldexp(a, -q)), q);",
     "double r = ldexp(trunc(ldexp(a, -q)), q);"),
    ("f16_10_bit_significand", "int q = e - 11;", "int q = e - 10;"),
    ("f16_no_subnormal_clamp", "if (q < -24)\n        q = -24;", ""),
    ("f16_overflow_at_max", "if (r > 65504.0)", "if (r >= 65504.0)"),
    ("f16_decode_bias", "v = ldexp((double)(1024 + frac), exp - 25);",
     "v = ldexp((double)(1024 + frac), exp - 24);"),
    ("f16_decode_subnormal_scale", "v = ldexp((double)frac, -24);",
     "v = ldexp((double)frac, -25);"),
    ("f16_decode_as_bf16", "return oracle_f16_to_double(((const uint16_t *)p)[i]);",
     "return oracle_bf16_to_double(((const uint16_t *)p)[i]);"),
    ("gemv_unrounded_y", "            y[i * H + j] = round_to(dtype, y[i * H + j]);\n", ""),
    ("gemv_A_transposed", "dec(A, dtype, n * H + k)", "dec(A, dtype, k * N + n)"),
    ("gemv_x_not_h", "oracle_residual_fwd(M, H, x, res, w, dtype, eps, h, y, rstd);",
     "oracle_rmsnorm_fwd(M, H, x, w, dtype, eps, y, rstd);"),
    ("gemv_tout_signed", "mag += fabs(term);", "mag += term;"),
    ("gemv_last_k_dropped", "for (int64_t k = 0; k < H; ++k) {\n                double term",
     "for (int64_t k = 0; k < H - 1; ++k) {\n                double term"),
    ("gemv_f16_rounded_as_bf16",
     "return oracle_f16_to_double(oracle_f16_from_double(v));",
     "return oracle_bf16_to_double(oracle_bf16_from_double(v));"),
    ("bwd2_eps_dropped", "double r = 1.0 / sqrt(mean_sq + eps);",
     "double r = 1.0 / sqrt(mean_sq);"),
    ("bwd2_r_power", "(3.0 * r * r * c * B - A - D)", "(3.0 * r * c * B - A - D)"),
    ("bwd2_coeff_3", "(3.0 * r * r * c * B - A - D)", "(2.0 * r * r * c * B - A - D)"),
    ("bwd2_D_dropped", "(3.0 * r * r * c * B - A - D)", "(3.0 * r * r * c * B - A)"),
    ("bwd2_gx_term_sign", "dx2[i * H + k] = u1 - u2 - u3 + u4;",
     "dx2[i * H + k] = u1 - u2 + u3 + u4;"),
    ("bwd2_ddy_gw_dropped", "ddy[i * H + k] = t1 - t2 + t3;", "ddy[i * H + k] = t1 - t2;"),
    ("bwd2_dw_second_term", "dw2[k] += v1 - v2;", "dw2[k] += v1;"),
    ("bwd2_A_uses_x", "A += g * wv * dyv;", "A += g * wv * xv;"),
    ("bwd2_B_over_H_missing", "double t1 = r * wv * g, t2 = (r3 * B / (double)H) * wv * xv",
     "double t1 = r * wv * g, t2 = (r3 * B) * wv * xv"),
    ("resid_subtract",
     "double s = dec(x, dtype, i * H + j) + dec(res, dtype, i * H + j);",
     "double s = dec(x, dtype, i * H + j) - dec(res, dtype, i * H + j);"),
    ("resid_unrounded_norm_input",
     "oracle_rmsnorm_fwd(M, H, h, w, dtype, eps, y, rstd);",
     "oracle_rmsnorm_fwd(M, H, x, w, dtype, eps, y, rstd);"),
    ("resid_dh_dropped", "dx[i * H + j] += g;", "dx[i * H + j] += 0.0 * g;"),
    ("resid_dh_sign", "dx[i * H + j] += g;", "dx[i * H + j] -= g;"),
]


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("mutants")


def test_mutant_table_is_unique():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, f"{name}: anchor occurs {src.count(old)}x"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: anchor not unique in oracle.c"
    msrc = workdir / f"{name}.c"
    msrc.write_text(src.replace(old, new))
    lib = obuild.build(force=True, src=str(msrc), out=str(workdir / f"{name}.so"))
    bad = oracle_pins.failing_pins(oracle.Oracle(lib))
    assert bad, f"planted mistake {name!r} passed every pin"
