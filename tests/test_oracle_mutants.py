"""The pins catch mistakes: plant one plausible mistake at a time in a copy of
the oracle's C source, build it, run the oracle's pin tests against it and
expect them to fail.

Each mutant is a mistake a careful author could make while writing the
oracle from the pages: a tie rule, a format's bias or saturation, a piece of
the FP4 rounding, a constant of the global scale, a dropped term or a
transposed operand in the closed forms of CJSO, a missing re-quantization, a
wrong candidate set in the decoupled search, a nibble order, a lost sign.  A
mutant that every pin lets through marks a part of the oracle that nothing
independent checks.  Mutants that cannot change any output (equivalent
rewrites) are not listed.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (name, exact text in nvfp4_oracle.c, replacement)
MUTANTS = [
    # number formats
    ("e2m1_ties_away_from_zero", "q = 0.5 * rne(2.0 * a);", "q = 0.5 * floor(2.0 * a + 0.5);"),
    ("e2m1_top_piece_step_one", "q = 2.0 * rne(0.5 * a);", "q = rne(a);"),
    ("e2m1_no_saturation", "if (q > 6.0) q = 6.0;", ""),
    ("e2m1_value_table", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}"),
    ("e4m3_bias_8", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("e4m3_subnormal_step", "(int)rne(r * 512.0)", "(int)rne(r * 256.0)"),
    ("e4m3_saturates_to_nan", "if (r >= 448.0) return 0x7E;", "if (r >= 448.0) return 0x7F;"),
    ("e4m3_truncates", "double t = rne(ldexp(r, 3 - e));", "double t = floor(ldexp(r, 3 - e));"),
    ("e4m3_floor_strict", "if (e4m3_value(mid) <= r) lo = mid; else hi = mid;",
     "if (e4m3_value(mid) < r) lo = mid; else hi = mid;"),
    ("e4m3_ceil_off_by_one", "  return hi;\n}\n\n/* fp32 -> bf16", "  return hi + 1;\n}\n\n/* fp32 -> bf16"),
    ("bf16_ties_away", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    # quantizer
    ("quotient_by_reciprocal", "float v = fabsf(x[j]) / s;", "float v = fabsf(x[j]) * (1.0f / s);"),
    ("quotient_scale_dropped_alpha", "float s = alpha * delta;\n  double p", "float s = delta;\n  double p"),
    ("P_signed", "p += fabs((double)x[j]) * q;", "p += (double)x[j] * q;"),
    ("R_not_squared", "rr += q * q;", "rr += q;"),
    ("zero_scale_block_unguarded", "if (s == 0.0f) {\n    memset", "if (0) {\n    memset"),
    ("code_sign_dropped", "int lo = mag[j] | (f32_signbit(x[j]) << 3);", "int lo = mag[j];"),
    ("nibbles_swapped", "out8[j / 2] = (uint8_t)(lo | (hi << 4));", "out8[j / 2] = (uint8_t)(hi | (lo << 4));"),
    ("block_amax_signed", "m = fmaxf(m, fabsf(x[j]));", "m = fmaxf(m, x[j]);"),
    ("alpha_m_fp8_480", "return amax / 2688.0f;", "return amax / 2880.0f;"),
    ("six_alpha_four", "c->six_alpha = alpha * 6.0f;", "c->six_alpha = alpha * 4.0f;"),
    # FourOverSix
    ("fos_factor", "e4m3_code((double)(delta6 * 1.5f))", "e4m3_code((double)(delta6 * 1.25f))"),
    ("fos_tie_prefers_m4", "int use4 = g4 < g6;", "int use4 = g4 <= g6;"),
    ("fos_error_sign", "return s * fmaf(s, R, -2.0f * P);", "return s * fmaf(s, R, 2.0f * P);"),
    ("fos_error_missing_factor_2", "return s * fmaf(s, R, -2.0f * P);", "return s * fmaf(s, R, -P);"),
    ("fos_error_compares_scale_of_m6", "float g4 = cand_err(c->alpha * delta4, P4, R4);",
     "float g4 = cand_err(c->alpha * delta6, P4, R4);"),
    # CJSO
    ("alpha_den_printed_form", "den += (unsigned __int128)(M * M) * R4;", "den += (unsigned __int128)(M * 512) * R4;"),
    ("alpha_num_dropped_delta", "const unsigned __int128 t = (unsigned __int128)(M * mP);",
     "const unsigned __int128 t = (unsigned __int128)(512 * mP);"),
    ("alpha_sum_units_too_coarse", "0xFFu) - 127 - 48;", "0xFFu) - 127 - 8;"),
    ("alpha_sum_rounds_half_up", "if (rem > half || (rem == half && (top & 1))) top += 1;", "if (rem >= half) top += 1;"),
    ("alpha_quotient_in_float", "return (float)(nd / dd);", "return (float)nd / (float)dd;"),
    ("delta_step_transposed", "float t = P / (c->alpha * R);", "float t = R / (c->alpha * P);"),
    ("delta_step_dropped_alpha", "float t = P / (c->alpha * R);", "float t = P / R;"),
    ("delta_step_without_requantize",
     "  quant_block(x, c->alpha, (float)e4m3_value(d), mag, &P, &R);\n  if (R > 0.0f) {",
     "  P = c->P[b];\n  R = c->R[b];\n  if (R > 0.0f) {"),
    ("cjso_skips_alpha_step", "set_alpha(&c, alpha_step(&c, c.alpha));\n      c.write_codes",
     "c.write_codes"),
    # decoupled search
    ("decoupled_grid_shifted", "float m = (float)((50 + k) / 100.0);", "float m = (float)((49 + k) / 100.0);"),
    ("decoupled_grid_narrow", "float m = (float)((50 + k) / 100.0);", "float m = (float)((75 + k / 2) / 100.0);"),
    ("decoupled_floor_only", "for (int h = 0; h < 2; ++h) {", "for (int h = 0; h < 1; ++h) {"),
    ("decoupled_stored_scale_is_dq", "float sd = c->alpha * (float)e4m3_value(cand[h]);",
     "float sd = c->alpha * dq;"),
    ("decoupled_starts_from_max_rule", "int d0 = c->dcode[b];\n  float delta0",
     "int d0 = max_rule_code(c, x);\n  float delta0"),
    # dequantization
    ("dequant_nibble_order", "int code = (codes[i / 2] >> (4 * (i & 1))) & 0xF;\n    float q",
     "int code = (codes[i / 2] >> (4 * (1 - (i & 1)))) & 0xF;\n    float q"),
    ("dequant_truncates", "out[i] = f32_to_bf16_rne(q * s);", "{ float t = q * s; uint32_t u; memcpy(&u, &t, 4); "
                                                               "out[i] = (uint16_t)(u >> 16); }"),
    ("dequant_scale_by_block_of_8", "float s = alpha * (float)e4m3_value(scales[i / BLOCK]);\n    out",
     "float s = alpha * (float)e4m3_value(scales[i / 8]);\n    out"),
    # W4A16 product
    ("gemv_skips_bf16_rounding", "double w = (double)bf16_to_f32(f32_to_bf16_rne(q * s));", "double w = (double)(q * s);"),
    ("gemv_activation_transposed", "acc += w * (double)bf16_to_f32(x[(int64_t)b * cols + c]);",
     "acc += w * (double)bf16_to_f32(x[c * batch + b]);"),
    ("gemv_output_transposed", "y[(int64_t)b * rows + r] = acc;", "y[r * batch + b] = acc;"),
    # tensor-core scale layout
    ("swizzle_row_tiles_fastest", "int64_t tile = (i / 128) * ct + k / 4;",
     "int64_t tile = (k / 4) * ((rows + 127) / 128) + i / 128;"),
    ("swizzle_interleave_swapped", "out[tile * 512 + (r % 32) * 16 + (r / 32) * 4 + c]",
     "out[tile * 512 + (r / 32) * 16 + (r % 32) * 4 + c]"),
    ("gemv_drops_code_sign", "if (code & 8) q = -q;\n        float s = alpha", "float s = alpha"),
]

PIN_FILES = [os.path.join(HERE, "test_oracle_method.py"), os.path.join(HERE, "test_oracle_formats.py")]


def _run_mutant(workdir, name, old, new):
    src = open(oracle.SRC).read()
    n = src.count(old)
    if n != 1:
        return name, "bad-site", f"pattern found {n} times"
    mdir = os.path.join(workdir, name)
    os.makedirs(mdir)
    msrc = os.path.join(mdir, "oracle_mutant.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(mdir, "liboracle_mutant.so")
    try:
        oracle.compile_source(msrc, so)
    except subprocess.CalledProcessError as e:
        return name, "no-build", str(e)
    env = dict(os.environ, NVFP4_ORACLE_LIB=so, PYTHONDONTWRITEBYTECODE="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"] + PIN_FILES
    try:
        r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    except subprocess.TimeoutExpired:
        return name, "caught", "timeout"  # a mutant that loops forever is caught too
    tail = r.stdout.strip().splitlines()[-1:] if r.stdout else []
    if r.returncode == 1:
        return name, "caught", " ".join(tail)
    if r.returncode == 0:
        return name, "survived", " ".join(tail)
    return name, f"error rc={r.returncode}", (r.stdout + r.stderr)[-400:]


def test_env_override_selects_the_library(tmp_path):
    so = os.path.join(str(tmp_path), "liboracle_copy.so")
    shutil.copy(oracle.build(), so)
    code = "import oracle; print(oracle.lib()._name)"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       env=dict(os.environ, NVFP4_ORACLE_LIB=so), timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == so, r.stderr


def test_every_planted_mistake_fails_a_pin(tmp_path):
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    oracle.build()
    workers = max(2, min(8, os.cpu_count() or 2))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda m: _run_mutant(str(tmp_path), *m), MUTANTS))
    bad = [r for r in results if r[1] != "caught"]
    assert not bad, "\n".join(f"{n}: {s} {d}" for n, s, d in bad)
