"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a copy of oracle/qk_oracle.c with one plausible slip (a wrong
bias, a dropped term, a swapped index, a transposed operand, the other
epilogue association ...), compiled to a temporary library.  The pins of
oracle_pins.py run against it; at least one must fail.

The E2M1 nibble order is deliberately not among them: swapping it in both
operands permutes element pairs inside one 32-element block, which leaves
every GEMM result unchanged, so no GEMM-level pin can (or needs to) see it.
"""
import os
import shutil
import tempfile

import pytest

import oracle
from oracle_pins import ALL_CHECKS

SRC = os.path.join(os.path.dirname(oracle.__file__), "qk_oracle.c")

MUTANTS = {
    "epilogue_association": ("x = x * sa[m];\n      x = x * sb[n];", "x = x * (sa[m] * sb[n]);"),
    "int8_bias_dropped": ("if (bias) x = x + qko_bf16_to_f32(bias[n]);", "(void)bias;"),
    "int8_transposed_B": ("acc += (int64_t)a[k] * (int64_t)b[k];", "acc += (int64_t)a[k] * (int64_t)B[k * N + n];"),
    "int8_range_check_dropped": ("if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;", ""),
    "e4m3_exponent_bias": ("mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, (int)e - 8);"),
    "e4m3_subnormal": ("mag = ldexp((double)m / 8.0, 1 - 7);", "mag = ldexp((double)m / 8.0, 0 - 7);"),
    "e4m3_no_nan": ("if (e == 15u && m == 7u) return NAN;", ""),
    "e2m1_exponent_bias": ("mag = ldexp(1.0 + (double)m / 2.0, (int)e - 1);", "mag = ldexp(1.0 + (double)m / 2.0, (int)e - 2);"),
    "ue8m0_bias": ("return ldexp(1.0, (int)code - 127);", "return ldexp(1.0, (int)code - 128);"),
    "bf16_truncates": ("u += 0x7fffu + lsb;", "(void)lsb;"),
    "f16_ties_away": ("nearbyint(v / spacing)", "floor(v / spacing + 0.5)"),
    "f16_overflow_saturates": ("if (r > 65504.0) return (uint16_t)(sign | 0x7c00u);",
                               "if (r > 65504.0) return (uint16_t)(sign | 0x7bffu);"),
    "f16_subnormal_spacing": ("if (e < -14) e = -14;", "if (e < -15) e = -15;"),
    "int8_fp32_out_rounded": ("((float*)out)[o] = x;", "((float*)out)[o] = qko_bf16_to_f32(qko_f32_to_bf16_rne(x));"),
    "int8_fp16_out_is_bf16": ("((uint16_t*)out)[o] = qko_f32_to_f16_rne(x);", "((uint16_t*)out)[o] = qko_f32_to_bf16_rne(x);"),
    "fp4_decoded_as_e4m3": ("return g_e2m1[nib];", "return g_e4m3[nib];"),
    "mx_block_index_dropped": ("g_ue8m0[sB[n * kb + blk]]", "g_ue8m0[sB[n * kb]]"),
    "mx_b_scale_dropped": ("acc += g_ue8m0[sA[m * kb + blk]] * g_ue8m0[sB[n * kb + blk]] * inner;",
                           "acc += g_ue8m0[sA[m * kb + blk]] * inner;"),
    "fp8_wrong_column_scale": ("double x = acc * (double)sa[m] * (double)sb[n];",
                               "double x = acc * (double)sa[m] * (double)sb[m % N];"),
    "fp8_bias_sign": ("if (bias) x += (double)qko_bf16_to_f32(bias[n]);", "if (bias) x -= (double)qko_bf16_to_f32(bias[n]);"),
    "encoder_ties_away": ("(err == best_err && (c & 1u) == 0u)", "(err == best_err && c > best)"),
    "ptpc_scale_divisor": ("float s = amax / 448.0f;", "float s = amax / 240.0f;"),
    "ptpc_zero_row_scale": ("if (amax == 0.0f) s = 1.0f;", "if (amax == 0.0f) s = 0.5f;"),
    "ptpc_division_in_double": ("float q = x[k] / s;", "double q = (double)x[k] / (double)s;"),
    "ptpc_reciprocal_multiply": ("float q = x[k] / s;", "float q = x[k] * (1.0f / s);"),
    "mx_quantize_floor_off_by_one": ("sexp = (e - 1) - emax;", "sexp = e - emax;"),
    "e2m1_encoder_ties_up": ("(err == best_err && (c & 1u) == 0u)", "(err <= best_err)"),
    "mx_emax": ("int emax = (fmt == QKO_FMT_MXFP8_E4M3) ? 8 : 2;", "int emax = (fmt == QKO_FMT_MXFP8_E4M3) ? 7 : 2;"),
    "ue4m3_exponent_bias": ("return ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
                            "return ldexp(1.0 + (double)m / 8.0, (int)e - 6);"),
    "nvfp4_blocks_of_32": ("const int64_t kb = K / 16;", "const int64_t kb = K / 32;"),
    "nvfp4_global_b_dropped": ("acc *= (double)ga * (double)gb;", "acc *= (double)ga;"),
    "nvfp4_scales_read_as_ue8m0": ("acc += g_ue4m3[sA[m * kb + blk]] * g_ue4m3[sB[n * kb + blk]] * inner;",
                                   "acc += g_ue8m0[sA[m * kb + blk]] * g_ue4m3[sB[n * kb + blk]] * inner;"),
    "mx_b32_groups_of_64": ("const int64_t g = n / 32;", "const int64_t g = n / 64;"),
    "mx_b32_b_block_index_dropped": ("g_ue8m0[sB32[g * kb + blk]]", "g_ue8m0[sB32[g * kb]]"),
    "blockscale_b_block_index_dropped": ("(double)sb[(n / 128) * KB + g]", "(double)sb[g]"),
    "blockscale_a_block_index_dropped": ("(double)sa[m * KB + g]", "(double)sa[m * KB]"),
    "blockscale_bias_dropped": ("if (bias) acc += (double)qko_bf16_to_f32(bias[n]);\n      ref[(m - m0) * ldr + (n - n0)] = acc;\n    }\n  }\n  return QKO_OK;\n}\n\n/* Number",
                                "(void)bias;\n      ref[(m - m0) * ldr + (n - n0)] = acc;\n    }\n  }\n  return QKO_OK;\n}\n\n/* Number"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="qk_oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    msrc = os.path.join(mutant_dir, f"{name}.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib_path = os.path.join(mutant_dir, f"lib{name}.so")
    import subprocess
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c99", "-shared", "-fPIC",
                    "-o", lib_path, msrc, "-lm"], check=True)
    lib = oracle.load(lib_path)
    failures = []
    for check in ALL_CHECKS:
        try:
            check(lib)
        except (AssertionError, ValueError):
            failures.append(check.__name__)
    assert failures, f"mutant {name} passed every pin"
