"""The oracle's pins must catch plausible mistakes.

Each mutant below plants one such mistake (a dropped term, a wrong sign, a
wrong index, a transposed operand, a wrong leading dimension, a decoder
slip) into a private copy of the oracle's C source, compiles it, and
requires at least one pin from ``oracle_pins`` to fail on it.  The real
oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle.oracle as oracle
from tests import oracle_pins

MUTANTS = {
    "transA_ignored": ("int64_t idx = p->transA ? k * p->lda + i : i * p->lda + k;",
                       "int64_t idx = p->transA ? i * p->lda + k : i * p->lda + k;"),
    "transB_swapped": ("int64_t idx = p->transB ? j * p->ldb + k : k * p->ldb + j;",
                       "int64_t idx = p->transB ? k * p->ldb + j : j * p->ldb + k;"),
    "lda_replaced_by_K": ("i * p->lda + k;", "i * p->K + k;"),
    "ldc_replaced_by_N": ("int64_t off = i * p->ldc + j;", "int64_t off = i * p->N + j;"),
    "beta_dropped": ("d += p->beta * c;", "d += c;"),
    "beta0_reads_C": ("if (p->beta != 0.0) {             /* beta == 0: C is not read */",
                      "if (1) {"),
    "alpha_dropped": ("double d = p->alpha * s;", "double d = s;"),
    "last_k_dropped": ("for (int64_t k = 0; k < p->K; ++k) {", "for (int64_t k = 0; k + 1 < p->K; ++k) {"),
    "first_k_dropped": ("for (int64_t k = 0; k < p->K; ++k) {", "for (int64_t k = 1; k < p->K; ++k) {"),
    "sign_of_product": ("double prod = a_hat(p, i, k) * b_hat(p, k, j);",
                        "double prod = fabs(a_hat(p, i, k)) * b_hat(p, k, j);"),
    "output_transposed": ("D[i * ldo + j] = one_element(p, i, j, &bound[i * ldo + j]);",
                          "D[i * ldo + j] = one_element(p, j % p->M, i % p->N, &bound[i * ldo + j]);"),
    "f16_exponent_bias": ("v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "bf16_subnormal_scale": ("v = ldexp((double)f, -133);", "v = ldexp((double)f, -126);"),
    "f16_sign_lost": ("    return sign ? -v : v;\n}\n\n/* bfloat16",
                      "    return v;\n}\n\n/* bfloat16"),
    "bound_abs_missing": ("sa += fabs(prod);", "sa += prod;"),
    "bound_beta_missing": ("b += fabs(p->beta) * fabs(c);", "b += 0.0;"),
    "c16_decoded_as_bf16": ("return p->c_dtype == ORACLE_F16 ? oracle_decode_f16(bits) : oracle_decode_bf16(bits);",
                            "return oracle_decode_bf16(bits);"),
    "ld_check_missing": ("if (K > 0 && lda < (transA ? M : K)) return -1;", ""),
    "e4m3_nan_missing": ("if (e == 15 && f == 7)\n        v = NAN;", "if (0)\n        v = NAN;"),
    "e4m3_exponent_bias": ("v = ldexp((double)(8 + f), e - 10);", "v = ldexp((double)(8 + f), e - 9);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "e5m2_subnormal_scale": ("v = ldexp((double)f, -16);", "v = ldexp((double)f, -15);"),
    "e5m2_no_infinity": ("v = (f == 0) ? INFINITY : NAN;\n    else\n        v = ldexp((double)(4 + f), e - 17);",
                         "v = ldexp((double)(4 + f), e - 17);\n    else\n        v = ldexp((double)(4 + f), e - 17);"),
    "fp8_read_as_16bit": ("return p->in_bytes == 1 ?", "return p->in_bytes == 0 ?"),
    "fp8_table_swapped": ("case ORACLE_E4M3: return g_e4m3_table;", "case ORACLE_E4M3: return g_e5m2_table;"),
    "mx_sfa_block_16": ("p->SFA[i * p->ld_sfa + k / MX_BLOCK]", "p->SFA[i * p->ld_sfa + k / 16]"),
    "mx_sfb_block_64": ("p->SFB[j * p->ld_sfb + k / MX_BLOCK]", "p->SFB[j * p->ld_sfb + k / 64]"),
    "mx_sfa_row_stride_of_sfb": ("p->SFA[i * p->ld_sfa + k / MX_BLOCK]", "p->SFA[i * p->ld_sfb + k / MX_BLOCK]"),
    "mx_sfb_dropped": ("if (p->SFB != NULL) v *=", "if (0) v *="),
    "mx_scale_bias_128": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 128)"),
    "mx_nan_scale_missing": ("e == 0xFFu ? NAN :", "0 ? NAN :"),
    "mx_scale_row_check_missing": ("if (p->K > 0 && (ld_sfa < kb || ld_sfb < kb)) return -1;", ""),
    "mx_16bit_accepted": ("if (p->in_bytes > 1) return -1;", ""),
    "e2m1_exponent_bias": ("v = ldexp((double)(2 + f), e - 2);", "v = ldexp((double)(2 + f), e - 1);"),
    "e2m1_subnormal_dropped": ("v = 0.5 * f;", "v = 0.0 * f;"),
    "e2m1_nibbles_swapped": ("return (idx % 2 == 0) ? (b & 0xFu) : (b >> 4);",
                             "return (idx % 2 == 0) ? (b >> 4) : (b & 0xFu);"),
    "e2m1_byte_index": ("const uint8_t b = ((const uint8_t*)X)[idx / 2];",
                        "const uint8_t b = ((const uint8_t*)X)[idx / 2 + (idx % 4 == 3)];"),
    "entries_use_col_as_row": ("D[e] = one_element(p, rows[e], cols[e], &bound[e]);",
                               "D[e] = one_element(p, rows[e], cols[e] % (p->N > 1 ? p->N - 1 : 1), &bound[e]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, "mutation site not found exactly once: %r" % old
    src = tmp_path / ("oracle_%s.c" % name)
    src.write_text(source.replace(old, new))
    lib = oracle.compile_library(str(src), str(tmp_path / ("liboracle_%s.so" % name)))
    # A mutant may read out of bounds and crash: run its pins in a child
    # process, where a crash also counts as caught.
    proc = subprocess.run([sys.executable, "-c", _CHILD, lib], cwd=_ROOT,
                          capture_output=True, text=True, timeout=600)
    caught = proc.returncode != 0 or "CAUGHT" in proc.stdout
    assert caught, "mutant %s passed every pin:\n%s%s" % (name, proc.stdout, proc.stderr)


_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_CHILD = """
import sys
import oracle.oracle as oracle
from tests import oracle_pins
orc = oracle.Oracle(sys.argv[1])
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except (AssertionError, ValueError) as e:
        print("CAUGHT", pin.__name__, e)
        sys.exit(0)
"""
