"""Plant one mistake at a time in a copy of the oracle (on the CPU) and check
that the pins catch it.

Each mutant (all of them stay in bounds) is a textual edit of oracle.c compiled into a temporary library;
the pin tests of test_oracle_pins.py then run against it and at least one must
fail.  This shows the pins are sensitive to the plausible mistakes: a dropped
term, a wrong sign, a wrong index, a transposed operand, a swapped nibble order
a wrong binary16 exponent or subnormal scale, and, in the scaled epilogue,
truncating or ties-away 16-bit rounding, a missing overflow, swapped scale
order and a missing 32-bit wrap.
"""
import os
import subprocess
import sys

import pytest

import oracle
from tests import test_oracle_dequant as dq
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTANTS = [
    ("f16_bias", "ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    ("f16_subnormal_scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("f16_sign_dropped", "return s ? -v : v;", "return v;"),
    ("f16_B_transposed",
     "oracle_f16_to_f64(A[i * lda + k]) * oracle_f16_to_f64(B[k * ldb + j])",
     "oracle_f16_to_f64(A[i * lda + k]) * oracle_f16_to_f64(B[j * ldb + k])"),
    ("f16_last_term_dropped",
     "    for (int64_t k = 0; k < K; ++k) {\n        /* an 11-bit",
     "    for (int64_t k = 0; k + 1 < K; ++k) {\n        /* an 11-bit"),
    ("f16_abs_sum_signed", "sabs += fabs(p);", "sabs += p;"),
    ("s8_B_transposed", "(int64_t)B[j * ldb + k]", "(int64_t)B[k * ldb + j]"),
    ("s8_first_term_dropped",
     "    for (int64_t k = 0; k < K; ++k)\n        acc += (int64_t)A[i * lda + k]",
     "    for (int64_t k = 1; k < K; ++k)\n        acc += (int64_t)A[i * lda + k]"),
    ("s8_A_k_reversed", "(int64_t)A[i * lda + k] * (int64_t)B",
     "(int64_t)A[i * lda + (K - 1 - k)] * (int64_t)B"),
    ("s4_nibble_order", "int nib = (k & 1) ? (byte >> 4) : (byte & 0x0f);",
     "int nib = (k & 1) ? (byte & 0x0f) : (byte >> 4);"),
    ("s4_unsigned", "return nib >= 8 ? nib - 16 : nib;", "return nib;"),
    ("s4_sign_threshold", "return nib >= 8 ? nib - 16 : nib;", "return nib > 8 ? nib - 16 : nib;"),
    ("s4_row_off_by_one", "const uint8_t *arow = A + i * (lda / 2);",
     "const uint8_t *arow = A + (i > 0 ? i - 1 : 0) * (lda / 2);"),
    ("rows_skipped_by_threads", "jobs[t].r0 = t * per;", "jobs[t].r0 = t * per + (t > 0);"),
    ("bf16_truncates", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))", "if (0)"),
    ("bf16_ties_away", "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))",
     "if (rest >= 0x8000u)"),
    ("f16_subnormal_quantum", "double q = nearbyint(a * ldexp(1.0, 24));",
     "double q = nearbyint(a * ldexp(1.0, 23));"),
    ("f16_no_overflow", "if (e > 15) return (uint16_t)(sign | 0x7c00u);", "if (e > 16) return (uint16_t)(sign | 0x7c00u);"),
    ("dequant_scales_swapped", "t = t * (sa ? sa[i] : 1.0f);\n            t = t * (sb ? sb[j] : 1.0f);",
     "t = t * (sb ? sb[j] : 1.0f);\n            t = t * (sa ? sa[i] : 1.0f);"),
    ("dequant_no_wrap", "int32_t v = (int32_t)(uint32_t)(uint64_t)acc[i * lda + j];",
     "int64_t v = acc[i * lda + j];"),
]

PIN_CALLS = [
    lambda g: pins.test_f16_decode_exhaustive(),
    lambda g: pins.test_mma_lab_worked_example(g),
    lambda g: pins.test_identity_and_permutation_f16(5, 7, 5),
    lambda g: pins.test_identity_and_permutation_f16(16, 24, 16),
    lambda g: pins.test_identity_and_permutation_s8_s4(5, 7, 6),
    lambda g: pins.test_identity_and_permutation_s8_s4(16, 24, 16),
    lambda g: pins.test_all_ones_and_extremes(17),
    lambda g: pins.test_all_ones_and_extremes(256),
    lambda g: pins.test_rank_one(),
    lambda g: pins.test_cancellation_adversary_s8(),
    lambda g: pins.test_s4_nibble_order_and_roundtrip(),
    lambda g: pins.test_brute_force_int(7, 9, 11),
    lambda g: pins.test_brute_force_f16_fraction(7, 9, 11),
    lambda g: dq.test_bf16_rounding_against_torch(),
    lambda g: dq.test_f16_rounding_against_numpy(),
    lambda g: dq.test_dequant_matches_exact_stepwise_rounding(),
    lambda g: dq.test_dequant_order_matters_and_is_a_then_b(),
    lambda g: dq.test_dequant_identity_scales(),
]


CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import test_oracle_mutants as tm
with oracle.swapped_library({so!r}):
    for i, call in enumerate(tm.PIN_CALLS):
        try:
            call({golden!r})
        except AssertionError:
            print("caught-by", i)
            sys.exit(0)
print("not-caught")
sys.exit(3)
"""


@pytest.fixture(scope="module")
def oracle_src():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, oracle_src, tmp_path, golden_dir):
    """Pins run in order in a child process and stop at the first one that
    fails; some mutants would read out of bounds on pins further down."""
    assert oracle_src.count(old) == 1, f"mutation site for {name} not unique/found"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(oracle_src.replace(old, new))
    so = tmp_path / f"liboracle_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", str(src), "-o", str(so), "-lm"])
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = CHILD.format(root=root, so=str(so), golden=str(golden_dir))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "caught-by" in r.stdout, \
        f"planted mistake {name} not caught: rc={r.returncode} {r.stdout[-300:]} {r.stderr[-300:]}"
