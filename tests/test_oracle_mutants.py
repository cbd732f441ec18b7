"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/t3_oracle.c (on the CPU, in a
temporary directory), builds it, and runs the pin suite against that copy in a
child process.  The suite must fail for every planted mistake: a dropped term,
a wrong sign, a wrong bit order, a transposed or shifted index, a missing
overflow check.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "t3_oracle.c")

MUTANTS = {
    "decode_sign_swapped": ("{0, +1, -1, 0}", "{0, -1, +1, 0}"),
    "code3_decodes_to_plus1": ("{0, +1, -1, 0}", "{0, +1, -1, +1}"),
    "bit_order_reversed": ("(byte >> (2 * (k % 4))) & 3", "(byte >> (2 * (3 - k % 4))) & 3"),
    "fwd_drops_last_term": ("for (int64_t k = 0; k < K; ++k)\n        acc += (int64_t)A[m * K + k]",
                            "for (int64_t k = 0; k + 1 < K; ++k)\n        acc += (int64_t)A[m * K + k]"),
    "dx_reversed_k": ("(int64_t)dY[m * N + n] * (int64_t)weight_of(Wp, K, n, k)",
                      "(int64_t)dY[m * N + n] * (int64_t)weight_of(Wp, K, n, K - 1 - k)"),
    "dw_wrong_column": ("(int64_t)A[m * K + k] * (int64_t)dY[m * N + n]",
                        "(int64_t)A[m * K + k] * (int64_t)dY[m * N + (N - 1 - n)]"),
    "dw_drops_first_row": ("for (int64_t m = 0; m < M; ++m)\n        acc += (int64_t)A[m * K + k] * (int64_t)dY",
                           "for (int64_t m = 1; m < M; ++m)\n        acc += (int64_t)A[m * K + k] * (int64_t)dY"),
    "pack_minus1_as_code3": ("(v == -1) ? 2 : 0", "(v == -1) ? 3 : 0"),
    "no_overflow_check": ("      if (!fits_i32(acc)) bad |= 2;\n      dW[i * N + n]", "      dW[i * N + n]"),
    "dx_transposed_weight_index": ("(int64_t)dY[m * N + n] * (int64_t)weight_of(Wp, K, n, k)",
                                   "(int64_t)dY[m * N + n] * (int64_t)weight_of(Wp, K, k % N, n % K)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(text.replace(old, new, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(mutant_src)],
                   check=True, capture_output=True)
    env = dict(os.environ, T3_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
