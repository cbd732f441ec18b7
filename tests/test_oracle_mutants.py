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


# ------------------------------------------------ scaled outputs (numpy oracle)
# Plausible mistakes in oracle.dequant / oracle.bf16_bits, swapped in with
# monkeypatch; at least one of the scaled-output pins must fail for each.

def _m_swapped_scale_order(x, row_scale=None, col_scale=None, kind=0, out=None):
    import numpy as np
    x = np.asarray(x, np.int32)
    rows, cols = x.shape
    rs = np.ones(rows, np.float32) if row_scale is None else np.asarray(row_scale, np.float32)
    cs = np.ones(cols, np.float32) if col_scale is None else np.asarray(col_scale, np.float32)
    y = (x.astype(np.float32) * cs[None, :]) * rs[:, None]
    return _finish(y, kind, out)


def _m_one_rounding(x, row_scale=None, col_scale=None, kind=0, out=None):
    import numpy as np
    x = np.asarray(x, np.int32)
    rows, cols = x.shape
    rs = np.ones(rows) if row_scale is None else np.asarray(row_scale, np.float64)
    cs = np.ones(cols) if col_scale is None else np.asarray(col_scale, np.float64)
    y = (x.astype(np.float64) * rs[:, None] * cs[None, :]).astype(np.float32)
    return _finish(y, kind, out)


def _m_add_before_scaling(x, row_scale=None, col_scale=None, kind=0, out=None):
    import numpy as np
    import oracle
    if kind != oracle.OUT_F32_ADD:
        return _ORIG_DEQUANT(x, row_scale, col_scale, kind, out)
    x = np.asarray(x, np.int32)
    rows, cols = x.shape
    rs = np.ones(rows, np.float32) if row_scale is None else np.asarray(row_scale, np.float32)
    cs = np.ones(cols, np.float32) if col_scale is None else np.asarray(col_scale, np.float32)
    return ((np.asarray(out, np.float32) + x.astype(np.float32)) * rs[:, None]) * cs[None, :]


def _m_bf16_truncates(y):
    import numpy as np
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


def _m_bf16_ties_away(y):
    import numpy as np
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x8000) >> 16).astype(np.uint16)


def _finish(y, kind, out):
    import numpy as np
    import oracle
    if kind == oracle.OUT_F32:
        return y
    if kind == oracle.OUT_BF16:
        return oracle.bf16_bits(y)
    return np.asarray(out, np.float32) + y


import oracle as _oracle_mod  # noqa: E402

_ORIG_DEQUANT = _oracle_mod.dequant

SCALED_MUTANTS = {
    "dequant_swapped_scale_order": ("dequant", _m_swapped_scale_order),
    "dequant_one_rounding_in_float64": ("dequant", _m_one_rounding),
    "dequant_adds_before_scaling": ("dequant", _m_add_before_scaling),
    "bf16_truncates": ("bf16_bits", _m_bf16_truncates),
    "bf16_ties_away_from_zero": ("bf16_bits", _m_bf16_ties_away),
}


@pytest.mark.parametrize("name", sorted(SCALED_MUTANTS))
def test_scaled_pins_catch_planted_mistake(name, monkeypatch):
    import test_oracle_pins as pins
    attr, fn = SCALED_MUTANTS[name]
    monkeypatch.setattr(_oracle_mod, attr, fn)
    caught = 0
    for pin in (pins.test_bf16_rounding_matches_torch_conversion, pins.test_bf16_rounding_hand_values,
                pins.test_dequant_steps_match_exact_rationals, pins.test_dequant_special_cases):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no scaled-output pin caught mutant {name}"


def _quant_mutant(ties_away=False, divisor=127.0, inv64=False, lo=-127, hi=127):
    def quantize_rows(x_bits):
        import numpy as np
        u = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = u.shape
        x = (u.astype(np.uint32) << 16).view(np.float32)
        amax = np.abs(x).max(axis=1) if K else np.zeros(M, np.float32)
        pos = amax > 0
        safe = np.where(pos, amax, np.float32(1))
        scale = np.where(pos, safe / np.float32(divisor), 0).astype(np.float32)
        if inv64:
            inv = np.where(pos, 127.0 / safe.astype(np.float64), 0.0)
            prod = (x.astype(np.float64) * inv[:, None])
        else:
            inv = np.where(pos, np.float32(divisor) / safe, 0).astype(np.float32)
            prod = x * inv[:, None]
        r = np.floor(prod + 0.5) if ties_away else np.rint(prod)
        return np.clip(r, lo, hi).astype(np.int8), scale
    return quantize_rows


QUANT_MUTANTS = {
    "quant_ties_rounded_up": _quant_mutant(ties_away=True),
    "quant_divides_by_128": _quant_mutant(divisor=128.0),
    "quant_product_in_float64": _quant_mutant(inv64=True),
    "quant_clamps_to_126": _quant_mutant(lo=-126, hi=126),
}


@pytest.mark.parametrize("name", sorted(QUANT_MUTANTS))
def test_quantizer_pins_catch_planted_mistake(name, monkeypatch):
    import test_oracle_pins as pins
    monkeypatch.setattr(_oracle_mod, "quantize_rows", QUANT_MUTANTS[name])
    caught = 0
    for pin in (pins.test_quantize_rows_hand_values_and_ties, pins.test_quantize_rows_against_exact_rationals,
                pins.test_quantize_rows_float32_rounding_of_the_product,
                pins.test_quantize_rows_properties):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no quantizer pin caught mutant {name}"


def _m_divides_by_scales(x, row_scale=None, col_scale=None, kind=0, out=None):
    import numpy as np
    x = np.asarray(x, np.int32)
    rows, cols = x.shape
    rs = np.ones(rows, np.float32) if row_scale is None else np.asarray(row_scale, np.float32)
    cs = np.ones(cols, np.float32) if col_scale is None else np.asarray(col_scale, np.float32)
    return _finish((x.astype(np.float32) / rs[:, None]) / cs[None, :], kind, out)


def _m_scale_is_amax(x_bits):
    import numpy as np
    q, s = _ORIG_QUANT(x_bits)
    return q, (s * np.float32(127.0)).astype(np.float32)


_ORIG_QUANT = _oracle_mod.quantize_rows

CHAIN_MUTANTS = {
    "dequant_divides_by_scales": ("dequant", _m_divides_by_scales),
    "quant_reports_amax_as_scale": ("quantize_rows", _m_scale_is_amax),
}


@pytest.mark.parametrize("name", sorted(CHAIN_MUTANTS))
def test_chain_pins_catch_planted_mistake(name, monkeypatch):
    """The f64-bound pins of quantize -> product -> dequantize catch mistakes
    in what the chain means, on their own."""
    import test_oracle_pins as pins
    attr, fn = CHAIN_MUTANTS[name]
    monkeypatch.setattr(_oracle_mod, attr, fn)
    caught = 0
    for pin in (pins.test_quantized_forward_within_f64_bound, pins.test_quantized_dx_within_f64_bound,
                pins.test_quantized_dw_within_f64_bound):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught == 3, f"the chain pins caught mutant {name} {caught} times of 3"
