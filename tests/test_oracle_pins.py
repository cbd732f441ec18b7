"""Pins for the CPU oracle: each test ties it to something other than itself.

What each pin rests on:
* the decode table printed on the pages (formula and prmt table),
* hand-computed 2x2 and 4x8 products (tests/golden/hand_cases.txt),
* closed forms and the int32 extremes, including the pages' bound of 131071
  rows for an int8 x int8 reduction,
* numpy's exact int64 matmul on the generator's own ternary matrix (never the
  oracle's unpack), for forward, dX and dW, ragged shapes included,
* brute force over every ternary W with K*N <= 8,
* invariants: linearity, dX as a forward on the transposed weights.
"""
import itertools

import numpy as np
import pytest

import oracle
import t3_synth
from conftest import read_golden


def _table_from_golden():
    lines = read_golden("decode_table.txt")
    word = int(lines[0][1], 16)
    table = {int(c): int(v) for c, v in lines[1:]}
    return word, table


# ---------------------------------------------------------------- decode ----

def test_decode_table_matches_both_printed_forms():
    word, table = _table_from_golden()
    # the printed prmt table: byte c of 0x00FF0100 read as int8 is the weight
    prmt_bytes = [(word >> (8 * c)) & 0xFF for c in range(4)]
    as_int8 = [b - 256 if b >= 128 else b for b in prmt_bytes]
    # the printed formula, evaluated bit by bit
    formula = [(c & 1) - ((c >> 1) & 1) for c in range(4)]
    for c in range(4):
        assert oracle.decode(c) == table[c] == as_int8[c] == formula[c]


def test_unpack_every_byte_value():
    """All 256 byte values: the 4 weights of each byte come out at bits 2j."""
    _, table = _table_from_golden()
    wp = np.arange(256, dtype=np.uint8).reshape(256, 1)  # N=256 rows, K=4
    w = oracle.unpack(wp, 4)
    for b in range(256):
        for j in range(4):
            assert w[j, b] == table[(b >> (2 * j)) & 3]


# ------------------------------------------------------------------ pack ----

def test_pack_all_81_tuples_round_trip_and_bytes():
    tuples = np.array(list(itertools.product([-1, 0, 1], repeat=4)), dtype=np.int8)  # 81x4
    w = np.ascontiguousarray(tuples.T)  # K=4, N=81
    wp = oracle.pack(w)
    assert wp.shape == (81, 1)
    code = {0: 0, 1: 1, -1: 2}
    for n in range(81):
        expect = sum(code[int(w[k, n])] << (2 * k) for k in range(4))
        assert wp[n, 0] == expect
    assert np.array_equal(oracle.unpack(wp, 4), w)


@pytest.mark.parametrize("K", list(range(1, 14)))
def test_pack_round_trip_every_k_mod_4(K):
    g = t3_synth.rng(100 + K)
    N = 7
    w = t3_synth.ternary(g, (K, N))
    wp = oracle.pack(w)
    assert wp.shape == (N, (K + 3) // 4)
    assert np.array_equal(oracle.unpack(wp, K), w)
    # pad positions k >= K of the last byte hold code 0
    if K % 4:
        pad_mask = 0xFF & ~((1 << (2 * (K % 4))) - 1)
        assert np.all(wp[:, -1] & pad_mask == 0)


def test_pack_rejects_non_ternary_and_writes_nothing():
    w = np.zeros((5, 3), dtype=np.int8)
    w[2, 1] = 2
    assert oracle.pack_status(w) == oracle.EVALUE
    w[2, 1] = -128
    assert oracle.pack_status(w) == oracle.EVALUE


def test_pack_hand_bytes_2x2_and_4x8():
    w22 = np.array([[1, -1], [0, 1]], dtype=np.int8)
    assert oracle.pack(w22).tolist() == [[0x01], [0x06]]
    w48 = _w_4x8()
    assert oracle.pack(w48).tolist() == [[0x55, 0x55], [0x99, 0x99], [0x00, 0x80], [0x00, 0x55]]


# ------------------------------------------------------------ hand cases ----

def _w_4x8():
    w = np.zeros((8, 4), dtype=np.int8)
    w[:, 0] = 1
    w[0::2, 1] = 1
    w[1::2, 1] = -1
    w[7, 2] = -1
    w[4:, 3] = 1
    return w


def test_hand_case_2x2():
    A = np.array([[1, 2], [3, 4]], dtype=np.int8)
    wp = np.array([[0x01], [0x06]], dtype=np.uint8)  # packed by hand
    assert oracle.fwd(A, wp).tolist() == [[1, 1], [3, 1]]
    assert oracle.dx(A, wp, 2).tolist() == [[-1, 2], [-1, 4]]
    dY = np.array([[5, 6], [7, 8]], dtype=np.int8)
    assert oracle.dw(A, dY).tolist() == [[26, 30], [38, 44]]


def test_hand_case_4x8():
    A = np.array([[1, 2, 3, 4, 5, 6, 7, 8],
                  [-1] * 8,
                  [127, -128, 0, 0, 0, 0, 0, 0],
                  [0, 0, 0, 0, 0, 0, 0, 1]], dtype=np.int8)
    wp = np.array([[0x55, 0x55], [0x99, 0x99], [0x00, 0x80], [0x00, 0x55]], dtype=np.uint8)
    assert oracle.fwd(A, wp).tolist() == [[36, -4, -8, 26],
                                          [-8, 0, 1, -4],
                                          [-1, 255, 0, 0],
                                          [1, -1, -1, 1]]


# ------------------------------------------------------------ closed forms --

@pytest.mark.parametrize("a", [-128, -1, 1, 127])
@pytest.mark.parametrize("K", [1, 5, 96, 1000])
def test_constant_inputs(a, K):
    M, N = 3, 5
    A = np.full((M, K), a, dtype=np.int8)
    plus = oracle.pack(np.ones((K, N), dtype=np.int8))
    minus = oracle.pack(-np.ones((K, N), dtype=np.int8))
    assert np.all(oracle.fwd(A, plus) == a * K)
    assert np.all(oracle.fwd(A, minus) == -a * K)
    # dX reduces over N: dY = a everywhere, W = +1 -> a*N
    dY = np.full((M, N), a, dtype=np.int8)
    assert np.all(oracle.dx(dY, plus, K) == a * N)
    assert np.all(oracle.dx(dY, minus, K) == -a * N)


def test_identity_weight_gives_a():
    g = t3_synth.rng(7)
    K = 37
    A = t3_synth.int8_uniform(g, (9, K))
    eye = oracle.pack(np.eye(K, dtype=np.int8))
    assert np.array_equal(oracle.fwd(A, eye), A.astype(np.int32))
    assert np.array_equal(oracle.dx(A, eye, K), A.astype(np.int32))


def test_int32_extremes():
    K = 8192
    A = np.full((2, K), -128, dtype=np.int8)
    assert np.all(oracle.fwd(A, oracle.pack(-np.ones((K, 3), dtype=np.int8))) == 128 * K)
    assert np.all(oracle.fwd(A, oracle.pack(np.ones((K, 3), dtype=np.int8))) == -128 * K)
    # int8 x int8: the pages bound the reduction at 131071 rows; at that length
    # (-128)*(-128)*131071 = 2147467264 still fits in int32, one more row does not.
    M = 131071
    A1 = np.full((M, 1), -128, dtype=np.int8)
    assert oracle.dw(A1, A1).tolist() == [[16384 * M]]
    A2 = np.full((M + 1, 1), -128, dtype=np.int8)
    with pytest.raises(oracle.OracleError):
        oracle.dw(A2, A2)


# ---------------------------------------------------- library routine -------

SHAPES = [(1, 1, 1), (3, 5, 7), (300, 272, 96), (17, 33, 130), (64, 64, 64), (5, 129, 255)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_against_numpy_matmul(M, N, K):
    g = t3_synth.rng(M * 1000 + N * 10 + K)
    A = t3_synth.int8_uniform(g, (M, K))
    w = t3_synth.ternary(g, (K, N))
    dY = t3_synth.int8_uniform(g, (M, N))
    wp = oracle.pack(w)
    A64, w64, dY64 = A.astype(np.int64), w.astype(np.int64), dY.astype(np.int64)
    assert np.array_equal(oracle.fwd(A, wp), A64 @ w64)
    assert np.array_equal(oracle.dx(dY, wp, K), dY64 @ w64.T)
    assert np.array_equal(oracle.dw(A, dY), A64.T @ dY64)


def test_raw_bytes_code3_and_pad_bits_ignored():
    """Random raw Wp (every code including 3, nonzero pad bits) against numpy on
    the golden decode table."""
    _, table = _table_from_golden()
    lut = np.array([table[c] for c in range(4)], dtype=np.int64)
    g = t3_synth.rng(11)
    for (M, N, K) in [(4, 9, 1), (6, 5, 10), (33, 31, 97), (8, 64, 255)]:
        KB = (K + 3) // 4
        raw = t3_synth.raw_bytes(g, (N, KB))
        A = t3_synth.int8_uniform(g, (M, K))
        dY = t3_synth.int8_uniform(g, (M, N))
        k = np.arange(K)
        codes = (raw[:, k // 4].astype(np.int64) >> (2 * (k % 4))) & 3  # [N][K]
        W = lut[codes].T  # [K][N]
        assert np.array_equal(oracle.fwd(A, raw), A.astype(np.int64) @ W)
        assert np.array_equal(oracle.dx(dY, raw, K), dY.astype(np.int64) @ W.T)


def test_rows_subset_matches_full():
    g = t3_synth.rng(5)
    M, N, K = 40, 23, 50
    A = t3_synth.int8_uniform(g, (M, K))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    dY = t3_synth.int8_uniform(g, (M, N))
    rows = np.array([39, 0, 17, 17, 5])
    assert np.array_equal(oracle.fwd(A, wp, rows), oracle.fwd(A, wp)[rows])
    assert np.array_equal(oracle.dx(dY, wp, K, rows), oracle.dx(dY, wp, K)[rows])
    krows = np.array([49, 0, 3])
    assert np.array_equal(oracle.dw(A, dY, krows), oracle.dw(A, dY)[krows])


# ----------------------------------------------------------- brute force ----

@pytest.mark.parametrize("K,N", [(1, 8), (2, 4), (4, 2), (8, 1)])
def test_brute_force_every_ternary_w(K, N):
    g = t3_synth.rng(K * 10 + N)
    M = 3
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    for vals in itertools.product([-1, 0, 1], repeat=K * N):
        w = np.array(vals, dtype=np.int8).reshape(K, N)
        wp = oracle.pack(w)
        C = oracle.fwd(A, wp)
        dX = oracle.dx(dY, wp, K)
        for m in range(M):
            for n in range(N):
                assert C[m, n] == sum(int(A[m, k]) * int(w[k, n]) for k in range(K))
            for k in range(K):
                assert dX[m, k] == sum(int(dY[m, n]) * int(w[k, n]) for n in range(N))


# ------------------------------------------------------------ invariants ----

def test_linearity_in_a():
    g = t3_synth.rng(21)
    M, N, K = 11, 13, 70
    A1 = g.integers(-64, 64, size=(M, K)).astype(np.int8)
    A2 = g.integers(-64, 64, size=(M, K)).astype(np.int8)
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    s = (A1.astype(np.int16) + A2).astype(np.int8)
    assert np.array_equal(oracle.fwd(s, wp), oracle.fwd(A1, wp) + oracle.fwd(A2, wp))


def test_dx_is_forward_on_transposed_weights():
    g = t3_synth.rng(22)
    M, N, K = 9, 30, 21
    w = t3_synth.ternary(g, (K, N))
    dY = t3_synth.int8_uniform(g, (M, N))
    wpT = oracle.pack(np.ascontiguousarray(w.T))  # a forward weight of shape [N][K]
    assert np.array_equal(oracle.dx(dY, oracle.pack(w), K), oracle.fwd(dY, wpT))


def test_dw_swaps_with_transposes():
    g = t3_synth.rng(23)
    M, N, K = 12, 7, 5
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    assert np.array_equal(oracle.dw(A, dY).T, oracle.dw(dY, A))


# ---------------------------------------------------------------- scaled outputs
# The scaled outputs restate a definition (float32 steps, bf16 rounding to
# nearest even); these pins check the oracle's numpy arithmetic against
# independent computations: torch's own bf16 conversion, and exact rational
# arithmetic rounded once per step.

def _f32_round(q) -> np.float32:
    """Nearest float32 (ties to even) of an exact rational whose float64
    value is exact (every case below keeps it so)."""
    return np.float32(float(q))


def test_bf16_rounding_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(5)
    y = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(1e3),
        # exact ties: a bf16 value plus half of its last place, both parities
        (np.arange(1, 513, dtype=np.float32) * np.float32(2.0 ** -7) + np.float32(1.0)
         + np.float32(2.0 ** -9)),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, 65504.0], dtype=np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_bits(y), ref)


def test_bf16_rounding_hand_values():
    # 1 + 2^-8 lies halfway between bf16 1.0 (0x3F80) and 1 + 2^-7: ties to even
    y = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 1.0 + 2.0 ** -8 + 2.0 ** -20],
                 dtype=np.float32)
    assert list(oracle.bf16_bits(y)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]


def test_dequant_steps_match_exact_rationals():
    from fractions import Fraction
    g = np.random.default_rng(6)
    rows, cols = 7, 9
    x = g.integers(-2 ** 31, 2 ** 31, (rows, cols), dtype=np.int64).astype(np.int32)
    x[0, :4] = [16777217, -16777219, 2 ** 24 + 3, 0]  # conversions that must round
    rs = (g.standard_normal(rows) * 3).astype(np.float32)
    cs = (g.standard_normal(cols) / 7).astype(np.float32)
    old = (g.standard_normal((rows, cols)) * 1e6).astype(np.float32)
    y = oracle.dequant(x, rs, cs)
    add = oracle.dequant(x, rs, cs, oracle.OUT_F32_ADD, old)
    for r in range(rows):
        for c in range(cols):
            xf = _f32_round(Fraction(int(x[r, c])))
            t = _f32_round(Fraction(float(xf)) * Fraction(float(rs[r])))
            want = _f32_round(Fraction(float(t)) * Fraction(float(cs[c])))
            if want == 0:  # rationals have no signed zero: IEEE gives the product of the signs
                want = np.float32(-0.0) if (np.signbit(xf) ^ np.signbit(rs[r]) ^ np.signbit(cs[c])) \
                    else np.float32(0.0)
            assert y[r, c] == want and np.signbit(y[r, c]) == np.signbit(want)
            assert add[r, c] == _f32_round(Fraction(float(old[r, c])) + Fraction(float(want)))


def test_dequant_special_cases():
    x = np.array([[0, 5, -7, 2 ** 24 + 1]], dtype=np.int32)
    # no scales: the nearest float of x
    np.testing.assert_array_equal(oracle.dequant(x), np.array([[0, 5, -7, 2 ** 24]], np.float32))
    # a negative scale turns 0 into -0.0
    z = oracle.dequant(x, np.array([-1.0], np.float32))
    assert z[0, 0] == 0.0 and np.signbit(z[0, 0])
    # "+=" with an old value of 0 is the plain output; bf16 of small integers is exact
    old = np.zeros((1, 4), np.float32)
    np.testing.assert_array_equal(oracle.dequant(x, kind=oracle.OUT_F32_ADD, out=old), oracle.dequant(x))
    b = oracle.dequant(np.array([[1, -2, 128]], np.int32), kind=oracle.OUT_BF16)
    assert list(b[0]) == [0x3F80, 0xC000, 0x4300]


# ------------------------------------------------------------ row quantizer

def _bf16(values):
    return (np.asarray(values, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _f32_nearest_even(q):
    """The float32 nearest to the rational q (ties to even), by integer
    arithmetic on the exact value; normal range."""
    from fractions import Fraction
    if q == 0:
        return np.float32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(Fraction(q))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if a >= Fraction(2) ** e:   # now 2^e <= a < 2^(e+1)
        pass
    else:
        e -= 1
    scaled = a / Fraction(2) ** (e - 23)   # in [2^23, 2^24)
    m, rem = divmod(scaled.numerator, scaled.denominator)
    twice = 2 * rem
    if twice > scaled.denominator or (twice == scaled.denominator and m % 2 == 1):
        m += 1
    return np.float32(sign * float(Fraction(m) * Fraction(2) ** (e - 23)))


def test_quantize_rows_hand_values_and_ties():
    q, s = oracle.quantize_rows(np.stack([_bf16([1, -2, 0.5, 127]), _bf16([0, 0, 0, 0]),
                                          _bf16([0.75, 1.5, 2.5, -127])]))
    assert q.tolist() == [[1, -2, 0, 127], [0, 0, 0, 0], [1, 2, 2, -127]]
    assert s.tolist() == [1.0, 0.0, 1.0]


def test_quantize_rows_against_exact_rationals():
    from fractions import Fraction
    g = np.random.default_rng(11)
    x = (g.standard_normal((12, 37)) * np.float32(10.0) ** g.integers(-3, 4, (12, 1))).astype(np.float32)
    bits = _bf16(x)
    q, s = oracle.quantize_rows(bits)
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    for m in range(12):
        amax = max(abs(float(v)) for v in xf[m])
        assert s[m] == _f32_nearest_even(Fraction(amax) / 127)
        inv = _f32_nearest_even(Fraction(127) / Fraction(amax))
        for k in range(37):
            prod = _f32_nearest_even(Fraction(float(xf[m, k])) * Fraction(float(inv)))
            fl = Fraction(float(prod))
            r = round(fl)  # Python rounds halves to even
            assert q[m, k] == max(-127, min(127, r))


def _exact_chain_q(xf, amax):
    from fractions import Fraction
    inv = _f32_nearest_even(Fraction(127) / Fraction(amax))
    prod = _f32_nearest_even(Fraction(xf) * Fraction(float(inv)))
    return max(-127, min(127, round(Fraction(float(prod)))))


def test_quantize_rows_float32_rounding_of_the_product():
    # x = amax / 2: the exact product is 63.5, and the float32 roundings of
    # 127 / amax and of x * inv decide between 63 and 64 (found by search)
    pairs = [(0.00982666015625, 0.0196533203125), (0.0128173828125, 0.025634765625),
             (0.01409912109375, 0.0281982421875), (0.0279541015625, 0.055908203125),
             (0.048583984375, 0.09716796875), (0.05029296875, 0.1005859375)]
    q, _ = oracle.quantize_rows(np.stack([_bf16([x, amax]) for x, amax in pairs]))
    assert [int(v) for v in q[:, 0]] == [_exact_chain_q(x, amax) for x, amax in pairs]
    assert sorted(set(int(v) for v in q[:, 0])) == [63, 64]


def test_quantize_rows_properties():
    g = np.random.default_rng(12)
    x = (g.standard_normal((64, 300)) * 3).astype(np.float32)
    bits = _bf16(x)
    q, s = oracle.quantize_rows(bits)
    xf = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.abs(q.astype(int)).max() <= 127
    am = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(64), am]) == 127)       # the row's maximum maps to +-127
    err = np.abs(q * s[:, None].astype(np.float64) - xf)
    assert np.all(err <= s[:, None] * 0.5 * (1 + 1e-5))       # half a step, plus float slack


# ------------------------------------------- the quantized chain against f64 --
# Quantize, take the exact integer product, dequantize: the result must stay
# within the quantization error of the f64 product of the original values
# (the pages bounded their quantized backward against an f64 reference).  Each
# element of a row quantized with scale s is off by at most s / 2 (plus a few
# float32 ulps of |x|); the dequantization adds a few ulps of the result.

def _bf16_matrix(g, shape, spread=True):
    mag = np.float32(2.0) ** g.integers(-6, 7, (shape[0], 1)).astype(np.float32) if spread else 1.0
    x = (g.standard_normal(shape) * mag).astype(np.float32)
    bits = oracle.bf16_bits(x)
    return bits, (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulps(v):
    return 4.0 * np.finfo(np.float32).eps * v


def test_quantized_forward_within_f64_bound():
    g = t3_synth.rng(4101)
    M, K, N = 48, 320, 40
    bits, x = _bf16_matrix(g, (M, K))
    w = t3_synth.ternary(g, (K, N))
    q, s = oracle.quantize_rows(bits)
    y = oracle.dequant(oracle.fwd(q, oracle.pack(w)), s, None).astype(np.float64)
    wf = w.astype(np.float64)
    truth = x @ wf
    bound = (s.astype(np.float64)[:, None] / 2) * (np.abs(wf).sum(0)[None, :]) \
        + _ulps(np.abs(x) @ np.abs(wf)) + _ulps(np.abs(truth))
    err = np.abs(y - truth)
    assert np.all(err <= bound)
    assert err.max() > 0  # the bound is not met trivially


def test_quantized_dx_within_f64_bound():
    g = t3_synth.rng(4102)
    M, N, K = 40, 288, 56
    bits, dy = _bf16_matrix(g, (M, N))
    w = t3_synth.ternary(g, (K, N))
    q, s = oracle.quantize_rows(bits)
    y = oracle.dequant(oracle.dx(q, oracle.pack(w), K), s, None).astype(np.float64)
    wf = w.astype(np.float64)
    truth = dy @ wf.T
    bound = (s.astype(np.float64)[:, None] / 2) * (np.abs(wf).sum(1)[None, :]) \
        + _ulps(np.abs(dy) @ np.abs(wf.T)) + _ulps(np.abs(truth))
    err = np.abs(y - truth)
    assert np.all(err <= bound)
    assert err.max() > 0


def test_quantized_dw_within_f64_bound():
    """dW with X and dY quantized per column (the scales the pages name for
    dW): dequant(dW(qX, qdY), sX as row scale, sdY as column scale)."""
    g = t3_synth.rng(4103)
    M, K, N = 200, 24, 32
    xb, x = _bf16_matrix(g, (M, K), spread=False)
    yb, dy = _bf16_matrix(g, (M, N), spread=False)
    qxt, sx = oracle.quantize_rows(np.ascontiguousarray(xb.T))
    qyt, sy = oracle.quantize_rows(np.ascontiguousarray(yb.T))
    qx, qy = np.ascontiguousarray(qxt.T), np.ascontiguousarray(qyt.T)
    y = oracle.dequant(oracle.dw(qx, qy), sx, sy).astype(np.float64)
    truth = x.T @ dy
    sxd, syd = sx.astype(np.float64), sy.astype(np.float64)
    # a dy - qa sa qd sd = a ed + ea qd sd, |ea| <= sa/2, |ed| <= sd/2, |qd sd| <= |dy| + sd/2
    bound = np.abs(x).T @ np.ones((M, N)) * (syd[None, :] / 2) \
        + (sxd[:, None] / 2) * (np.ones((K, M)) @ (np.abs(dy) + syd[None, :] / 2)) \
        + _ulps(np.abs(x).T @ np.abs(dy)) + _ulps(np.abs(truth))
    err = np.abs(y - truth)
    assert np.all(err <= bound)
    assert err.max() > 0
