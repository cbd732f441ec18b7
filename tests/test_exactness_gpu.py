"""GPU parity at the exactness limits of the tensor-core accumulators.

The products reach exact int32 results through f16 (fwd, dX, dW) tensor-core
operands summed in f32.  An f32 sum of integers is exact while every partial
sum stays below 2^24 in magnitude, so the library cuts each reduction into
chunks that cannot pass that bound (65536 terms of |a w| <= 128 for the
ternary products, 1024 rows of |a dy| <= 16384 for dW) and adds the chunks in
int32.  That is exact only if the tensor core keeps every low bit of its f32
accumulator up to the bound.  These tests drive each accumulator to within
2^10 of its bound and then add terms of +-1 in the same accumulation group,
where any dropped low bit shows as a mismatch against the oracle (every
element is compared; the oracle computes each distinct input row once and
rows with equal inputs must have equal outputs).

Sources of the bounds: "t27c PTX backend: ternary x int8 GEMM kernel emitted
by a .t27 spec (int8 mma.sync), ptx-run glue", "What this adds" (int32 C from
int8 x ternary); "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8
tensor-core PTX written by t27", kernel 2 (int32 accumulation, reduction
length <= 131071).
"""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CHUNK = 65536                 # terms of one exact accumulation group (ternary products)
R = CHUNK + 8192              # reduction length: a whole chunk and part of the next
N_CLASSES = 6


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    t3.load()
    yield
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device wait timed out, detail={detail:#x}"


def row_classes(g):
    """N_CLASSES activation rows of length R, each a pattern of 'big' runs
    (|a| = 128 or 127, which with |w| = 1 make every product +-128 or +-127)
    and 'small' runs (a in {-1, 0, +1}):
      0: big [0, C-8), small after: partial sums reach 128 (C - 8) = 2^23 - 1024,
         then 8 small terms in the same chunk, then a chunk of small terms;
      1: big [0, C-4096), small to C, big [C, C+4096), small after;
      2: small [0, 4096), big [4096, C+4096) across the chunk boundary, small after;
      3: big of value 127 [0, C-16), small after;
      4: big [0, C-8) with a = -128 and +127 alternating in blocks of 4096
         (the partial sum swings in both directions), small after;
      5: uniform random int8 over the whole reduction."""
    C = CHUNK
    small = lambda n: g.integers(-1, 2, size=n, dtype=np.int16).astype(np.int8)
    rows = np.empty((N_CLASSES, R), dtype=np.int8)
    r = rows[0]; r[:C - 8] = -128; r[C - 8:] = small(R - C + 8)
    r = rows[1]; r[:] = small(R); r[:C - 4096] = -128; r[C:C + 4096] = -128
    r = rows[2]; r[:] = small(R); r[4096:C + 4096] = -128
    r = rows[3]; r[:C - 16] = 127; r[C - 16:] = small(R - C + 16)
    r = rows[4]; r[:] = small(R)
    blocks = (np.arange(C - 8) // 4096) % 2
    r[:C - 8] = np.where(blocks == 0, -128, 127).astype(np.int8)
    rows[5] = t3_synth.int8_uniform(g, R)
    return rows


def class_of_row(M):
    # every class lands in every TMEM lane quadrant and both CTAs of a pair
    m = np.arange(M)
    return (m * 7 + m // 128) % N_CLASSES


# a window of random codes along the reduction, where every row class has
# small activations (or random ones); every other position has weight +-1,
# its sign chosen per output column, so that big activations make big products
SMALL_WINDOWS = [(CHUNK + 4096, R)]


def expand_and_check(got, cls, want_by_class, what):
    want = want_by_class[cls]
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} mismatches of {got.size}; first at "
                           f"{bad[0].tolist()}: got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}")


def fwd_weights(g, N):
    """Packed Wp [N][R/4]: w = s_n (a random sign per column) at every
    reduction index outside SMALL_WINDOWS, random 2-bit codes inside them."""
    s = g.integers(0, 2, size=N)
    wp = np.where(s[:, None] == 1, np.uint8(0x55), np.uint8(0xAA)).astype(np.uint8)
    wp = np.repeat(wp, R // 4, axis=1)
    for (k0, k1) in SMALL_WINDOWS:
        wp[:, k0 // 4:k1 // 4] = t3_synth.raw_bytes(g, (N, (k1 - k0) // 4))
    return np.ascontiguousarray(wp)


@pytest.mark.parametrize("N,schedule", [
    (38 * 192, "whole tiles"),      # 76 tiles of 256x192: one full wave of CTA pairs
    (35 * 192, "split"),            # 70 tiles: the reduction of every tile is split into
                                    # ~530-stage pieces that reach the bound inside a piece
])
def test_forward_chunk_limit(N, schedule):
    g = t3_synth.rng(65536 + N)
    M = 512
    classes = row_classes(g)
    cls = class_of_row(M)
    A = np.ascontiguousarray(classes[cls])
    wp = fwd_weights(g, N)
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), K=R, C=C)
    want = oracle.fwd(classes, wp)
    # partial sums of class 0 reach 2^23 - 1024 before its small terms
    assert np.abs(want[0].astype(np.int64)).max() >= 128 * (CHUNK - 8) - 8
    expand_and_check(C.cpu().numpy(), cls, want, f"fwd chunk limit ({schedule})")


@pytest.mark.parametrize("K,schedule", [
    (38 * 192, "whole tiles"),
    (35 * 192, "split"),
])
def test_dx_chunk_limit(K, schedule):
    """dX = dY . W^T reduces over N: the same row classes along N, W[k][n]
    = s_k outside the windows of n, random codes inside them."""
    g = t3_synth.rng(73728 + K)
    M = 512
    classes = row_classes(g)
    cls = class_of_row(M)
    dY = np.ascontiguousarray(classes[cls])
    s = g.integers(0, 2, size=K)
    # codes of one Wp row: k = 4j + i at bits 2i of byte j, code 1 for +1, 2 for -1
    codes = np.where(s == 1, 1, 2).astype(np.uint8)
    codes = np.concatenate([codes, np.zeros((-K) % 4, np.uint8)]).reshape(-1, 4)
    sign_row = (codes[:, 0] | (codes[:, 1] << 2) | (codes[:, 2] << 4) | (codes[:, 3] << 6)).astype(np.uint8)
    wp = np.repeat(sign_row[None, :], R, axis=0)
    for (n0, n1) in SMALL_WINDOWS:
        wp[n0:n1] = t3_synth.raw_bytes(g, (n1 - n0, wp.shape[1]))
    wp = np.ascontiguousarray(wp)
    dX = torch.empty((M, K), dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dx(torch.from_numpy(dY).cuda(), torch.from_numpy(wp).cuda(), K, dX=dX)
    want = oracle.dx(classes, wp, K)
    assert np.abs(want[0].astype(np.int64)).max() >= 128 * (CHUNK - 8) - 8
    expand_and_check(dX.cpu().numpy(), cls, want, f"dX chunk limit ({schedule})")


def test_dw_chunk_limit_both_signs():
    """dW chunks of 1024 rows: 1023 rows of -128 x -128 (partial 2^24 - 16384)
    or -128 x 127, then one row of +-1 products, in each of two chunks, with
    the signs flipped in the second; columns alternate the sign of dY."""
    g = t3_synth.rng(1023)
    M, K, N = 2048, 96, 160
    A = np.empty((M, K), dtype=np.int8)
    dY = np.empty((M, N), dtype=np.int8)
    col = np.where(np.arange(N) % 2 == 0, -128, 127).astype(np.int8)
    A[:1023] = -128
    dY[:1023] = col
    A[1024:2047] = 127
    dY[1024:2047] = np.clip(-col.astype(np.int16), -128, 127).astype(np.int8)
    for r in (1023, 2047):
        A[r] = g.choice(np.array([-1, 1], dtype=np.int8), size=K)
        dY[r] = g.choice(np.array([-1, 1], dtype=np.int8), size=N)
    dW = torch.empty((K, N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dw(torch.from_numpy(A).cuda(), torch.from_numpy(dY).cuda(), dW=dW)
    want = oracle.dw(A, dY)
    got = dW.cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"dW chunk limit: {len(bad)} mismatches; first {bad[0].tolist()}"


# ------------------------------------------------------------------ small M
# The small-M forward multiplies e4m3 weights (+-1) by activation digits in
# e4m3 (bytes 0..15, each exactly byte * 2^-9) and sums in f32 in TMEM, one
# accumulator per issuing thread, over runs of up to 2048 units of 512
# reduction elements: an accumulator adds at most 2048 * 512 / issuers terms
# of magnitude <= 15 (units of 2^-9), 7.9 M units with two issuers, inside
# 2^24.  K = 4 * 2048 * 512 over one 256-row tile gives each of the two CTA
# pairs that share the tile a slice of exactly two full runs.  Digits of 15
# (a = 127: u = a + 128 = 255; or a = -128 for the signed digits of M = 32)
# fill the accumulators for all but the last unit of every run, whose terms
# are digits 0 or 1 times weights -1, 0 or +1.

SLICE = 2048 * 512
K_SMALL_M = 4 * SLICE


def small_m_rows(g, signed):
    """4 row classes of length K_SMALL_M (see the module comment above)."""
    rows = np.empty((4, K_SMALL_M), dtype=np.int8)
    if signed:
        small_vals = np.array([1, 16, -16, 0, -1], dtype=np.int8)   # hi/lo digits 0 or +-1
        big = (127, -128, 127)
    else:
        small_vals = np.array([-127, -112, -128], dtype=np.int8)   # u = 1, 16, 0
        big = (127, 127, 127)
    rows[0] = big[0]
    rows[1] = big[1]
    rows[2] = t3_synth.int8_uniform(g, K_SMALL_M)
    rows[3] = big[2]
    rows[3].reshape(-1, 512)[1::2] = small_vals[-1]          # every other unit: small values
    for r in (0, 1, 3):
        for q in range(4):
            end = (q + 1) * SLICE
            rows[r, end - 512:end] = g.choice(small_vals, size=512)
    return rows


@pytest.mark.parametrize("M", [1, 8, 31, 32])
def test_small_m_run_limit(M):
    g = t3_synth.rng(4 * SLICE + M)
    N = 256
    classes = small_m_rows(g, signed=(M == 32))
    cls = (np.arange(M) * 3 + np.arange(M) // 4) % 4
    A = np.ascontiguousarray(classes[cls])
    # weights +1 (code 1, byte 0x55) except random codes in the last unit of every slice
    wp = np.full((N, K_SMALL_M // 4), 0x55, dtype=np.uint8)
    for q in range(4):
        end = (q + 1) * SLICE // 4
        wp[:, end - 128:end] = t3_synth.raw_bytes(g, (N, 128))
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), K=K_SMALL_M, C=C)
    want = oracle.fwd(classes, wp)
    expand_and_check(C.cpu().numpy(), cls, want, f"small-M run limit M={M}")
