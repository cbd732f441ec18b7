"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit-exact.

Inputs come from t3_synth (seeded); the weights are packed by the library's
packer for the GPU and by the oracle's own packer for the oracle (the two are
compared in the CPU tests).  Every output is compared element by element in
full, the full-size workloads included (in the launch configuration the bench
uses), except the large unaligned case, which is compared on sampled rows.
Output buffers carry canary words before and after the result.
"""
import functools

import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CANARY = 0x5A5A5A5A  # an int32 value that marks untouched words
PAD = 64                         # canary words on each side of an output


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), f"built for sm_103a, found sm_{major}{minor}"
    t3.load()
    yield
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device wait timed out, detail={detail:#x}"


@functools.lru_cache(maxsize=4)
def workload_inputs(name):
    return t3_synth.make_inputs(t3_synth.BY_NAME[name])


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _guarded(rows, cols):
    buf = torch.full((rows * cols + 2 * PAD,), CANARY, dtype=torch.int32, device="cuda")
    return buf, buf[PAD:PAD + rows * cols].view(rows, cols)


def _check_guard(buf, rows, cols):
    h = buf.cpu().numpy()
    assert np.all(h[:PAD] == CANARY) and np.all(h[PAD + rows * cols:] == CANARY), "canary overwritten"


def run_fwd(A, wp):
    M, K = A.shape
    N = wp.shape[0]
    buf, C = _guarded(M, N)
    t3.t3_gemm_fwd(_dev(A), _dev(wp), K=K, C=C)
    torch.cuda.synchronize()
    _check_guard(buf, M, N)
    return C.cpu().numpy()


def run_dx(dY, wp, K):
    M, N = dY.shape
    buf, dX = _guarded(M, K)
    t3.t3_gemm_bwd_dx(_dev(dY), _dev(wp), K, dX=dX)
    torch.cuda.synchronize()
    _check_guard(buf, M, K)
    return dX.cpu().numpy()


def run_dw(A, dY):
    M, K = A.shape
    N = dY.shape[1]
    buf, dW = _guarded(K, N)
    t3.t3_gemm_bwd_dw(_dev(A), _dev(dY), dW=dW)
    torch.cuda.synchronize()
    _check_guard(buf, K, N)
    return dW.cpu().numpy()


def assert_same(got, want, what):
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} mismatches of {got.size}; first at {bad[0].tolist()}: "
                           f"got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}")


def inputs(M, N, K, seed, p_zero=1.0 / 3.0):
    g = t3_synth.rng(seed)
    A = t3_synth.int8_uniform(g, (M, K))
    w = t3_synth.ternary(g, (K, N), p_zero)
    dY = t3_synth.int8_uniform(g, (M, N))
    return A, w, dY


# ------------------------------------------------------------ small, full ---

def test_ragged_300x272x96_forward():
    """The pages' ragged case: every guard path (K=96 makes the packed row
    24 bytes, which TMA cannot stride, so the plain-load producer runs)."""
    wl = t3_synth.BY_NAME["fwd_ragged_300x272x96"]
    A, w, _ = t3_synth.make_inputs(wl)
    assert_same(run_fwd(A, t3.t3_pack_ternary(w)), oracle.fwd(A, oracle.pack(w)), "fwd 300x272x96")


SMALL = [(1, 1, 1), (1, 16, 16), (128, 128, 32), (5, 7, 3), (70, 33, 65), (129, 257, 64),
         (256, 256, 128), (200, 300, 200), (33, 513, 130), (300, 272, 96), (130, 1000, 1024)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_small_shapes_all_three(M, N, K):
    A, w, dY = inputs(M, N, K, seed=M * 7 + N * 3 + K)
    wp_gpu, wp_ref = t3.t3_pack_ternary(w), oracle.pack(w)
    assert_same(run_fwd(A, wp_gpu), oracle.fwd(A, wp_ref), f"fwd {M}x{N}x{K}")
    assert_same(run_dx(dY, wp_gpu, K), oracle.dx(dY, wp_ref, K), f"dX {M}x{N}x{K}")
    assert_same(run_dw(A, dY), oracle.dw(A, dY), f"dW {M}x{N}x{K}")


def test_random_tiny_shapes():
    g = np.random.default_rng(1234)
    for it in range(12):
        M, N, K = (int(x) for x in g.integers(1, 71, size=3))
        A, w, dY = inputs(M, N, K, seed=5000 + it)
        wp = t3.t3_pack_ternary(w)
        assert_same(run_fwd(A, wp), oracle.fwd(A, wp), f"fwd {M}x{N}x{K}")
        assert_same(run_dx(dY, wp, K), oracle.dx(dY, wp, K), f"dX {M}x{N}x{K}")
        assert_same(run_dw(A, dY), oracle.dw(A, dY), f"dW {M}x{N}x{K}")


def test_raw_codes_and_pad_bits():
    """Random packed bytes: code 3 everywhere it lands and nonzero pad bits."""
    g = t3_synth.rng(77)
    for (M, N, K) in [(9, 40, 13), (150, 260, 255), (64, 300, 1030)]:
        wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4))
        A = t3_synth.int8_uniform(g, (M, K))
        dY = t3_synth.int8_uniform(g, (M, N))
        assert_same(run_fwd(A, wp), oracle.fwd(A, wp), f"fwd raw {M}x{N}x{K}")
        assert_same(run_dx(dY, wp, K), oracle.dx(dY, wp, K), f"dX raw {M}x{N}x{K}")


def test_unaligned_pointers_take_global_load_modes():
    """Operands at odd byte offsets cannot be TMA sources: the converters load
    them from global memory (single bytes); results are the same."""
    M, N, K = 150, 200, 320
    A, w, dY = inputs(M, N, K, seed=99)
    wp = t3.t3_pack_ternary(w)
    def shifted(a):
        flat = np.ascontiguousarray(a).reshape(-1)
        buf = torch.empty(flat.size + 1, dtype=torch.from_numpy(flat).dtype, device="cuda")
        buf[1:] = torch.from_numpy(flat).cuda()
        return buf[1:].view(a.shape)
    C = torch.empty((M, N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(shifted(A), shifted(wp), K=K, C=C)
    assert_same(C.cpu().numpy(), oracle.fwd(A, wp), "fwd unaligned")
    dX = torch.empty((M, K), dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dx(shifted(dY), shifted(wp), K, dX=dX)
    assert_same(dX.cpu().numpy(), oracle.dx(dY, wp, K), "dX unaligned")
    dW = torch.empty((K, N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dw(shifted(A), shifted(dY), dW=dW)
    assert_same(dW.cpu().numpy(), oracle.dw(A, dY), "dW unaligned")


# ------------------------------------------------------ exactness extremes --

def test_int32_extremes_and_long_reductions():
    # 128 * K at K = 8192
    K, M, N = 8192, 130, 300
    A = np.full((M, K), -128, dtype=np.int8)
    wp = t3.t3_pack_ternary(-np.ones((K, N), dtype=np.int8))
    C = run_fwd(A, wp)
    assert np.all(C == 128 * K)
    # dW over 1782 rows at the extreme: 16384 * 1782 > 2^24, so the f32
    # accumulator alone could not hold it exactly; the chunked sum must.
    M2 = 1782
    A2 = np.full((M2, 96), -128, dtype=np.int8)
    dW = run_dw(A2, A2[:, :80].copy())
    assert np.all(dW == 16384 * M2)


def test_adversarial_large_then_small_terms():
    """A large running sum followed by +-1 terms: any loss of low bits in the
    f32 accumulation shows up as a mismatch."""
    g = t3_synth.rng(31)
    M, N, K = 256, 256, 4096
    A = np.empty((M, K), dtype=np.int8)
    A[:, : K // 2] = 127
    A[:, K // 2:] = g.choice(np.array([-1, 1], dtype=np.int8), size=(M, K - K // 2))
    w = t3_synth.ternary(g, (K, N), 0.0)
    w[: K // 2] = 1
    wp = t3.t3_pack_ternary(w)
    assert_same(run_fwd(A, wp), oracle.fwd(A, oracle.pack(w)), "fwd adversarial")
    # dW: rows of 127*127 products then +-1 products, across the chunk boundary
    M3 = 1500
    A3 = np.empty((M3, 64), dtype=np.int8)
    A3[:1000] = 127
    A3[1000:] = g.choice(np.array([-1, 1], dtype=np.int8), size=(M3 - 1000, 64))
    dY3 = A3[:, ::-1].copy()
    assert_same(run_dw(A3, dY3), oracle.dw(A3, dY3), "dW adversarial")


# ------------------------------------------------------------ full-size ---
# Every workload in the bench's launch configuration, every element compared
# with the oracle.

@pytest.mark.parametrize("name", ["fwd_square_4096", "fwd_16384x3456x1280"] +
                         [f"fwd_{m}x{n}x{k}" for (m, n, k) in t3_synth.PAGES_FWD_SHAPES])
def test_full_size_forward(name):
    wl = t3_synth.BY_NAME[name]
    A, w, _ = workload_inputs(name)
    wp = t3.t3_pack_ternary(w)
    C = torch.empty((wl.M, wl.N), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(_dev(A), _dev(wp), K=wl.K, C=C)
    assert_same(C.cpu().numpy(), oracle.fwd(A, oracle.pack(w)), name)


@pytest.mark.parametrize("M", [1782, 16384])
def test_full_size_backward(M):
    N, K = 3456, 1280
    wl = t3_synth.BY_NAME["bwd_1782x3456x1280"]
    A, w, dY = (t3_synth.make_inputs(wl) if M == wl.M else inputs(M, N, K, seed=2))
    wp = t3.t3_pack_ternary(w)
    dX = t3.t3_gemm_bwd_dx(_dev(dY), _dev(wp), K)
    dW = t3.t3_gemm_bwd_dw(_dev(A), _dev(dY))
    assert_same(dX.cpu().numpy(), oracle.dx(dY, oracle.pack(w), K), f"dX M={M}")
    assert_same(dW.cpu().numpy(), oracle.dw(A, dY), f"dW M={M}")


@pytest.mark.parametrize("M", [1, 8, 27])
@pytest.mark.parametrize("NK", [(3456, 1280), (8192, 8192)])
def test_small_m_forward(M, NK):
    N, K = NK
    wl = t3_synth.BY_NAME[f"skinny_m{M}_n{N}_k{K}"]
    A, w, _ = workload_inputs(wl.name)
    wp = t3.t3_pack_ternary(w)
    assert_same(run_fwd(A, wp), oracle.fwd(A, oracle.pack(w)), wl.name)


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 32, 33])
def test_small_m_boundaries(M):
    """Rows on both sides of the small-M path's limits (16 and 32 rows), with
    several k-groups, TMA and plain-load weight paths, bulk and atomic outputs."""
    for (N, K) in [(300, 1100), (1024, 2048), (130, 2500), (256, 64)]:
        A, w, _ = inputs(M, N, K, seed=M * 13 + N + K)
        wp = t3.t3_pack_ternary(w)
        assert_same(run_fwd(A, wp), oracle.fwd(A, oracle.pack(w)), f"fwd {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (8, 10240, 8192),    # 40 tiles of 256 rows: clusters of up to 4 CTA pairs, several tiles each
    (32, 10240, 8192),
    (27, 24576, 8192),   # 96 tiles: clusters of 2 pairs, three tiles each
    (1, 24576, 4100),    # ragged last unit, packed rows not 16-byte aligned
    (16, 3456 * 3, 1280),
    (5, 300, 70000),     # one tile, a long reduction split over the cluster's pairs
])
def test_small_m_cluster_schedules(M, N, K):
    """Small-M shapes whose tiles and k-slices exercise every cluster shape
    of the small-M path: one tile per cluster or several (the first pair's
    partial buffers reused), one to four pairs per cluster."""
    A, w, _ = inputs(M, N, K, seed=M + N + K)
    wp = oracle.pack(w)
    assert_same(run_fwd(A, wp), oracle.fwd(A, wp), f"fwd {M}x{N}x{K}")


def test_small_m_output_not_zeroed_first():
    """The small-M path overwrites C without reading it: garbage in C before
    the call (and a previous product's result) leaves no trace."""
    g = t3_synth.rng(404)
    for (M, N, K) in [(8, 1024, 4096), (27, 3456, 1280)]:
        A = t3_synth.int8_uniform(g, (M, K))
        wp = oracle.pack(t3_synth.ternary(g, (K, N)))
        C = torch.randint(-2**31, 2**31 - 1, (M, N), dtype=torch.int32, device="cuda")
        t3.t3_gemm_fwd(_dev(A), _dev(wp), K=K, C=C)
        t3.t3_gemm_fwd(_dev(A), _dev(wp), K=K, C=C)
        torch.cuda.synchronize()
        assert_same(C.cpu().numpy(), oracle.fwd(A, wp), f"fwd {M}x{N}x{K} over garbage")


def test_small_m_extremes():
    K = 8192
    for M in (1, 27):
        A = np.full((M, K), -128, dtype=np.int8)
        wp = t3.t3_pack_ternary(-np.ones((K, 200), dtype=np.int8))
        assert np.all(run_fwd(A, wp) == 128 * K)


def test_repeated_calls_same_result():
    A, w, dY = inputs(300, 600, 700, seed=8)
    wp = t3.t3_pack_ternary(w)
    first = run_fwd(A, wp)
    for _ in range(3):
        assert np.array_equal(run_fwd(A, wp), first)


def test_small_m_chained_calls_see_earlier_outputs():
    """Back-to-back small-M calls on one stream, each reading the previous
    call's output bytes as its input (activations, then packed weights): every
    call must see the finished result of the one before it, whatever overlap
    the launches allow."""
    g = t3_synth.rng(21)
    A0 = t3_synth.int8_uniform(g, (8, 1024))
    wp0 = oracle.pack(t3_synth.ternary(g, (1024, 512)))
    wp1 = oracle.pack(t3_synth.ternary(g, (2048, 300)))
    A2 = t3_synth.int8_uniform(g, (5, 1600))
    C0 = torch.empty((8, 512), dtype=torch.int32, device="cuda")
    C1 = torch.empty((8, 300), dtype=torch.int32, device="cuda")
    C2 = torch.empty((5, 24), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(_dev(A0), _dev(wp0), K=1024, C=C0)
    t3.t3_gemm_fwd(C0.view(torch.int8).view(8, 2048), _dev(wp1), K=2048, C=C1)
    t3.t3_gemm_fwd(_dev(A2), C1.view(torch.uint8).view(24, 400), K=1600, C=C2)
    torch.cuda.synchronize()
    c0, c1, c2 = C0.cpu().numpy(), C1.cpu().numpy(), C2.cpu().numpy()
    assert_same(c0, oracle.fwd(A0, wp0), "chained call 1")
    assert_same(c1, oracle.fwd(c0.view(np.int8).reshape(8, 2048), wp1), "chained call 2")
    assert_same(c2, oracle.fwd(A2, c1.view(np.uint8).reshape(24, 400)), "chained call 3")


def test_empty_reduction_writes_zeros():
    C = torch.full((5, 7), 3, dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(torch.empty((5, 0), dtype=torch.int8, device="cuda"),
                   torch.empty((7, 0), dtype=torch.uint8, device="cuda"), K=0, C=C)
    # dX over an empty N and dW over an empty M: zeros, whatever was there
    dX = torch.full((5, 9), 3, dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dx(torch.empty((5, 0), dtype=torch.int8, device="cuda"),
                      torch.empty((0, 3), dtype=torch.uint8, device="cuda"), 9, dX=dX)
    dW = torch.full((6, 4), 3, dtype=torch.int32, device="cuda")
    t3.t3_gemm_bwd_dw(torch.empty((0, 6), dtype=torch.int8, device="cuda"),
                      torch.empty((0, 4), dtype=torch.int8, device="cuda"), dW=dW)
    torch.cuda.synchronize()
    for out in (C, dX, dW):
        assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("M,N,K", [(512, 1024, 4000), (300, 4000, 1008), (257, 336, 272)])
def test_weight_rows_not_16_byte_aligned(M, N, K):
    # ceil(K/4) a multiple of 4 but not of 16: the pair pipeline loads the
    # weight words itself instead of by TMA
    g = t3_synth.rng(M + N + K)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    np.testing.assert_array_equal(run_fwd(A, wp), oracle.fwd(A, wp))
    np.testing.assert_array_equal(run_dx(dY, wp, K), oracle.dx(dY, wp, K))


@pytest.mark.parametrize("M,N,K", [(1782, 729, 243), (300, 243, 729), (257, 1001, 999), (64, 17, 33)])
def test_rows_not_16_byte_aligned(M, N, K):
    # activation and weight rows TMA cannot address: the pair pipeline's
    # converters load them from global memory (words or single bytes)
    g = t3_synth.rng(3 * M + N + K)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    np.testing.assert_array_equal(run_fwd(A, wp), oracle.fwd(A, wp))
    np.testing.assert_array_equal(run_dx(dY, wp, K), oracle.dx(dY, wp, K))
    # dW: operands loaded by its converters; N % 4 != 0 adds element by element
    np.testing.assert_array_equal(run_dw(A, dY), oracle.dw(A, dY))


def test_unaligned_large_sampled_rows():
    M, N, K = 4096, 4096, 4088
    g = t3_synth.rng(4088)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, 4088))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    rows = np.array([0, 1, 255, 256, 2047, 4095])
    np.testing.assert_array_equal(run_fwd(A, wp)[rows], oracle.fwd(A, wp, rows))
    wp2 = oracle.pack(t3_synth.ternary(g, (K, 4088)))
    np.testing.assert_array_equal(run_dx(dY, wp2, K)[rows], oracle.dx(dY, wp2, K, rows))
    krows = np.array([0, 127, 128, 2047, 4087])
    np.testing.assert_array_equal(run_dw(A, dY)[krows], oracle.dw(A, dY, krows))


# ------------------------------------------------ split (stream-K) schedule --
# When whole tiles would leave pairs idle for long (few tiles, long
# reductions), the pair pipeline deals the full waves as whole tiles and
# splits the remaining tiles' reduction stages evenly over all pairs; those
# pieces add onto rows zeroed by a chained grid.  The shapes below take that
# schedule (it needs operands TMA can address), including pieces that cross
# an exact chunk boundary, outputs that need atomic adds, and a partial wave
# after a whole one.

@pytest.mark.parametrize("M,N,K", [
    (300, 400, 4096),    # 6 tiles of 32 stages, all split
    (40, 20, 70016),     # 1 tile of 547 stages: pieces cross the 65536-element chunk bound
    (300, 271, 4096),    # output rows not 16-byte aligned: pieces add with atomics
    (1792, 2112, 2048),  # 77 tiles: one wave whole, 1 tile split, zeroed band shared
    (300, 400, 4032),    # a ragged last stage (K % 128 = 64) inside the last pieces
    (1792, 2111, 2048),  # 77 tiles, output rows not 16-byte aligned: plain stores of the
                         # whole tiles in the zeroed band, atomic adds for the split one
])
def test_split_schedule_forward(M, N, K):
    A, w, _ = inputs(M, N, K, seed=M + 3 * N + K)
    wp = oracle.pack(w)
    assert_same(run_fwd(A, wp), oracle.fwd(A, wp), f"fwd split {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [
    (300, 4096, 448),    # dX 300x448 over a 4096-long reduction, all split
    (27, 3456, 1280),    # small M: 7 tiles of 27 stages
    (40, 70016, 64),     # 547 stages, the chunk bound inside pieces
    (300, 4096, 447),    # dX rows not 16-byte aligned: atomic adds
    (1792, 2048, 2112),  # 77 tiles: one wave whole, the rest split
    (300, 4032, 448),    # a ragged last stage of the reduction (N % 128 = 64)
])
def test_split_schedule_dx(M, N, K):
    _, w, dY = inputs(M, N, K, seed=7 * M + N + K)
    wp = oracle.pack(w)
    assert_same(run_dx(dY, wp, K), oracle.dx(dY, wp, K), f"dX split {M}x{N}x{K}")


def test_split_schedule_chained_calls_see_earlier_outputs():
    """Split-schedule products back to back on one stream, each reading the
    previous output's bytes as its input: the zeroing grid of a call must not
    start before the call before it has finished, nor the product before its
    inputs exist."""
    g = t3_synth.rng(23)
    A0 = t3_synth.int8_uniform(g, (300, 4096))
    wp0 = oracle.pack(t3_synth.ternary(g, (4096, 400)))
    wp1 = oracle.pack(t3_synth.ternary(g, (1600, 272)))
    A2 = t3_synth.int8_uniform(g, (64, 4352))
    C0 = torch.empty((300, 400), dtype=torch.int32, device="cuda")
    C1 = torch.empty((300, 272), dtype=torch.int32, device="cuda")
    C2 = torch.empty((64, 300), dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(_dev(A0), _dev(wp0), K=4096, C=C0)
    t3.t3_gemm_fwd(C0.view(torch.int8).view(300, 1600), _dev(wp1), K=1600, C=C1)
    t3.t3_gemm_fwd(_dev(A2), C1.view(torch.uint8).view(300, 1088), K=4352, C=C2)
    torch.cuda.synchronize()
    c0, c1, c2 = C0.cpu().numpy(), C1.cpu().numpy(), C2.cpu().numpy()
    assert_same(c0, oracle.fwd(A0, wp0), "split chained call 1")
    assert_same(c1, oracle.fwd(c0.view(np.int8).reshape(300, 1600), wp1), "split chained call 2")
    assert_same(c2, oracle.fwd(A2, c1.view(np.uint8).reshape(300, 1088)), "split chained call 3")


def test_random_long_reduction_shapes():
    """Random few-tile shapes with long reductions (most take the split
    schedule, with pieces of random lengths and boundaries), fwd and dX, in
    full against the oracle."""
    g = np.random.default_rng(2026)
    for it in range(8):
        M = int(g.integers(33, 700))
        N = int(g.integers(1, 6)) * 64 + int(g.integers(0, 2)) * 32
        K = int(g.integers(8, 80)) * 64
        A, w, dY = inputs(M, N, K, seed=9000 + it)
        wp = oracle.pack(w)
        assert_same(run_fwd(A, wp), oracle.fwd(A, wp), f"fwd {M}x{N}x{K}")
        _, w2, dY2 = inputs(M, K, N, seed=9100 + it)   # dX over a K-long reduction
        wp2 = oracle.pack(w2)
        assert_same(run_dx(dY2, wp2, N), oracle.dx(dY2, wp2, N), f"dX {M}x{K}x{N}")


def test_random_dw_shapes():
    """dW over random reductions (partial 128-row stages, 1024-row chunk
    boundaries, a second chunk of any length) and random widths (TMA-aligned
    or not), in full against the oracle."""
    g = np.random.default_rng(77)
    for it in range(8):
        M = int(g.integers(1, 3000))
        K = int(g.integers(1, 400)) if it % 2 else int(g.integers(1, 25)) * 16
        N = int(g.integers(1, 400)) if it % 3 == 2 else int(g.integers(1, 25)) * 16
        A = t3_synth.int8_uniform(t3_synth.rng(9200 + it), (M, K))
        dY = t3_synth.int8_uniform(t3_synth.rng(9300 + it), (M, N))
        assert_same(run_dw(A, dY), oracle.dw(A, dY), f"dW {M}x{N}x{K}")


def test_million_term_reductions():
    """Reductions of 2^20 terms (16 exact f32 chunks of 65536, spread over
    every CTA pair by the split schedule): extreme values, whose sum 128 * 2^20
    is exact only if every chunk is added in int32, and random values against
    the oracle, for the forward and dX."""
    R = 1 << 20
    A = np.full((40, R), -128, dtype=np.int8)
    wp = t3.t3_pack_ternary(-np.ones((R, 16), dtype=np.int8))
    assert np.all(run_fwd(A, wp) == 128 * R)
    dY = np.full((40, R), -128, dtype=np.int8)
    wp_dx = t3.t3_pack_ternary(-np.ones((64, R), dtype=np.int8))
    assert np.all(run_dx(dY, wp_dx, 64) == 128 * R)
    g = t3_synth.rng(1 << 20)
    A2 = t3_synth.int8_uniform(g, (33, R))
    wp2 = oracle.pack(t3_synth.ternary(g, (R, 8)))
    assert_same(run_fwd(A2, wp2), oracle.fwd(A2, wp2), "fwd 33x8x2^20")
    dY2 = t3_synth.int8_uniform(g, (33, R))
    wp3 = oracle.pack(t3_synth.ternary(g, (64, R)))
    assert_same(run_dx(dY2, wp3, 64), oracle.dx(dY2, wp3, 64), "dX 33x2^20x64")


def test_dw_at_the_row_bound():
    """dW over the pages' largest reduction, 131071 rows (128 exact chunks of
    1024): -128 * -128 on every row sums to 2147467264, just inside int32;
    random values there against the oracle."""
    Mb = 131071
    A = np.full((Mb, 16), -128, dtype=np.int8)
    dY = np.full((Mb, 32), -128, dtype=np.int8)
    assert np.all(run_dw(A, dY) == 16384 * Mb)
    g = t3_synth.rng(Mb)
    A2 = t3_synth.int8_uniform(g, (Mb, 16))
    dY2 = t3_synth.int8_uniform(g, (Mb, 48))
    assert_same(run_dw(A2, dY2), oracle.dw(A2, dY2), "dW 131071 rows")
