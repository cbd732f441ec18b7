"""The CUDA-core route for small products (M*N*K up to the library's limit,
2^29 by default), with the library's default routing, against the oracle,
element by element: the pages' HSLM layer widths (243 and 729 at 27 and 1782
rows) for all three products, ragged shapes on both sides of the 64-element
tiles and chunks, raw code bytes (code 3, pad bits), operands one byte past a
16-byte boundary, the reduction split over CTAs (atomic adds onto a zeroed
output), each product at its int32 bound, and the limit's two sides giving
the same result."""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")

pytestmark = [pytest.mark.gpu, pytest.mark.small_route]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _same(got, want, what):
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} mismatches of {got.size}; first at {bad[0].tolist()}: "
                           f"got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}")


def _all_three(M, N, K, seed, raw=True):
    g = t3_synth.rng(seed)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4)) if raw else oracle.pack(t3_synth.ternary(g, (K, N)))
    C = t3.t3_gemm_fwd(_dev(A), _dev(wp), K=K)
    dX = t3.t3_gemm_bwd_dx(_dev(dY), _dev(wp), K)
    dW = t3.t3_gemm_bwd_dw(_dev(A), _dev(dY))
    torch.cuda.synchronize()
    _same(C.cpu().numpy(), oracle.fwd(A, wp), f"fwd {M}x{N}x{K}")
    _same(dX.cpu().numpy(), oracle.dx(dY, wp, K), f"dX {M}x{N}x{K}")
    _same(dW.cpu().numpy(), oracle.dw(A, dY), f"dW {M}x{N}x{K}")


@pytest.mark.parametrize("M", [27, 1782])
@pytest.mark.parametrize("N,K", [(729, 243), (243, 729)])
def test_hslm_widths(M, N, K):
    _all_three(M, N, K, seed=M + N + K, raw=False)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 1), (1, 5, 3), (3, 1, 7), (64, 64, 64), (63, 65, 64), (65, 63, 65), (129, 127, 191),
    (300, 272, 96),  # the pages' ragged forward shape
    (33, 200, 1000), (100, 7, 4093), (5, 300, 300),
])
def test_ragged_shapes_raw_codes(M, N, K):
    _all_three(M, N, K, seed=7 * M + 3 * N + K, raw=True)


def test_unaligned_bases():
    """Every operand one byte past a 16-byte boundary, the outputs 4 bytes past
    one: rows of any length are read byte-wise or as words where they allow."""
    M, N, K = 201, 140, 260
    g = t3_synth.rng(11)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4))

    def shifted(a, dtype, off):
        store = torch.zeros(a.size + 64, dtype=dtype, device="cuda")
        view = store[off:off + a.size].view(a.shape)
        view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
        return view

    A_d = shifted(A, torch.int8, 1)
    dY_d = shifted(dY, torch.int8, 1)
    wp_d = shifted(wp, torch.uint8, 1)
    outs = {name: torch.zeros(rows * cols + 8, dtype=torch.int32, device="cuda")[1:1 + rows * cols].view(rows, cols)
            for name, rows, cols in (("C", M, N), ("dX", M, K), ("dW", K, N))}
    t3.t3_gemm_fwd(A_d, wp_d, K=K, C=outs["C"])
    t3.t3_gemm_bwd_dx(dY_d, wp_d, K, dX=outs["dX"])
    t3.t3_gemm_bwd_dw(A_d, dY_d, outs["dW"])
    torch.cuda.synchronize()
    _same(outs["C"].cpu().numpy(), oracle.fwd(A, wp), "fwd")
    _same(outs["dX"].cpu().numpy(), oracle.dx(dY, wp, K), "dX")
    _same(outs["dW"].cpu().numpy(), oracle.dw(A, dY), "dW")


@pytest.mark.parametrize("op", ["fwd", "dx", "dw"])
def test_split_reduction_adds_onto_zeros(op):
    """One or two output tiles over a long reduction: the reduction is split
    over many CTAs that add atomically; the output starts as garbage."""
    g = t3_synth.rng(21)
    if op == "fwd":
        M, N, K = 40, 70, 60001  # rows of A not word-aligned: the CUDA cores up to 2^29
        A = t3_synth.int8_uniform(g, (M, K))
        wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4))
        C = torch.full((M, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
        t3.t3_gemm_fwd(_dev(A), _dev(wp), K=K, C=C)
        torch.cuda.synchronize()
        _same(C.cpu().numpy(), oracle.fwd(A, wp), "fwd")
    elif op == "dx":
        M, N, K = 50, 60000, 70
        dY = t3_synth.int8_uniform(g, (M, N))
        wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4))
        dX = torch.full((M, K), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
        t3.t3_gemm_bwd_dx(_dev(dY), _dev(wp), K, dX=dX)
        torch.cuda.synchronize()
        _same(dX.cpu().numpy(), oracle.dx(dY, wp, K), "dX")
    else:
        M, N, K = 60000, 70, 50
        A = t3_synth.int8_uniform(g, (M, K))
        dY = t3_synth.int8_uniform(g, (M, N))
        dW = torch.full((K, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
        t3.t3_gemm_bwd_dw(_dev(A), _dev(dY), dW)
        torch.cuda.synchronize()
        _same(dW.cpu().numpy(), oracle.dw(A, dY), "dW")


def test_int32_bounds():
    """Each product at the largest reduction the library accepts, with the
    extreme values: fwd and dX at 16777215 terms of 128 (|sum| = 2^31 - 128),
    dW at 131071 terms of 16384 (2^31 - 16384)."""
    R = 16777215
    A = np.full((1, R), -128, dtype=np.int8)
    wp = oracle.pack(np.ones((R, 2), dtype=np.int8))
    C = t3.t3_gemm_fwd(_dev(A), _dev(wp), K=R)
    torch.cuda.synchronize()
    assert C.cpu().numpy().tolist() == [[-128 * R, -128 * R]]
    dY = np.full((1, R), -128, dtype=np.int8)
    wpx = oracle.pack(np.ones((1, R), dtype=np.int8))  # K = 1, N = R
    dX = t3.t3_gemm_bwd_dx(_dev(dY), _dev(wpx), 1)
    torch.cuda.synchronize()
    assert dX.cpu().numpy().tolist() == [[-128 * R]]
    M = 131071
    A2 = np.full((M, 3), -128, dtype=np.int8)
    dY2 = np.full((M, 5), -128, dtype=np.int8)
    dW = t3.t3_gemm_bwd_dw(_dev(A2), _dev(dY2))
    torch.cuda.synchronize()
    assert np.all(dW.cpu().numpy() == 16384 * M)


def test_both_sides_of_the_limit_agree():
    """The same small products through the CUDA cores (default limit) and
    through the tensor cores (limit 0): identical int32 outputs."""
    M, N, K = 700, 301, 519  # rows of A, dY and Wp not word-aligned: all three on the CUDA cores
    g = t3_synth.rng(31)
    A = _dev(t3_synth.int8_uniform(g, (M, K)))
    dY = _dev(t3_synth.int8_uniform(g, (M, N)))
    wp = _dev(oracle.pack(t3_synth.ternary(g, (K, N))))
    small = (t3.t3_gemm_fwd(A, wp, K=K), t3.t3_gemm_bwd_dx(dY, wp, K), t3.t3_gemm_bwd_dw(A, dY))
    prev = t3.t3_set_small_product_limit(0)
    try:
        big = (t3.t3_gemm_fwd(A, wp, K=K), t3.t3_gemm_bwd_dx(dY, wp, K), t3.t3_gemm_bwd_dw(A, dY))
    finally:
        t3.t3_set_small_product_limit(prev)
    torch.cuda.synchronize()
    for s, b, name in zip(small, big, ("fwd", "dX", "dW")):
        assert torch.equal(s, b), name
