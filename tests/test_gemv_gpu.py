"""The small-M forward's CUDA-core route (one or two activation rows, and up
to eight over at most 4 MB of packed weights) against the oracle, element by
element: every row-count variant of the kernel (1, 2, 4 and 8 rows per
register block), 16-byte and byte-wise weight and activation loads, fewer
weight rows than SMs, ragged reductions, raw code bytes, the largest K whose
activation copy fits shared memory and the first K past it (which takes the
tensor-core route), and the int32 extremes."""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _fwd(A_dev, wp_dev, M, N, K):
    C = torch.full((M, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    t3.t3_gemm_fwd(A_dev, wp_dev, K=K, C=C)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def _same(got, want, what):
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{what}: {len(bad)} mismatches of {got.size}; first at {bad[0].tolist()}: "
                           f"got {got[tuple(bad[0])]}, want {want[tuple(bad[0])]}")


SHAPES = [
    (64, 8192),    # one row of A's copy per 16 KB: eight rows fill its 64 KB exactly
    (100, 1100),   # fewer weight rows than SMs; packed rows of 275 bytes (byte-wise loads)
    (1531, 448),   # packed rows of 112 bytes (16-byte loads); a ragged last row group
    (300, 61),     # K below one 64-code chunk
    (2048, 2000),  # packed rows of 500 bytes
]


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", SHAPES)
def test_cuda_core_route_matches_oracle(M, N, K):
    g = t3_synth.rng(1000 * M + N + K)
    A = t3_synth.int8_uniform(g, (M, K))
    wp = t3_synth.raw_bytes(g, (N, (K + 3) // 4))  # raw bytes: code 3 and pad codes too
    got = _fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), M, N, K)
    _same(got, oracle.fwd(A, wp), f"fwd {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2, 8])
def test_unaligned_weight_and_activation_bases(M):
    """Wp and A one byte past a 16-byte boundary (and K a multiple of 64, so
    only the base decides the load width)."""
    N, K = 777, 1024
    g = t3_synth.rng(77 + M)
    A = t3_synth.int8_uniform(g, (M, K))
    wp = t3_synth.raw_bytes(g, (N, K // 4))
    a_store = torch.zeros(M * K + 16, dtype=torch.int8, device="cuda")
    w_store = torch.zeros(N * (K // 4) + 16, dtype=torch.uint8, device="cuda")
    a_dev = a_store[1:1 + M * K].view(M, K)
    w_dev = w_store[1:1 + N * (K // 4)].view(N, K // 4)
    a_dev.copy_(torch.from_numpy(A))
    w_dev.copy_(torch.from_numpy(wp))
    _same(_fwd(a_dev, w_dev, M, N, K), oracle.fwd(A, wp), f"unaligned fwd {M}x{N}x{K}")


def test_first_k_past_the_activation_copy_takes_the_tensor_cores():
    """Eight rows at K = 8256 need 66 KB for A's copy: the call takes the
    tensor-core route, with the same result."""
    M, N, K = 8, 64, 8256
    g = t3_synth.rng(8256)
    A = t3_synth.int8_uniform(g, (M, K))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    _same(_fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), M, N, K), oracle.fwd(A, wp),
          f"fwd {M}x{N}x{K}")


def test_int32_extremes_on_the_cuda_cores():
    """|C| = 128 K at the longest reduction whose copy of one activation row
    fits (K = 65536): all -128 against all -1 and all +1, and alternating
    signs that cancel."""
    K, N = 65536, 24
    A = np.full((1, K), -128, dtype=np.int8)
    w = np.empty((K, N), dtype=np.int8)
    w[:, :8] = -1
    w[:, 8:16] = 1
    w[:, 16:] = np.where(np.arange(K)[:, None] % 2 == 0, 1, -1)
    wp = oracle.pack(w)
    got = _fwd(torch.from_numpy(A).cuda(), torch.from_numpy(wp).cuda(), 1, N, K)
    assert np.all(got[0, :8] == 128 * K) and np.all(got[0, 8:16] == -128 * K) and np.all(got[0, 16:] == 0)
    _same(got, oracle.fwd(A, wp), "extremes")
