"""GPU parity of the device packer (t3_pack_ternary_device) against the oracle's
packer, byte for byte, through the C ABI.

Covers the tile edges (K and N not multiples of the 64 x 256 tile, K not a
multiple of 4), both load paths (TMA for 16-byte rows, plain loads for
unaligned rows), both store
paths (8-byte words and single bytes), canaries around the output, invalid
values (packed as 0 and reported as T3_EVALUE), and a packed result feeding
the forward product.
"""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CANARY = 0xA5
PAD = 256  # canary bytes on each side of Wp


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    t3.load()
    yield
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set, detail={detail:#x}"


def _device_pack(w, w_offset=0, wp_offset=0):
    """Packs w on the GPU; w and Wp may start `offset` bytes into their buffers."""
    K, N = w.shape
    KB = (K + 3) // 4
    wbuf = torch.zeros(K * N + w_offset + 16, dtype=torch.int8, device="cuda")
    wd = wbuf[w_offset:w_offset + K * N].view(K, N)
    wd.copy_(torch.from_numpy(np.ascontiguousarray(w)))
    out = torch.full((N * KB + 2 * PAD + wp_offset,), CANARY, dtype=torch.uint8, device="cuda")
    wp = out[PAD + wp_offset:PAD + wp_offset + N * KB].view(N, KB)
    t3.t3_pack_ternary_device(wd, wp)
    torch.cuda.synchronize()
    h = out.cpu().numpy()
    assert np.all(h[:PAD + wp_offset] == CANARY), "bytes before Wp written"
    assert np.all(h[PAD + wp_offset + N * KB:] == CANARY), "bytes after Wp written"
    return wp.cpu().numpy()


# rows of w that are a multiple of 16 bytes take the TMA-fed kernel (tiles of
# 128 k x 128 n, zero-filled past K and N), the others the plain-load one
# (tiles of 64 k x 256 n)
SHAPES = [(1, 1), (3, 5), (4, 16), (5, 7), (63, 127), (64, 128), (65, 129), (96, 272),
          (1000, 333), (130, 4096), (1280, 3456), (13, 64), (257, 1024), (8191, 16),
          (4100, 2048), (192, 112), (640, 400), (127, 144), (129, 256)]


@pytest.mark.parametrize("K,N", SHAPES)
def test_device_pack_matches_oracle(K, N):
    w = t3_synth.ternary(t3_synth.rng(1000 + K * 7 + N), (K, N))
    np.testing.assert_array_equal(_device_pack(w), oracle.pack(w))


@pytest.mark.parametrize("K,N", [(128, 256), (1000, 4096), (97, 160)])
@pytest.mark.parametrize("w_off,wp_off", [(0, 0), (1, 0), (0, 3), (5, 1)])
def test_device_pack_alignment_paths(K, N, w_off, wp_off):
    # offsets move w off 16-byte rows (byte loads) and Wp off 8-byte words
    w = t3_synth.ternary(t3_synth.rng(2000 + K + N + w_off), (K, N), p_zero=0.5)
    np.testing.assert_array_equal(_device_pack(w, w_off, wp_off), oracle.pack(w))


def test_device_pack_all_zero_and_all_ones():
    for value in (0, 1, -1):
        w = np.full((67, 131), value, dtype=np.int8)
        np.testing.assert_array_equal(_device_pack(w), oracle.pack(w))


@pytest.mark.parametrize("N", [300, 320])
def test_device_pack_invalid_values_pack_as_zero_and_are_reported(N):
    K = 200
    w = t3_synth.ternary(t3_synth.rng(77), (K, N))
    bad = [(0, 0, 2), (17, 5, -2), (199, 299, 127), (64, 128, -128), (3, 150, 100)]
    for k, n, v in bad:
        w[k, n] = v
    got = _device_pack(w)
    clean = w.copy()
    for k, n, _ in bad:
        clean[k, n] = 0
    np.testing.assert_array_equal(got, oracle.pack(clean))
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_EVALUE and detail == (9 << 8) | 6
    rc, detail = t3.t3_last_device_error()  # the word was cleared
    assert rc == t3.T3_OK and detail == 0


def test_device_pack_empty_and_bad_arguments():
    empty = torch.zeros((0, 5), dtype=torch.int8, device="cuda")
    wp = t3.t3_pack_ternary_device(empty)
    assert tuple(wp.shape) == (5, 0)
    lib = t3.load()
    assert lib.t3_pack_ternary_device(None, None, 4, 4, None) == t3.T3_EINVAL
    assert lib.t3_pack_ternary_device(None, None, -1, 4, None) == t3.T3_EINVAL


def test_device_pack_feeds_the_forward():
    M, K, N = 300, 1000, 333
    g = t3_synth.rng(31)
    A = t3_synth.int8_uniform(g, (M, K))
    w = t3_synth.ternary(g, (K, N))
    wd = torch.from_numpy(w).cuda()
    wp = t3.t3_pack_ternary_device(wd)
    C = t3.t3_gemm_fwd(torch.from_numpy(A).cuda(), wp, K=K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().numpy(), oracle.fwd(A, oracle.pack(w)))


def test_device_pack_full_size_8192():
    K = N = 8192
    w = t3_synth.ternary(t3_synth.rng(8192), (K, N))
    np.testing.assert_array_equal(_device_pack(w), oracle.pack(w))
