"""GPU parity of the row quantizer (t3_quantize_rows_bf16) against the oracle,
bit for bit (int8 codes and float scales), and the chain it feeds: bf16
activations -> int8 + row scales -> scaled forward -> float output."""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    t3.load()
    yield
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set, detail={detail:#x}"


def _bf16_bits(x):
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _rows(g, M, K):
    mag = np.float32(10.0) ** g.integers(-6, 7, (M, 1)).astype(np.float32)
    return _bf16_bits((g.standard_normal((M, K)) * mag).astype(np.float32))


def _run(bits, offset=0):
    M, K = bits.shape
    buf = torch.zeros(M * K + offset + 8, dtype=torch.int16, device="cuda")
    x = buf[offset:offset + M * K].view(M, K).view(torch.bfloat16)
    x.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    q, s = t3.t3_quantize_rows_bf16(x)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 1), (3, 5), (7, 13), (64, 128), (300, 1280), (33, 4104)])
def test_quantize_matches_oracle(M, K):
    bits = _rows(t3_synth.rng(M * 7 + K), M, K)
    bits[0, :] = 0                     # a zero row
    q, s = _run(bits)
    qo, so = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantize_unaligned_rows_take_the_scalar_path():
    bits = _rows(t3_synth.rng(3), 40, 256)
    q, s = _run(bits, offset=1)        # 2 bytes off 16-byte alignment
    qo, so = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantize_ties_and_float32_rounding_rows():
    pairs = [(0.00982666015625, 0.0196533203125), (0.0128173828125, 0.025634765625),
             (0.01409912109375, 0.0281982421875), (0.0279541015625, 0.055908203125),
             (0.75, 127.0), (1.5, 127.0), (2.5, 127.0), (-2.5, 127.0)]
    bits = np.stack([_bf16_bits(np.array([x, amax, 0, 0, 0, 0, 0, 0], np.float32)) for x, amax in pairs])
    q, s = _run(bits)
    qo, so = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantize_empty_rows_give_zero_scales():
    x = torch.zeros((5, 0), dtype=torch.bfloat16, device="cuda")
    q, s = t3.t3_quantize_rows_bf16(x)
    torch.cuda.synchronize()
    assert q.shape == (5, 0) and np.all(s.cpu().numpy() == 0)


def test_quantize_layer_activations_in_full():
    bits = _rows(t3_synth.rng(16384), 16384, 1280)
    q, s = _run(bits)
    qo, so = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(q, qo)
    np.testing.assert_array_equal(s.view(np.uint32), so.view(np.uint32))


def test_quantize_then_scaled_forward():
    g = t3_synth.rng(44)
    M, K, N = 300, 1280, 272
    bits = _rows(g, M, K)
    w = t3_synth.ternary(g, (K, N))
    wp = oracle.pack(w)
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, s = t3.t3_quantize_rows_bf16(x)
    C = t3.t3_gemm_fwd_scaled(q, torch.from_numpy(wp).cuda(), K, s, None, t3.T3_OUT_F32)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rows(bits)
    want = oracle.dequant(oracle.fwd(qo, wp), so, None)
    np.testing.assert_array_equal(C.cpu().numpy().view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------- the fused forward --
# t3_gemm_fwd_bf16: the row quantizer inside the forward product (the bf16
# tiles are quantized by the pair pipeline's converters).  Its result must be
# that of the chain it replaces, oracle.quantize_rows then oracle.fwd, bit for
# bit, and its scales those of the quantizer.

def _fused(bits, wp, offset=0):
    M, K = bits.shape
    buf = torch.zeros(M * K + offset + 8, dtype=torch.int16, device="cuda")
    x = buf[offset:offset + M * K].view(M, K).view(torch.bfloat16)
    x.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    C, s, inv = t3.t3_gemm_fwd_bf16(x, torch.from_numpy(wp).cuda())
    torch.cuda.synchronize()
    return C.cpu().numpy(), s.cpu().numpy(), inv.cpu().numpy()


def _inv_want(bits):
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(x).max(axis=1)
    with np.errstate(divide="ignore", over="ignore"):
        return np.where(amax > 0, np.float32(127) / amax, np.float32(0)).astype(np.float32)


@pytest.mark.parametrize("M,N,K", [(33, 272, 64), (300, 200, 1280), (257, 201, 192),
                                   (1000, 384, 4096)])
def test_fused_forward_matches_quantize_then_forward(M, N, K):
    g = t3_synth.rng(M * 3 + N + K)
    bits = _rows(g, M, K)
    bits[1] = 0                                    # a zero row: scale 0, codes 0
    bits[2] = _bf16_bits(np.full(K, 1e-37, np.float32) * np.sign(g.standard_normal(K)))
    bits[2, :5] = 0                                # 127 / amax overflows: codes +-127 and 0
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    C, s, inv = _fused(bits, wp)
    q, s_want = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(s.view(np.uint32), s_want.view(np.uint32))
    np.testing.assert_array_equal(inv.view(np.uint32), _inv_want(bits).view(np.uint32))
    np.testing.assert_array_equal(C, oracle.fwd(q, wp))


def test_fused_forward_ties_and_the_library_chain():
    """Rows whose products fall on .5 (ties to even) and the library's own
    unfused chain (t3_quantize_rows_bf16, then t3_gemm_fwd) giving the same C."""
    M, N, K = 96, 192, 128
    g = t3_synth.rng(55)
    vals = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 63.5, -63.5], np.float32)
    bits = _bf16_bits(g.choice(vals, size=(M, K)))
    bits[:, 0] = _bf16_bits(np.full(M, 127.0, np.float32))   # amax 127: inv = 1
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    C, s, _ = _fused(bits, wp)
    q, s_want = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(C, oracle.fwd(q, wp))
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q_lib, _ = t3.t3_quantize_rows_bf16(x)
    C_lib = t3.t3_gemm_fwd(q_lib, torch.from_numpy(wp).cuda(), K=K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C, C_lib.cpu().numpy())


def test_fused_forward_layer_shape():
    M, N, K = 16384, 3456, 1280
    g = t3_synth.rng(16384)
    bits = _bf16_bits((g.standard_normal((M, K)) * 3).astype(np.float32))
    wp = oracle.pack(t3_synth.ternary(g, (K, N)))
    C, s, _ = _fused(bits, wp)
    q, s_want = oracle.quantize_rows(bits)
    np.testing.assert_array_equal(s.view(np.uint32), s_want.view(np.uint32))
    np.testing.assert_array_equal(C, oracle.fwd(q, wp))


def test_fused_forward_rejects_shapes_it_does_not_take():
    lib = t3.load()
    f = lib.t3_gemm_fwd_bf16
    x = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    wp = torch.zeros((16, 32), dtype=torch.uint8, device="cuda")
    C = torch.empty((64, 16), dtype=torch.int32, device="cuda")
    sc = torch.empty(64, dtype=torch.float32, device="cuda")
    inv = torch.empty(64, dtype=torch.float32, device="cuda")
    P = lambda t: t.data_ptr()
    assert f(P(x), P(wp), P(C), P(sc), P(inv), 32, 16, 128, None) == t3.T3_EINVAL   # M <= 32
    assert f(P(x), P(wp), P(C), P(sc), P(inv), 64, 16, 96, None) == t3.T3_EINVAL    # K % 64
    assert f(P(x) + 2, P(wp), P(C), P(sc), P(inv), 63, 16, 128, None) == t3.T3_EINVAL  # X unaligned
