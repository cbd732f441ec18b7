"""GPU parity of the scaled outputs against the oracle, bit for bit:
t3_dequant_i32 and the three products with float / bf16 / float "+=" output.

Expected values are the oracle's exact integer products passed through the
oracle's dequant (float32 steps, bf16 rounding to nearest even).  Shapes are
chosen so that both routes run: the pair pipeline's scaling epilogue (fwd with
M > 32 and dX, aligned output rows) and the exact int32 product followed by
the dequantization (small M, rows that are not 16-byte aligned, dW, K = 0).
"""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KINDS = [t3.T3_OUT_F32, t3.T3_OUT_BF16, t3.T3_OUT_F32_ADD]


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    t3.load()
    yield
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set, detail={detail:#x}"


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _scales(g, n, which):
    if not which:
        return None, None
    v = (g.standard_normal(n) * 0.01).astype(np.float32)
    v[::7] *= -1.0  # negative scales, and with them signed zeros
    return v, _dev(v)


def _old(g, rows, cols):
    o = (g.standard_normal((rows, cols)) * 100).astype(np.float32)
    return o, _dev(o)


def _host_bits(t, kind):
    if kind == t3.T3_OUT_BF16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def _want_bits(x, rs, cs, kind, old):
    y = oracle.dequant(x, rs, cs, kind, old)
    return y if kind == t3.T3_OUT_BF16 else np.ascontiguousarray(y, np.float32).view(np.uint32)


def _run_scaled(call, rows, cols, kind, g, rs_d, cs_d, workspace):
    old, out = (None, None)
    if kind == t3.T3_OUT_F32_ADD:
        old, out = _old(g, rows, cols)
    ws = torch.empty((rows, cols), dtype=torch.int32, device="cuda") if workspace else None
    res = call(rs_d, cs_d, kind, out, ws)
    torch.cuda.synchronize()
    return res, old


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (7, 12), (64, 128), (129, 1001), (300, 272)])
@pytest.mark.parametrize("kind", KINDS)
def test_dequant_matches_oracle(rows, cols, kind):
    g = t3_synth.rng(rows * 31 + cols + kind)
    x = g.integers(-2 ** 31, 2 ** 31, (rows, cols), dtype=np.int64).astype(np.int32)
    if x.size >= 3:
        x.flat[:3] = [0, 16777217, -16777219]  # a zero and two conversions that round
    rs, rs_d = _scales(g, rows, True)
    cs, cs_d = _scales(g, cols, cols % 2 == 0)
    old, out = (None, None)
    if kind == t3.T3_OUT_F32_ADD:
        old, out = _old(g, rows, cols)
    res = t3.t3_dequant_i32(_dev(x), kind, rs_d, cs_d, out=out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(res, kind), _want_bits(x, rs, cs, kind, old))


def test_dequant_in_place_float():
    g = t3_synth.rng(91)
    x = g.integers(-2 ** 31, 2 ** 31, (33, 64), dtype=np.int64).astype(np.int32)
    rs, rs_d = _scales(g, 33, True)
    buf = _dev(x)
    out = buf.view(torch.float32)
    t3.t3_dequant_i32(buf, t3.T3_OUT_F32, rs_d, None, out=out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(out, t3.T3_OUT_F32), _want_bits(x, rs, None, 0, None))
    lib = t3.load()
    p = buf.data_ptr()
    assert lib.t3_dequant_i32(p, p, 33, 64, None, None, t3.T3_OUT_BF16, None) == t3.T3_EINVAL


FWD_SHAPES = [(300, 272, 96),   # pair pipeline, scaling epilogue
              (300, 271, 96),   # float rows not 16-byte aligned: exact int32, then dequant
              (8, 272, 96),     # small M: exact int32, then dequant
              (257, 400, 1280)]


@pytest.mark.parametrize("M,N,K", FWD_SHAPES)
@pytest.mark.parametrize("kind", KINDS)
def test_forward_scaled(M, N, K, kind):
    g = t3_synth.rng(M + N + K + kind)
    A = t3_synth.int8_uniform(g, (M, K))
    w = t3_synth.ternary(g, (K, N))
    wp = oracle.pack(w)
    rs, rs_d = _scales(g, M, True)
    cs, cs_d = _scales(g, N, True)
    A_d, wp_d = _dev(A), _dev(wp)
    res, old = _run_scaled(
        lambda r, c, k, o, ws: t3.t3_gemm_fwd_scaled(A_d, wp_d, K, r, c, k, C=o, workspace=ws),
        M, N, kind, g, rs_d, cs_d, workspace=True)
    np.testing.assert_array_equal(_host_bits(res, kind),
                                  _want_bits(oracle.fwd(A, wp), rs, cs, kind, old))


@pytest.mark.parametrize("M,N,K", [(300, 96, 272), (300, 96, 97), (40, 1280, 3456)])
@pytest.mark.parametrize("kind", KINDS)
def test_dx_scaled(M, N, K, kind):
    g = t3_synth.rng(7 * M + N + K + kind)
    dY = t3_synth.int8_uniform(g, (M, N))
    w = t3_synth.ternary(g, (K, N))
    wp = oracle.pack(w)
    rs, rs_d = _scales(g, M, True)
    cs, cs_d = _scales(g, K, kind != t3.T3_OUT_F32)
    dY_d, wp_d = _dev(dY), _dev(wp)
    res, old = _run_scaled(
        lambda r, c, k, o, ws: t3.t3_gemm_bwd_dx_scaled(dY_d, wp_d, K, r, c, k, dX=o, workspace=ws),
        M, K, kind, g, rs_d, cs_d, workspace=True)
    np.testing.assert_array_equal(_host_bits(res, kind),
                                  _want_bits(oracle.dx(dY, wp, K), rs, cs, kind, old))


@pytest.mark.parametrize("M,N,K", [(300, 272, 96), (1782, 256, 128)])
@pytest.mark.parametrize("kind", KINDS)
def test_dw_scaled(M, N, K, kind):
    g = t3_synth.rng(3 * M + N + K + kind)
    A = t3_synth.int8_uniform(g, (M, K))
    dY = t3_synth.int8_uniform(g, (M, N))
    rs, rs_d = _scales(g, K, True)
    cs, cs_d = _scales(g, N, True)
    A_d, dY_d = _dev(A), _dev(dY)
    res, old = _run_scaled(
        lambda r, c, k, o, ws: t3.t3_gemm_bwd_dw_scaled(A_d, dY_d, r, c, k, dW=o, workspace=ws),
        K, N, kind, g, rs_d, cs_d, workspace=(kind != t3.T3_OUT_F32))
    np.testing.assert_array_equal(_host_bits(res, kind),
                                  _want_bits(oracle.dw(A, dY), rs, cs, kind, old))


def test_scaled_float_without_workspace_converts_in_place():
    g = t3_synth.rng(5)
    A = t3_synth.int8_uniform(g, (8, 96))
    wp = oracle.pack(t3_synth.ternary(g, (96, 272)))
    rs, rs_d = _scales(g, 8, True)
    C = t3.t3_gemm_fwd_scaled(_dev(A), _dev(wp), 96, rs_d, None, t3.T3_OUT_F32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(C, 0), _want_bits(oracle.fwd(A, wp), rs, None, 0, None))


def test_scaled_needs_workspace_for_bf16_and_add_off_the_epilogue():
    g = t3_synth.rng(6)
    A = _dev(t3_synth.int8_uniform(g, (8, 96)))   # small M: no scaling epilogue
    wp = _dev(oracle.pack(t3_synth.ternary(g, (96, 272))))
    with pytest.raises(t3.T3Error):
        t3.t3_gemm_fwd_scaled(A, wp, 96, None, None, t3.T3_OUT_BF16)
    out = torch.zeros((8, 272), dtype=torch.float32, device="cuda")
    with pytest.raises(t3.T3Error):
        t3.t3_gemm_fwd_scaled(A, wp, 96, None, None, t3.T3_OUT_F32_ADD, C=out)


def test_scaled_empty_reduction_gives_scaled_zeros():
    g = t3_synth.rng(8)
    A = torch.zeros((300, 0), dtype=torch.int8, device="cuda")
    wp = torch.zeros((272, 0), dtype=torch.uint8, device="cuda")
    rs, rs_d = _scales(g, 300, True)
    C = t3.t3_gemm_fwd_scaled(A, wp, 0, rs_d, None, t3.T3_OUT_F32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_host_bits(C, 0),
                                  _want_bits(np.zeros((300, 272), np.int32), rs, None, 0, None))


def test_layer_shape_scaled_sampled_rows():
    wl = t3_synth.BY_NAME["fwd_16384x3456x1280"]
    A, w, dY = t3_synth.make_inputs(wl)
    M, K = A.shape
    N = w.shape[1]
    wp = oracle.pack(w)
    g = t3_synth.rng(12)
    rs, rs_d = _scales(g, M, True)
    cs, cs_d = _scales(g, N, True)
    rows = np.array([0, 1, 255, 256, 8191, 16383])
    C = t3.t3_gemm_fwd_scaled(_dev(A), _dev(wp), K, rs_d, cs_d, t3.T3_OUT_BF16)
    dX = t3.t3_gemm_bwd_dx_scaled(_dev(dY), _dev(wp), K, rs_d, None, t3.T3_OUT_F32)
    torch.cuda.synchronize()
    c_rows = oracle.fwd(A, wp, rows)
    np.testing.assert_array_equal(_host_bits(C, 1)[rows], _want_bits(c_rows, rs[rows], cs, 1, None))
    x_rows = oracle.dx(dY, wp, K, rows)
    np.testing.assert_array_equal(_host_bits(dX, 0)[rows], _want_bits(x_rows, rs[rows], None, 0, None))
