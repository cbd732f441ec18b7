"""t3_gemm_bwd_dw_scaled_noalloc: the scaled dW product with its int32
intermediate in the library's fixed per-device buffer instead of a caller
workspace.  GPU parity against the oracle (every output kind, repeated calls
that reuse the buffer, the layer's dW size) and the size limit, which is
checked before any CUDA call.  Collected last (file name)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")

CAPACITY = 8 * 1024 * 1024  # int32 entries of the fixed buffer


def test_noalloc_rejects_dw_larger_than_its_buffer_before_any_cuda_call():
    lib = t3.load()
    f = lib.t3_gemm_bwd_dw_scaled_noalloc
    # K * N one past the buffer, and far past it; null pointers are never read
    assert f(None, None, None, 4, CAPACITY // 1024 + 1, 1024, None, None, t3.T3_OUT_BF16, None) == t3.T3_EINVAL
    assert f(None, None, None, 4, 8192, 8192, None, None, t3.T3_OUT_F32, None) == t3.T3_EINVAL
    assert f(None, None, None, 4, 8, 8, None, None, 7, None) == t3.T3_EINVAL      # unknown kind
    assert f(None, None, None, -1, 8, 8, None, None, 0, None) == t3.T3_EINVAL     # negative size
    assert f(None, None, None, 4, 0, 8, None, None, 0, None) == t3.T3_OK          # empty output


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bits(t, kind):
    if kind == t3.T3_OUT_BF16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def _want(x, rs, cs, kind, old):
    y = oracle.dequant(x, rs, cs, kind, old)
    return y if kind == t3.T3_OUT_BF16 else np.ascontiguousarray(y, np.float32).view(np.uint32)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", [t3.T3_OUT_F32, t3.T3_OUT_BF16, t3.T3_OUT_F32_ADD])
def test_noalloc_dw_matches_oracle_and_reuses_its_buffer(kind):
    for M, N, K, seed in [(300, 272, 96, 1), (1782, 256, 128, 2), (33, 80, 64, 3)]:
        g = t3_synth.rng(100 * seed + kind)
        A = t3_synth.int8_uniform(g, (M, K))
        dY = t3_synth.int8_uniform(g, (M, N))
        rs = (g.standard_normal(K) * 0.01).astype(np.float32)
        cs = (g.standard_normal(N) * 0.01).astype(np.float32)
        old, out = None, None
        if kind == t3.T3_OUT_F32_ADD:
            old = (g.standard_normal((K, N)) * 10).astype(np.float32)
            out = _dev(old)
        res = t3.t3_gemm_bwd_dw_scaled_noalloc(_dev(A), _dev(dY), _dev(rs), _dev(cs), kind, dW=out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(res, kind), _want(oracle.dw(A, dY), rs, cs, kind, old))
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set, detail={detail:#x}"


@pytest.mark.gpu
def test_noalloc_dw_layer_size_sampled_rows():
    wl = t3_synth.BY_NAME["fwd_16384x3456x1280"]
    A, w, dY = t3_synth.make_inputs(wl)
    K, N = A.shape[1], dY.shape[1]
    assert K * N <= CAPACITY
    g = t3_synth.rng(77)
    rs = (g.standard_normal(K) * 0.01).astype(np.float32)
    cs = (g.standard_normal(N) * 0.01).astype(np.float32)
    res = t3.t3_gemm_bwd_dw_scaled_noalloc(_dev(A), _dev(dY), _dev(rs), _dev(cs), t3.T3_OUT_BF16)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 1279])
    x = oracle.dw(A, dY, rows)
    np.testing.assert_array_equal(_bits(res, 1)[rows], _want(x, rs[rows], cs, 1, None))
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set, detail={detail:#x}"


_RESIDENCY_PROBE = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch
import ternary_weight_int8_t3_gb300 as t3
t3.load()
dev = torch.device("cuda")
A = torch.zeros((64, 128), dtype=torch.int8, device=dev)
wp = torch.zeros((256, 32), dtype=torch.uint8, device=dev)
C = torch.empty((64, 256), dtype=torch.int32, device=dev)
dY = torch.zeros((64, 256), dtype=torch.int8, device=dev)
dW = torch.empty((128, 256), dtype=torch.float32, device=dev)
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
t3.t3_gemm_fwd(A, wp, K=128, C=C)
t3.t3_gemm_bwd_dw_scaled(A, dY, None, None, t3.T3_OUT_F32, dW=dW)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
t3.t3_gemm_bwd_dw_scaled_noalloc(A, dY, None, None, t3.T3_OUT_F32, dW=dW)
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
print(json.dumps({"other_calls": free0 - free1, "first_noalloc_call": free1 - free2}))
"""


@pytest.mark.gpu
def test_noalloc_buffer_is_reserved_only_by_its_own_callers():
    """In a fresh process with lazy module loading, the first fwd and scaled
    dW calls (which use the same kernels as the no-alloc entry point) do not
    reserve the fixed buffer's 32 MiB; the first no-alloc call does."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    out = subprocess.run([sys.executable, "-c", _RESIDENCY_PROBE, root], env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    got = json.loads(out.stdout.strip().splitlines()[-1])
    mib = 1024 * 1024
    assert got["other_calls"] < 32 * mib, got
    assert got["first_noalloc_call"] >= 32 * mib, got
