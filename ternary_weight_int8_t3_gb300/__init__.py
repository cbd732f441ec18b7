"""Python binding of the t3 C ABI (include/t3.h): argument marshalling only.

Every product runs in the CUDA kernels of ``libt3.so``; this module checks
dtypes, shapes and devices, allocates outputs with torch when the caller does
not pass them, and forwards raw pointers and the current CUDA stream.  There
is no fallback: if the library is missing or cannot load, every call raises.

Function names follow the C ABI:
  t3_pack_ternary(w)                       host packer, w int8 [K][N]
  t3_pack_ternary_device(w, wp=None)       the same on the GPU (w a CUDA tensor)
  t3_gemm_fwd(A, Wp, K=None, C=None)       C  = A . W        (int32 [M][N])
  t3_gemm_bwd_dx(dY, Wp, K, dX=None)       dX = dY . W^T     (int32 [M][K])
  t3_gemm_bwd_dw(A, dY, dW=None)           dW = A^T . dY     (int32 [K][N])
  t3_quantize_rows_bf16(x)                 (int8 q, per-row scale) from bf16 x
  t3_gemm_fwd_bf16(x, Wp)                  the quantizer fused into the forward
  t3_dequant_i32(x, kind, row_scale, col_scale, out=None)   scaled float/bf16 output
  t3_gemm_fwd_scaled / t3_gemm_bwd_dx_scaled / t3_gemm_bwd_dw_scaled
                                           the products with that output
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libt3.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "t3.h")

T3_OK, T3_EINVAL, T3_EVALUE, T3_EOVERFLOW, T3_ECUDA, T3_ETIMEOUT, T3_EDEVICE = 0, -1, -2, -3, -4, -5, -6
T3_OUT_F32, T3_OUT_BF16, T3_OUT_F32_ADD = 0, 1, 2

_lock = threading.Lock()
_lib = None


class T3Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def build(force: bool = False) -> str:
    """Compiles libt3.so for sm_103a (nvcc); returns its path."""
    from . import _build
    return _build.build(force=force)


def load():
    """Loads libt3.so (building it first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        if not _build.up_to_date():
            _build.build()
        lib = ctypes.CDLL(LIB_PATH)
        p, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.t3_pack_ternary.argtypes = [p, p, i64, i64]
        for name in ("t3_gemm_fwd", "t3_gemm_bwd_dx", "t3_gemm_bwd_dw"):
            f = getattr(lib, name)
            f.argtypes = [p, p, p, i64, i64, i64, p]
            f.restype = ctypes.c_int
        lib.t3_pack_ternary.restype = ctypes.c_int
        lib.t3_pack_ternary_device.argtypes = [p, p, i64, i64, p]
        lib.t3_pack_ternary_device.restype = ctypes.c_int
        lib.t3_quantize_rows_bf16.argtypes = [p, p, p, i64, i64, p]
        lib.t3_quantize_rows_bf16.restype = ctypes.c_int
        lib.t3_gemm_fwd_bf16.argtypes = [p, p, p, p, p, i64, i64, i64, p]
        lib.t3_gemm_fwd_bf16.restype = ctypes.c_int
        lib.t3_dequant_i32.argtypes = [p, p, i64, i64, p, p, ctypes.c_int, p]
        lib.t3_dequant_i32.restype = ctypes.c_int
        for name in ("t3_gemm_fwd_scaled", "t3_gemm_bwd_dx_scaled", "t3_gemm_bwd_dw_scaled"):
            f = getattr(lib, name)
            f.argtypes = [p, p, p, i64, i64, i64, p, p, ctypes.c_int, p, p]
            f.restype = ctypes.c_int
        lib.t3_gemm_bwd_dw_scaled_noalloc.argtypes = [p, p, p, i64, i64, i64, p, p, ctypes.c_int, p]
        lib.t3_gemm_bwd_dw_scaled_noalloc.restype = ctypes.c_int
        lib.t3_status_string.argtypes = [ctypes.c_int]
        lib.t3_status_string.restype = ctypes.c_char_p
        lib.t3_last_device_error.argtypes = [p, ctypes.POINTER(ctypes.c_int32)]
        lib.t3_last_device_error.restype = ctypes.c_int
        lib.t3_selftest_wait_timeout.argtypes = [i64, p]
        lib.t3_selftest_wait_timeout.restype = ctypes.c_int
        lib.t3_set_small_product_limit.argtypes = [i64]
        lib.t3_set_small_product_limit.restype = i64
        lib.t3_version.argtypes = []
        lib.t3_version.restype = ctypes.c_int
        _lib = lib
        return lib


def declared_functions() -> list[str]:
    """Names of the functions include/t3.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(t3_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return load().t3_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != T3_OK:
        raise T3Error(status, where)


# ------------------------------------------------------------------- host ---

def t3_pack_ternary(w) -> np.ndarray:
    """Packs ternary w (int8 [K][N], values in {-1,0,+1}; numpy or CPU tensor)
    into Wp (uint8 [N][ceil(K/4)]) with the library's host packer."""
    if hasattr(w, "detach"):
        w = w.detach().cpu().numpy()
    w = np.ascontiguousarray(w)
    if w.dtype != np.int8 or w.ndim != 2:
        raise TypeError("w must be a 2-D int8 array [K][N]")
    K, N = w.shape
    wp = np.empty((N, (K + 3) // 4), dtype=np.uint8)
    rc = load().t3_pack_ternary(ctypes.c_void_p(w.ctypes.data), ctypes.c_void_p(wp.ctypes.data),
                                K, N)
    _check(rc, "t3_pack_ternary")
    return wp


# ----------------------------------------------------------------- device ---

def _torch():
    import torch
    return torch


def _dev_ptr(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr() if t.numel() else 0)


def _stream(t, stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(s.cuda_stream)


def t3_pack_ternary_device(w, wp=None, stream=None):
    """Packs ternary w (CUDA int8 tensor [K][N]) into Wp (CUDA uint8
    [N][ceil(K/4)]) on the GPU, asynchronously on `stream`.  A value outside
    {-1, 0, +1} packs as 0 and is reported by t3_last_device_error."""
    torch = _torch()
    if not isinstance(w, torch.Tensor) or w.dim() != 2:
        raise TypeError("w must be a 2-D CUDA int8 tensor [K][N]")
    K, N = w.shape
    if wp is None:
        wp = torch.empty((N, (K + 3) // 4), dtype=torch.uint8, device=w.device)
    if tuple(wp.shape) != (N, (K + 3) // 4):
        raise ValueError(f"wp must be [{N}][{(K + 3) // 4}], got {tuple(wp.shape)}")
    rc = load().t3_pack_ternary_device(_dev_ptr(w, torch.int8, "w"), _dev_ptr(wp, torch.uint8, "wp"),
                                       K, N, _stream(w, stream))
    _check(rc, "t3_pack_ternary_device")
    return wp


def t3_gemm_fwd(A, Wp, K: int | None = None, C=None, stream=None):
    """C[m][n] = sum_k A[m][k] W[k][n].  A int8 [M][K], Wp uint8 [N][ceil(K/4)]."""
    torch = _torch()
    M, Ka = A.shape
    K = Ka if K is None else K
    if Ka != K:
        raise ValueError("A must be [M][K]")
    N = Wp.shape[0]
    if Wp.dim() != 2 or Wp.shape[1] != (K + 3) // 4:
        raise ValueError("Wp must be [N][ceil(K/4)]")
    if C is None:
        _dev_ptr(A, torch.int8, "A")
        C = torch.empty((M, N), dtype=torch.int32, device=A.device)
    elif tuple(C.shape) != (M, N):
        raise ValueError("C must be [M][N]")
    args = (_dev_ptr(A, torch.int8, "A"), _dev_ptr(Wp, torch.uint8, "Wp"),
            _dev_ptr(C, torch.int32, "C"))
    with torch.cuda.device(A.device):
        rc = load().t3_gemm_fwd(*args, M, N, K, _stream(A, stream))
    _check(rc, "t3_gemm_fwd")
    return C


def t3_gemm_bwd_dx(dY, Wp, K: int, dX=None, stream=None):
    """dX[m][k] = sum_n dY[m][n] W[k][n].  dY int8 [M][N], Wp uint8 [N][ceil(K/4)]."""
    torch = _torch()
    M, N = dY.shape
    if Wp.dim() != 2 or tuple(Wp.shape) != (N, (K + 3) // 4):
        raise ValueError("Wp must be [N][ceil(K/4)]")
    if dX is None:
        _dev_ptr(dY, torch.int8, "dY")
        dX = torch.empty((M, K), dtype=torch.int32, device=dY.device)
    elif tuple(dX.shape) != (M, K):
        raise ValueError("dX must be [M][K]")
    args = (_dev_ptr(dY, torch.int8, "dY"), _dev_ptr(Wp, torch.uint8, "Wp"),
            _dev_ptr(dX, torch.int32, "dX"))
    with torch.cuda.device(dY.device):
        rc = load().t3_gemm_bwd_dx(*args, M, N, K, _stream(dY, stream))
    _check(rc, "t3_gemm_bwd_dx")
    return dX


def t3_gemm_bwd_dw(A, dY, dW=None, stream=None):
    """dW[k][n] = sum_m A[m][k] dY[m][n].  A int8 [M][K], dY int8 [M][N]."""
    torch = _torch()
    M, K = A.shape
    if dY.shape[0] != M:
        raise ValueError("A and dY must have the same number of rows")
    N = dY.shape[1]
    if dW is None:
        _dev_ptr(A, torch.int8, "A")
        dW = torch.empty((K, N), dtype=torch.int32, device=A.device)
    elif tuple(dW.shape) != (K, N):
        raise ValueError("dW must be [K][N]")
    args = (_dev_ptr(A, torch.int8, "A"), _dev_ptr(dY, torch.int8, "dY"),
            _dev_ptr(dW, torch.int32, "dW"))
    with torch.cuda.device(A.device):
        rc = load().t3_gemm_bwd_dw(*args, M, N, K, _stream(A, stream))
    _check(rc, "t3_gemm_bwd_dw")
    return dW


# ------------------------------------------------------------ scaled outputs

def _scaled_out(out, kind, rows, cols, device, name):
    torch = _torch()
    dtype = torch.bfloat16 if kind == T3_OUT_BF16 else torch.float32
    if kind not in (T3_OUT_F32, T3_OUT_BF16, T3_OUT_F32_ADD):
        raise ValueError(f"unknown output kind {kind}")
    if out is None:
        if kind == T3_OUT_F32_ADD:
            raise ValueError(f"{name}: the += kind needs the existing output")
        out = torch.empty((rows, cols), dtype=dtype, device=device)
    if tuple(out.shape) != (rows, cols):
        raise ValueError(f"{name} must be [{rows}][{cols}]")
    return out, _dev_ptr(out, dtype, name)


def _scale_ptr(v, n, name):
    if v is None:
        return ctypes.c_void_p(0)
    if v.dim() != 1 or v.shape[0] != n:
        raise ValueError(f"{name} must have {n} entries")
    return _dev_ptr(v, _torch().float32, name)


def _ws_ptr(ws, rows, cols):
    if ws is None:
        return ctypes.c_void_p(0)
    if tuple(ws.shape) != (rows, cols):
        raise ValueError(f"workspace must be [{rows}][{cols}]")
    return _dev_ptr(ws, _torch().int32, "workspace")


def t3_quantize_rows_bf16(x, q=None, row_scale=None, stream=None):
    """(q, row_scale): bf16 x [M][K] quantized to int8 with one absmax scale
    per row (see include/t3.h)."""
    torch = _torch()
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise TypeError("x must be a 2-D CUDA bfloat16 tensor [M][K]")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if row_scale is None:
        row_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    if tuple(q.shape) != (M, K) or tuple(row_scale.shape) != (M,):
        raise ValueError("q must be [M][K] and row_scale [M]")
    args = (_dev_ptr(x, torch.bfloat16, "x"), _dev_ptr(q, torch.int8, "q"),
            _dev_ptr(row_scale, torch.float32, "row_scale"), M, K, _stream(x, stream))
    with torch.cuda.device(x.device):
        rc = load().t3_quantize_rows_bf16(*args)
    _check(rc, "t3_quantize_rows_bf16")
    return q, row_scale


def t3_gemm_fwd_bf16(x, Wp, C=None, row_scale=None, row_inv=None, stream=None):
    """(C, row_scale, row_inv): the forward product of the row-quantized bf16
    activations x [M][K] with the packed weights Wp [N][ceil(K/4)], the
    quantizer fused into the product (see include/t3.h); C int32 [M][N]."""
    torch = _torch()
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise TypeError("x must be a 2-D CUDA bfloat16 tensor [M][K]")
    M, K = x.shape
    N = Wp.shape[0]
    if Wp.dim() != 2 or Wp.shape[1] != (K + 3) // 4:
        raise ValueError("Wp must be [N][ceil(K/4)]")
    if C is None:
        C = torch.empty((M, N), dtype=torch.int32, device=x.device)
    if row_scale is None:
        row_scale = torch.empty((M,), dtype=torch.float32, device=x.device)
    if row_inv is None:
        row_inv = torch.empty((M,), dtype=torch.float32, device=x.device)
    if tuple(C.shape) != (M, N) or tuple(row_scale.shape) != (M,) or tuple(row_inv.shape) != (M,):
        raise ValueError("C must be [M][N], row_scale and row_inv [M]")
    args = (_dev_ptr(x, torch.bfloat16, "x"), _dev_ptr(Wp, torch.uint8, "Wp"),
            _dev_ptr(C, torch.int32, "C"), _dev_ptr(row_scale, torch.float32, "row_scale"),
            _dev_ptr(row_inv, torch.float32, "row_inv"), M, N, K, _stream(x, stream))
    with torch.cuda.device(x.device):
        rc = load().t3_gemm_fwd_bf16(*args)
    _check(rc, "t3_gemm_fwd_bf16")
    return C, row_scale, row_inv


def t3_dequant_i32(x, kind=T3_OUT_F32, row_scale=None, col_scale=None, out=None, stream=None):
    """out = ((float)x * row_scale[r]) * col_scale[c] as float (T3_OUT_F32),
    bf16 (T3_OUT_BF16) or added to `out` (T3_OUT_F32_ADD).  x int32 [R][C]."""
    torch = _torch()
    rows, cols = x.shape
    out, po = _scaled_out(out, kind, rows, cols, x.device, "out")
    args = (_dev_ptr(x, torch.int32, "x"), po, rows, cols, _scale_ptr(row_scale, rows, "row_scale"),
            _scale_ptr(col_scale, cols, "col_scale"), kind, _stream(x, stream))
    with torch.cuda.device(x.device):
        rc = load().t3_dequant_i32(*args)
    _check(rc, "t3_dequant_i32")
    return out


def t3_gemm_fwd_scaled(A, Wp, K=None, row_scale=None, col_scale=None, kind=T3_OUT_F32, C=None,
                       workspace=None, stream=None):
    """C (scaled, float or bf16 [M][N]) of A . W; row_scale [M], col_scale [N]."""
    torch = _torch()
    M, Ka = A.shape
    K = Ka if K is None else K
    if Ka != K:
        raise ValueError("A must be [M][K]")
    N = Wp.shape[0]
    if Wp.dim() != 2 or Wp.shape[1] != (K + 3) // 4:
        raise ValueError("Wp must be [N][ceil(K/4)]")
    C, pc = _scaled_out(C, kind, M, N, A.device, "C")
    args = (_dev_ptr(A, torch.int8, "A"), _dev_ptr(Wp, torch.uint8, "Wp"), pc, M, N, K,
            _scale_ptr(row_scale, M, "row_scale"), _scale_ptr(col_scale, N, "col_scale"), kind,
            _ws_ptr(workspace, M, N), _stream(A, stream))
    with torch.cuda.device(A.device):
        rc = load().t3_gemm_fwd_scaled(*args)
    _check(rc, "t3_gemm_fwd_scaled")
    return C


def t3_gemm_bwd_dx_scaled(dY, Wp, K: int, row_scale=None, col_scale=None, kind=T3_OUT_F32,
                          dX=None, workspace=None, stream=None):
    """dX (scaled, float or bf16 [M][K]) of dY . W^T; row_scale [M], col_scale [K]."""
    torch = _torch()
    M, N = dY.shape
    if Wp.dim() != 2 or tuple(Wp.shape) != (N, (K + 3) // 4):
        raise ValueError("Wp must be [N][ceil(K/4)]")
    dX, px = _scaled_out(dX, kind, M, K, dY.device, "dX")
    args = (_dev_ptr(dY, torch.int8, "dY"), _dev_ptr(Wp, torch.uint8, "Wp"), px, M, N, K,
            _scale_ptr(row_scale, M, "row_scale"), _scale_ptr(col_scale, K, "col_scale"), kind,
            _ws_ptr(workspace, M, K), _stream(dY, stream))
    with torch.cuda.device(dY.device):
        rc = load().t3_gemm_bwd_dx_scaled(*args)
    _check(rc, "t3_gemm_bwd_dx_scaled")
    return dX


def t3_gemm_bwd_dw_scaled(A, dY, row_scale=None, col_scale=None, kind=T3_OUT_F32, dW=None,
                          workspace=None, stream=None):
    """dW (scaled, float or bf16 [K][N]) of A^T . dY; row_scale [K] (A's column
    scales), col_scale [N] (dY's column scales)."""
    torch = _torch()
    M, K = A.shape
    if dY.shape[0] != M:
        raise ValueError("A and dY must have the same number of rows")
    N = dY.shape[1]
    dW, pw = _scaled_out(dW, kind, K, N, A.device, "dW")
    args = (_dev_ptr(A, torch.int8, "A"), _dev_ptr(dY, torch.int8, "dY"), pw, M, N, K,
            _scale_ptr(row_scale, K, "row_scale"), _scale_ptr(col_scale, N, "col_scale"), kind,
            _ws_ptr(workspace, K, N), _stream(A, stream))
    with torch.cuda.device(A.device):
        rc = load().t3_gemm_bwd_dw_scaled(*args)
    _check(rc, "t3_gemm_bwd_dw_scaled")
    return dW


def t3_gemm_bwd_dw_scaled_noalloc(A, dY, row_scale=None, col_scale=None, kind=T3_OUT_F32,
                                  dW=None, stream=None):
    """t3_gemm_bwd_dw_scaled with the int32 intermediate in the library's fixed
    per-device buffer (K * N <= 8,388,608; calls on one device must not overlap)."""
    torch = _torch()
    M, K = A.shape
    if dY.shape[0] != M:
        raise ValueError("A and dY must have the same number of rows")
    N = dY.shape[1]
    dW, pw = _scaled_out(dW, kind, K, N, A.device, "dW")
    args = (_dev_ptr(A, torch.int8, "A"), _dev_ptr(dY, torch.int8, "dY"), pw, M, N, K,
            _scale_ptr(row_scale, K, "row_scale"), _scale_ptr(col_scale, N, "col_scale"), kind,
            _stream(A, stream))
    with torch.cuda.device(A.device):
        rc = load().t3_gemm_bwd_dw_scaled_noalloc(*args)
    _check(rc, "t3_gemm_bwd_dw_scaled_noalloc")
    return dW


def t3_last_device_error(stream=None):
    """(status, detail): T3_ETIMEOUT and the recorded code if a bounded device
    wait gave up since the last call; synchronizes the stream."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    detail = ctypes.c_int32(0)
    rc = load().t3_last_device_error(ctypes.c_void_p(s.cuda_stream), ctypes.byref(detail))
    return rc, detail.value


def t3_set_small_product_limit(macs: int) -> int:
    """Products of at most `macs` multiply-adds (macs / 8 when every operand's
    rows are 4-byte aligned) run on the CUDA cores, larger ones on the tensor
    cores (default 2**29; 0: always the tensor cores).  Returns the previous
    limit."""
    return int(load().t3_set_small_product_limit(int(macs)))


def t3_selftest_wait_timeout(limit_ns: int, stream=None):
    """Launches the bounded-wait self-test: one CTA waits on a barrier that
    nothing completes and gives up after limit_ns of device time, recording
    its code for t3_last_device_error."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(load().t3_selftest_wait_timeout(int(limit_ns), ctypes.c_void_p(s.cuda_stream)),
           "t3_selftest_wait_timeout")


def t3_version() -> int:
    return load().t3_version()
