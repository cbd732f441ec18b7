"""TEST INFRASTRUCTURE ONLY: the plain CPU oracle for the ternary x int8 GEMMs.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product library never does, and this package
imports nothing from it.

The arithmetic lives in ``t3_oracle.c`` (plain C, int64 sums, table decode);
this module compiles it with the host C compiler and wraps it with numpy
arrays.  What each function follows on the pages is cited in the C source:

* "t27c PTX backend: ternary x int8 GEMM kernel emitted by a .t27 spec (int8
  mma.sync), ptx-run glue", section "What this adds" -- forward product, the
  2-bit decode formula, the row reference.
* "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as int8 tensor-core PTX
  written by t27", kernel 1 (dX) and kernel 2 (dW).

The scaled outputs (``dequant``, ``bf16_bits``) are written here in numpy
float32 arithmetic, which rounds every conversion, product and sum to the
nearest float (ties to even), as their definition asks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "t3_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EVALUE, EOVERFLOW = 0, -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compiles t3_oracle.c into liboracle.so (gcc, OpenMP when available)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # T3_ORACLE_LIB names a deliberately broken copy of the oracle, used
            # only by the mutation test that checks the pins catch mistakes.
            path = os.environ.get("T3_ORACLE_LIB")
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            p, i64 = ctypes.c_void_p, ctypes.c_int64
            for name in ("oracle_fwd", "oracle_dx", "oracle_dw"):
                f = getattr(lib, name)
                f.argtypes = [p, p, p, i64, i64, i64]
                f.restype = ctypes.c_int
            for name in ("oracle_fwd_rows", "oracle_dx_rows", "oracle_dw_rows"):
                f = getattr(lib, name)
                f.argtypes = [p, p, p, i64, i64, i64, p, i64]
                f.restype = ctypes.c_int
            lib.oracle_pack.argtypes = [p, p, i64, i64]
            lib.oracle_pack.restype = ctypes.c_int
            lib.oracle_unpack.argtypes = [p, p, i64, i64]
            lib.oracle_unpack.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what} failed with status {rc}")


def _c_int8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.int8:
        raise TypeError(f"expected int8, got {a.dtype}")
    return a


def packed_row_bytes(K: int) -> int:
    return (K + 3) // 4


def decode(code: int) -> int:
    """Weight of one 2-bit code (table {0, +1, -1, 0})."""
    return _load().oracle_decode(int(code))


def pack(w) -> np.ndarray:
    """w: int8 [K][N] in {-1,0,+1} -> Wp uint8 [N][ceil(K/4)]."""
    w = _c_int8(w)
    K, N = w.shape
    wp = np.zeros((N, packed_row_bytes(K)), dtype=np.uint8)
    _check(_load().oracle_pack(_ptr(w), _ptr(wp), K, N), "oracle_pack")
    return wp


def pack_status(w) -> int:
    """Status code of packing w (OK or EVALUE), for the error-path tests."""
    w = _c_int8(w)
    K, N = w.shape
    wp = np.zeros((N, packed_row_bytes(K)), dtype=np.uint8)
    return _load().oracle_pack(_ptr(w), _ptr(wp), K, N)


def unpack(wp, K: int) -> np.ndarray:
    """Wp uint8 [N][ceil(K/4)] -> W int8 [K][N]."""
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    N = wp.shape[0]
    assert wp.shape == (N, packed_row_bytes(K))
    w = np.zeros((K, N), dtype=np.int8)
    _check(_load().oracle_unpack(_ptr(wp), _ptr(w), K, N), "oracle_unpack")
    return w


def _rows_arg(rows, total):
    if rows is None:
        return None, total
    r = np.ascontiguousarray(rows, dtype=np.int64)
    return r, r.size


def fwd(A, Wp, rows=None) -> np.ndarray:
    """C = A . W.  A int8 [M][K]; Wp [N][ceil(K/4)].  Returns int32 [len(rows) or M][N]."""
    A = _c_int8(A)
    M, K = A.shape
    Wp = np.ascontiguousarray(Wp, dtype=np.uint8)
    N = Wp.shape[0]
    assert Wp.shape == (N, packed_row_bytes(K))
    r, nr = _rows_arg(rows, M)
    C = np.zeros((nr, N), dtype=np.int32)
    rc = _load().oracle_fwd_rows(_ptr(A), _ptr(Wp), _ptr(C), M, N, K,
                                 None if r is None else _ptr(r), nr)
    _check(rc, "oracle_fwd")
    return C


def dx(dY, Wp, K: int, rows=None) -> np.ndarray:
    """dX = dY . W^T.  dY int8 [M][N]; Wp [N][ceil(K/4)].  Returns int32 [rows][K]."""
    dY = _c_int8(dY)
    M, N = dY.shape
    Wp = np.ascontiguousarray(Wp, dtype=np.uint8)
    assert Wp.shape == (N, packed_row_bytes(K))
    r, nr = _rows_arg(rows, M)
    dX = np.zeros((nr, K), dtype=np.int32)
    rc = _load().oracle_dx_rows(_ptr(dY), _ptr(Wp), _ptr(dX), M, N, K,
                                None if r is None else _ptr(r), nr)
    _check(rc, "oracle_dx")
    return dX


def dw(A, dY, rows=None) -> np.ndarray:
    """dW = A^T . dY.  A int8 [M][K]; dY int8 [M][N].  Returns int32 [rows of K][N]."""
    A = _c_int8(A)
    dY = _c_int8(dY)
    M, K = A.shape
    assert dY.shape[0] == M
    N = dY.shape[1]
    r, nr = _rows_arg(rows, K)
    dW = np.zeros((nr, N), dtype=np.int32)
    rc = _load().oracle_dw_rows(_ptr(A), _ptr(dY), _ptr(dW), M, N, K,
                                None if r is None else _ptr(r), nr)
    _check(rc, "oracle_dw")
    return dW


OUT_F32, OUT_BF16, OUT_F32_ADD = 0, 1, 2


def bf16_bits(y) -> np.ndarray:
    """float32 values -> bf16 bit patterns (uint16), rounded to nearest, ties
    to even: add half an ulp of the kept 16 bits (0x7FFF, plus the kept
    lowest bit for ties) and keep the high half.  Finite inputs."""
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def dequant(x, row_scale=None, col_scale=None, kind: int = OUT_F32, out=None) -> np.ndarray:
    """The scaled output of an exact int32 result x [rows][cols]: the step after
    the products in "spec(igla): hslm_bwd_ptx -- HSLM backward dX and dW as
    int8 tensor-core PTX written by t27", where the host rescales the integer
    results (dX per row, dW per column of X and of dY) and the products have
    "+=" forms.  y = ((float)x * row_scale[r]) * col_scale[c], every step a
    float32 operation; None scales are ones.  Returns y (OUT_F32), its bf16
    bit patterns (OUT_BF16), or out + y (OUT_F32_ADD, `out` the old float32
    values)."""
    x = np.asarray(x, dtype=np.int32)
    rows, cols = x.shape
    rs = np.ones(rows, np.float32) if row_scale is None else np.asarray(row_scale, np.float32)
    cs = np.ones(cols, np.float32) if col_scale is None else np.asarray(col_scale, np.float32)
    y = x.astype(np.float32) * rs[:, None]
    y = y * cs[None, :]
    if kind == OUT_F32:
        return y
    if kind == OUT_BF16:
        return bf16_bits(y)
    if kind == OUT_F32_ADD:
        return np.asarray(out, dtype=np.float32) + y
    raise ValueError(f"unknown output kind {kind}")


def quantize_rows(x_bits):
    """bf16 activations (bit patterns, uint16 [M][K]) -> (int8 q [M][K], float32
    scale [M]): the step before the products, symmetric absmax per row (the
    second page names per-row scales for dX but gives no quantizer).
    amax = max |x|; scale = amax / 127 and inv = 127 / amax as float32
    divisions; q = rint(x * inv) with the product rounded to float32 and rint
    to nearest, ties to even, clamped to [-127, 127]; zero rows give q = 0,
    scale = 0; a product 0 * inf counts as 0."""
    u = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = u.shape
    x = (u.astype(np.uint32) << 16).view(np.float32)
    amax = np.abs(x).max(axis=1) if K else np.zeros(M, np.float32)
    pos = amax > 0
    safe = np.where(pos, amax, np.float32(1))
    scale = np.where(pos, safe / np.float32(127), np.float32(0)).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        inv = np.where(pos, np.float32(127) / safe, np.float32(0)).astype(np.float32)
        prod = x * inv[:, None]
    prod = np.where(np.isnan(prod), np.float32(0), prod)
    q = np.clip(np.rint(prod), -127, 127).astype(np.int8)
    return q, scale


def num_threads() -> int:
    """Threads the oracle's OpenMP loops run on."""
    return _load().oracle_num_threads()
