"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/t3.h declares, packs like the oracle, and rejects bad
arguments before touching the GPU.  No compute call runs here."""
import ctypes
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return t3.load()


def test_every_declared_symbol_is_exported(lib):
    names = t3.declared_functions()
    assert set(names) >= {"t3_pack_ternary", "t3_gemm_fwd", "t3_gemm_bwd_dx", "t3_gemm_bwd_dw",
                          "t3_status_string", "t3_last_device_error", "t3_version"}
    for name in names:
        assert hasattr(lib, name), name


def test_library_has_no_oracle_or_cpu_fallback():
    pkg = os.path.join(ROOT, "ternary_weight_int8_t3_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "t3_oracle" not in text and "oracle_" not in text, f


def test_selftest_rejects_limits_out_of_range_before_any_cuda_call(lib):
    f = lib.t3_selftest_wait_timeout
    for limit in (-1, 0, 999, 2_000_000_001, 1 << 40):
        assert f(limit, None) == t3.T3_EINVAL


def test_small_product_limit_round_trips_without_a_gpu(lib):
    prev = t3.t3_set_small_product_limit(12345)
    try:
        assert prev >= 0
        assert t3.t3_set_small_product_limit(-7) == 12345
        assert t3.t3_set_small_product_limit(1 << 29) == 0  # negative counts as 0
    finally:
        t3.t3_set_small_product_limit(prev)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = t3.status_string(code)
        assert s.startswith("T3_"), s
    assert t3.status_string(12345) == "unknown t3 status"
    assert t3.t3_version() >= 100


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 7, 8, 13, 64, 96, 255, 1280])
def test_pack_matches_oracle(K):
    g = t3_synth.rng(K)
    for N in (1, 3, 272):
        w = t3_synth.ternary(g, (K, N))
        assert np.array_equal(t3.t3_pack_ternary(w), oracle.pack(w))


def test_pack_rejects_bad_values_and_writes_nothing(lib):
    w = np.zeros((9, 4), dtype=np.int8)
    w[8, 3] = -2
    wp = np.full((4, 3), 0xAB, dtype=np.uint8)
    rc = lib.t3_pack_ternary(ctypes.c_void_p(w.ctypes.data), ctypes.c_void_p(wp.ctypes.data), 9, 4)
    assert rc == t3.T3_EVALUE
    assert np.all(wp == 0xAB)
    with pytest.raises(t3.T3Error):
        t3.t3_pack_ternary(w)


def test_pack_size_errors(lib):
    assert lib.t3_pack_ternary(None, None, -1, 3) == t3.T3_EINVAL
    assert lib.t3_pack_ternary(None, None, 0, 3) == t3.T3_OK
    assert lib.t3_pack_ternary(None, None, 4, 3) == t3.T3_EINVAL


FAKE = ctypes.c_void_p(4096)  # never dereferenced: every case returns first


@pytest.mark.parametrize("fn", ["t3_gemm_fwd", "t3_gemm_bwd_dx", "t3_gemm_bwd_dw"])
def test_gemm_argument_errors_before_launch(lib, fn):
    f = getattr(lib, fn)
    assert f(FAKE, FAKE, FAKE, -1, 4, 4, None) == t3.T3_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, -1, 4, None) == t3.T3_EINVAL
    assert f(FAKE, FAKE, FAKE, 4, 4, -1, None) == t3.T3_EINVAL
    assert f(FAKE, FAKE, FAKE, 1 << 31, 4, 4, None) == t3.T3_EINVAL
    assert f(None, FAKE, FAKE, 4, 4, 4, None) == t3.T3_EINVAL
    assert f(FAKE, None, FAKE, 4, 4, 4, None) == t3.T3_EINVAL
    assert f(FAKE, FAKE, None, 4, 4, 4, None) == t3.T3_EINVAL


def test_gemm_empty_outputs_are_noops(lib):
    # an empty output: nothing to write, no device touched
    assert lib.t3_gemm_fwd(None, None, None, 0, 5, 5, None) == t3.T3_OK
    assert lib.t3_gemm_fwd(None, None, None, 5, 0, 5, None) == t3.T3_OK
    assert lib.t3_gemm_bwd_dx(None, None, None, 0, 5, 5, None) == t3.T3_OK
    assert lib.t3_gemm_bwd_dx(None, None, None, 5, 5, 0, None) == t3.T3_OK
    assert lib.t3_gemm_bwd_dw(None, None, None, 5, 0, 5, None) == t3.T3_OK
    assert lib.t3_gemm_bwd_dw(None, None, None, 5, 5, 0, None) == t3.T3_OK


def test_gemm_overflow_bounds(lib):
    # |A W| <= 128 per term: exact int32 up to a reduction of 16777215
    assert lib.t3_gemm_fwd(FAKE, FAKE, FAKE, 1, 1, 16777216, None) == t3.T3_EOVERFLOW
    assert lib.t3_gemm_bwd_dx(FAKE, FAKE, FAKE, 1, 16777216, 1, None) == t3.T3_EOVERFLOW
    # int8 x int8: the pages' bound of 131071 rows
    assert lib.t3_gemm_bwd_dw(FAKE, FAKE, FAKE, 131072, 1, 1, None) == t3.T3_EOVERFLOW


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    A = torch.zeros((4, 8), dtype=torch.int8)
    Wp = torch.zeros((3, 2), dtype=torch.uint8)
    with pytest.raises(TypeError):
        t3.t3_gemm_fwd(A, Wp)


def test_missing_library_fails_loudly(tmp_path):
    """Without libt3.so and without a compiler the binding raises; it never
    computes anything another way."""
    pkg = tmp_path / "ternary_weight_int8_t3_gb300"
    shutil.copytree(os.path.join(ROOT, "ternary_weight_int8_t3_gb300"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "include"), tmp_path / "include")
    code = ("import ternary_weight_int8_t3_gb300 as t3\n"
            "try:\n    t3.load()\nexcept Exception as e:\n    print('RAISED', type(e).__name__)\n"
            "else:\n    print('LOADED')\n")
    fake = tmp_path / "nvcc"
    fake.write_text("#!/bin/sh\necho 'no compiler here' >&2\nexit 1\n")
    fake.chmod(0o755)
    env = dict(os.environ, NVCC=str(fake))
    r = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, env=env, capture_output=True,
                       text=True, timeout=120)
    assert "RAISED RuntimeError" in r.stdout, r.stdout + r.stderr
