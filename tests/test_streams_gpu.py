"""Calls on several streams at once: the products of two independent problems
(large and small M, forward and both backward products, the device packer)
enqueued alternately on two non-blocking streams, without synchronizing in
between, each result compared in full with the oracle.  The library keeps no
per-call state across streams, so the interleaving must not change a bit."""
import numpy as np
import pytest

import oracle
import t3_synth
import ternary_weight_int8_t3_gb300 as t3

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_two_streams_interleaved():
    problems = [(300, 640, 1280, 31), (1, 2048, 1024, 32), (27, 1024, 768, 33), (700, 384, 256, 34)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    inputs, outputs = [], []
    for (M, N, K, seed) in problems:
        g = t3_synth.rng(seed)
        A = t3_synth.int8_uniform(g, (M, K))
        w = t3_synth.ternary(g, (K, N))
        dY = t3_synth.int8_uniform(g, (M, N))
        inputs.append((A, w, dY))
    torch.cuda.synchronize()
    for rep in range(3):
        for i, (M, N, K, _) in enumerate(problems):
            A, w, dY = inputs[i]
            s = streams[(i + rep) % 2]
            with torch.cuda.stream(s):
                w_d = _dev(w)
                wp_d = t3.t3_pack_ternary_device(w_d, stream=s)
                C = t3.t3_gemm_fwd(_dev(A), wp_d, K=K, stream=s)
                dX = t3.t3_gemm_bwd_dx(_dev(dY), wp_d, K, stream=s)
                dW = t3.t3_gemm_bwd_dw(_dev(A), _dev(dY), stream=s)
            outputs.append((i, wp_d, C, dX, dW))
    torch.cuda.synchronize()
    rc, detail = t3.t3_last_device_error()
    assert rc == t3.T3_OK, f"device error word set ({detail:#x})"
    want = {}
    for i, (M, N, K, _) in enumerate(problems):
        A, w, dY = inputs[i]
        wp = oracle.pack(w)
        want[i] = (wp, oracle.fwd(A, wp), oracle.dx(dY, wp, K), oracle.dw(A, dY))
    for i, wp_d, C, dX, dW in outputs:
        wp, c, x, g = want[i]
        M, N, K, _ = problems[i]
        np.testing.assert_array_equal(wp_d.cpu().numpy(), wp, err_msg=f"pack {problems[i]}")
        np.testing.assert_array_equal(C.cpu().numpy(), c, err_msg=f"fwd {problems[i]}")
        np.testing.assert_array_equal(dX.cpu().numpy(), x, err_msg=f"dX {problems[i]}")
        np.testing.assert_array_equal(dW.cpu().numpy(), g, err_msg=f"dW {problems[i]}")
