"""Seeded synthetic inputs shared by the tests, the bench and the smoke run.

This module holds no arithmetic of the method: it draws int8 activations,
ternary weight matrices and raw byte buffers from numpy's PCG64 generator and
names the workloads.  Packing, decoding and every product live elsewhere (the
library under test and, separately, the oracle).

Workloads follow the pages' shapes: the ragged 300x272x96 forward case of the
"Bit-exact" table and the 16384x3456x1280 forward shape of the "Throughput"
table in "t27c PTX backend: ternary x int8 GEMM kernel emitted by a .t27 spec
(int8 mma.sync), ptx-run glue"; the 1782-row backward of "spec(igla):
hslm_bwd_ptx -- HSLM backward dX and dW as int8 tensor-core PTX written by
t27" ("Measured: RTX 4090").  The pages print no generator, so activations are
uniform over [-128, 127] and weights take the stated ternary mix.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def int8_uniform(g: np.random.Generator, shape) -> np.ndarray:
    """int8 uniform over [-128, 127]."""
    return g.integers(-128, 128, size=shape, dtype=np.int16).astype(np.int8)


def ternary(g: np.random.Generator, shape, p_zero: float = 1.0 / 3.0) -> np.ndarray:
    """int8 values in {-1, 0, +1}: 0 with probability p_zero, +1 and -1 equally likely."""
    p_pm = (1.0 - p_zero) / 2.0
    return g.choice(np.array([-1, 0, 1], dtype=np.int8), size=shape,
                    p=[p_pm, p_zero, p_pm]).astype(np.int8)


def raw_bytes(g: np.random.Generator, shape) -> np.ndarray:
    """Uniform random bytes (every 2-bit code, pad bits included)."""
    return g.integers(0, 256, size=shape, dtype=np.int16).astype(np.uint8)


@dataclass(frozen=True)
class Workload:
    name: str
    op: str            # "fwd", "bwd" (dX and dW), "skinny" (forward, small M)
    M: int
    N: int
    K: int
    seed: int
    p_zero: float      # probability of a zero weight


# The workloads: ragged forward, square forward, the pages' largest forward
# shape, the 1782-row backward, the small-M forward sweep, and the other forward
# shapes of the pages' throughput table ("t27c PTX backend: ternary x int8 GEMM
# kernel emitted by a .t27 spec", section "Measured: RTX 4090"), M x N x K.
PAGES_FWD_SHAPES = [(4096, 3456, 1280), (4096, 1280, 3456), (4096, 1280, 1280),
                    (16384, 1280, 3456), (16384, 1280, 1280)]
WORKLOADS = [
    Workload("fwd_ragged_300x272x96", "fwd", 300, 272, 96, 0, 1.0 / 3.0),
    Workload("fwd_square_4096", "fwd", 4096, 4096, 4096, 1, 0.5),
    Workload("fwd_16384x3456x1280", "fwd", 16384, 3456, 1280, 2, 1.0 / 3.0),
    Workload("bwd_1782x3456x1280", "bwd", 1782, 3456, 1280, 3, 1.0 / 3.0),
] + [
    Workload(f"fwd_{m}x{n}x{k}", "fwd", m, n, k, 5 + i, 1.0 / 3.0)
    for i, (m, n, k) in enumerate(PAGES_FWD_SHAPES)
] + [
    Workload(f"skinny_m{m}_n{n}_k{k}", "skinny", m, n, k, 4, 1.0 / 3.0)
    for (n, k) in ((3456, 1280), (8192, 8192)) for m in (1, 8, 27)
]

BY_NAME = {w.name: w for w in WORKLOADS}


def make_inputs(wl: Workload):
    """Returns (A [M][K] int8, w [K][N] ternary int8, dY [M][N] int8) for a workload.

    The draws happen in a fixed order from one generator per workload seed, so
    every consumer sees the same bytes."""
    g = rng(wl.seed)
    A = int8_uniform(g, (wl.M, wl.K))
    w = ternary(g, (wl.K, wl.N), wl.p_zero)
    dY = int8_uniform(g, (wl.M, wl.N))
    return A, w, dY
