"""Oracle for the fused gate-up epilogue -- TEST INFRASTRUCTURE ONLY (tests
may import it; the library never does; no code is shared).

"Hibana: Fast Agentic Inference on Unified-Memory Devices", section
"Adaptive speculation": a verify round runs the drafted tokens through the
model's feed-forward layers, whose first matmul is the fused gate and up
projection; its product feeds the down projection as E4M3 activations with
one fp32 scale per token (the same activation format every matmul here
takes).  The pages name the fusion only, so the readings here are the
plainest ones:

1. layout: the N = 2F rows of the packed weight hold, for each block of 64
   features (the last block may be shorter, R = min(64, F - 64 b) features),
   the block's R gate rows followed by its R up rows, so block b is rows
   [128 b, 128 b + 2 R) -- exactly one 128-row tile;
2. g and u are the matmul outputs of a feature's gate and up rows (a_scale
   applied), h = SiLU(g) * u with SiLU(x) = x / (1 + e^-x), in fp64;
3. per token m: amax = max_f |h[m, f]|, s[m] = amax / 448 (so the largest
   value lands on the largest E4M3 magnitude), s[m] = 1 when amax = 0;
4. q[m, f] = E4M3(h[m, f] / s[m]), rounded to nearest, ties to even,
   saturating at +-448 (the packer's E4M3 rounding, oracle.e4m3_round).

The matmul outputs come from the C oracle (fp64 sums in k order, rounded once
to fp32); everything after that is fp64 here.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

BLOCK = 64          # features per block (one 128-row tile holds its gate and up rows)
E4M3_MAX = 448.0


def rows_of_feature(F: int, f: int) -> tuple[int, int]:
    """(gate row, up row) of feature f in the 2F-row packed weight."""
    b, j = divmod(f, BLOCK)
    R = min(BLOCK, F - BLOCK * b)
    return 2 * BLOCK * b + j, 2 * BLOCK * b + R + j


def silu(x: float) -> float:
    if x < -700.0:                      # e^-x overflows fp64; x / (1 + e^-x) tends to -0 there
        return -0.0
    return x / (1.0 + math.exp(-x))


def gate_up_from_y(y: np.ndarray):
    """(q uint8 [M, F], s float64 [M], h float64 [M, F]) from the fp32 matmul
    output y [M, 2F] of the fused gate-up weight."""
    y = np.asarray(y)
    M, N = y.shape
    assert N % 2 == 0
    F = N // 2
    h = np.empty((M, F), dtype=np.float64)
    for f in range(F):
        gr, ur = rows_of_feature(F, f)
        for m in range(M):
            h[m, f] = silu(float(y[m, gr])) * float(y[m, ur])
    s = np.empty(M, dtype=np.float64)
    q = np.empty((M, F), dtype=np.uint8)
    for m in range(M):
        amax = float(np.max(np.abs(h[m]))) if F else 0.0
        s[m] = amax / E4M3_MAX if amax > 0.0 else 1.0
        for f in range(F):
            q[m, f] = oracle.e4m3_round(h[m, f] / s[m])
    return q, s, h


def gate_up(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int):
    """The whole fused step: matmul against the packed 2F-row weight, then
    steps 2-4.  Returns (q, s, h, y, bound) -- y and its error bound as
    oracle.gemm gives them."""
    y, bound = oracle.gemm(a, a_scale, codes, scales, codebooks, M, N, K)
    q, s, h = gate_up_from_y(y)
    return q, s, h, y, bound
