"""Exact-rational brute force for tiny codebook-quantised matmuls.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is a second,
independent statement of the same definitions as ``cbq_oracle.c``, written
with Python integers and ``fractions.Fraction`` so that it has no rounding at
all: the C oracle is pinned against it on shapes from 1x32x1 to 4x64x8.

Format (from "Hibana: Fast Agentic Inference on Unified-Memory Devices",
section "Model surgery / Three-bit weights": 8-entry FP8 codebook, 3-bit
codes, one 8-bit scale per 32 weights): the 12 bytes of a group form one
little-endian 96-bit integer and code j is ``(G >> 3j) & 7``.
"""
from __future__ import annotations

from fractions import Fraction


def e4m3(b: int) -> Fraction:
    """OCP E4M3 byte -> exact value (NaN bytes 0x7F/0xFF are rejected)."""
    b &= 0xFF
    sign = -1 if b & 0x80 else 1
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        raise ValueError("E4M3 NaN has no rational value")
    if e == 0:
        return sign * Fraction(m, 8) * Fraction(1, 2 ** 6)
    return sign * (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))


def e8m0(s: int) -> Fraction:
    if s == 255:
        raise ValueError("E8M0 NaN has no rational value")
    return Fraction(2) ** (s - 127)


def group_int(codes_row: bytes, g: int) -> int:
    return int.from_bytes(bytes(codes_row[12 * g: 12 * g + 12]), "little")


def code(codes_row: bytes, k: int) -> int:
    return (group_int(codes_row, k // 32) >> (3 * (k % 32))) & 7


def weight(codes_row, scales_row, cb_row, k: int) -> Fraction:
    return e4m3(int(cb_row[code(codes_row, k)])) * e8m0(int(scales_row[k // 32]))


def gemm_exact(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int):
    """Exact y[m][n] as Fractions.  ``a`` is [M][K] E4M3 bytes, ``a_scale``
    a list of floats (taken exactly), the packed arrays are per-row byte rows."""
    out = []
    for m in range(M):
        row = []
        s = Fraction(float(a_scale[m]))
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += e4m3(int(a[m][k])) * weight(codes[n], scales[n], codebooks[n], k)
            row.append(s * acc)
        out.append(row)
    return out
