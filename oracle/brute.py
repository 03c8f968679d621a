"""Exact-rational brute force for tiny codebook-quantised matmuls.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is a second,
independent statement of the same definitions as ``cbq_oracle.c``, written
with Python integers and ``fractions.Fraction`` so that it has no rounding at
all: the C oracle is pinned against it on shapes from 1x32x1 to 4x64x8.

Format (from "Hibana: Fast Agentic Inference on Unified-Memory Devices",
section "Model surgery / Three-bit weights": 8-entry FP8 codebook, 3-bit
codes, one 8-bit scale per 32 weights): the 12 bytes of a group form one
little-endian 96-bit integer and code j is ``(G >> 3j) & 7``; groups sit in
128-row tiles, k-tile-major inside a tile (``group_offset``).
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


def group_offset(N: int, K: int, n: int, g: int) -> int:
    """Byte offset of group (n, g): 128-row tiles (the last one holding the
    remaining R rows) starting at 128t * 3K/8; inside a tile, k-tile
    c = g // 4 is a block of R rows x W bytes, W = 12 x (its groups, 4 but
    in a last partial k-tile)."""
    t, i = divmod(n, 128)
    R = min(128, N - 128 * t)
    c = g // 4
    W = 12 * min(4, K // 32 - 4 * c)
    return 128 * t * (3 * K // 8) + c * R * 48 + i * W + (g % 4) * 12


def group_int(codes, N: int, K: int, n: int, g: int) -> int:
    flat = bytes(bytearray(codes.reshape(-1) if hasattr(codes, "reshape") else codes))
    o = group_offset(N, K, n, g)
    return int.from_bytes(flat[o:o + 12], "little")


def code(codes, N: int, K: int, n: int, k: int) -> int:
    return (group_int(codes, N, K, n, k // 32) >> (3 * (k % 32))) & 7


def weight(codes, scales, codebooks, N: int, K: int, n: int, k: int) -> Fraction:
    return e4m3(int(codebooks[n][code(codes, N, K, n, k)])) * e8m0(int(scales[n][k // 32]))


def gemm_exact(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int):
    """Exact y[m][n] as Fractions.  ``a`` is [M][K] E4M3 bytes, ``a_scale``
    a list of floats (taken exactly), ``codes`` the packed stream."""
    flat = bytes(bytearray(codes.reshape(-1) if hasattr(codes, "reshape") else codes))
    out = []
    for m in range(M):
        row = []
        s = Fraction(float(a_scale[m]))
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                o = group_offset(N, K, n, k // 32)
                c = (int.from_bytes(flat[o:o + 12], "little") >> (3 * (k % 32))) & 7
                w = e4m3(int(codebooks[n][c])) * e8m0(int(scales[n][k // 32]))
                acc += e4m3(int(a[m][k])) * w
            row.append(s * acc)
        out.append(row)
    return out
