"""Oracle for the two-bit draft head -- TEST INFRASTRUCTURE ONLY (tests, the
smoke check and the benchmark's CPU legs may import it; the library never
does; no code is shared).

"Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
surgery / Two-bit draft head": the drafter's output head scores every token
of the vocabulary; a 2-bit copy of it is cheap but noisy, so it only
shortlists 16 candidates, which the FP8 head then rescores.  The pages fix
neither format nor the tie rules; the readings (also in the C oracle's
header):

1. the 2-bit head mirrors the 3-bit format: per row a 4-entry E4M3 codebook,
   2-bit codes (code j of a 32-weight group at bits 2j..2j+1 of its 64-bit
   little-endian group), one E8M0 scale per group, groups in 128-row tiles;
   2 + 8/32 = 2.25 bits per weight;
2. scores s[m, n] = a_scale[m] * sum_k a[m, k] w2[n, k] (C oracle, fp64 sum in
   k order, one rounding to fp32);
3. the shortlist of token m: the 16 rows with the highest scores, in
   descending score order, equal scores -> lower row id first (a row's score
   is compared as the fp32 value);
4. the FP8 head: E4M3 weights [N][K] row-major with one fp32 scale per row;
   the rescored logit of shortlisted row n is a_scale[m] * row_scale[n] *
   sum_k a[m, k] E4M3(w8[n, k]) (fp64 sum in k order, one rounding to fp32);
5. the token picked: the shortlisted row with the highest rescored logit,
   equal logits -> the one earlier in the shortlist.
"""
from __future__ import annotations

import numpy as np

import oracle

SHORTLIST = 16


def footprint_bytes(N: int, K: int) -> tuple[int, int, int]:
    """(codes, scales, codebooks) bytes of an N x K two-bit head."""
    return K * N // 4, K * N // 32, 4 * N


def scores(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int):
    """(s fp32 [M, N], bound fp64 [M, N]) of the 2-bit head."""
    a, codes, scales, codebooks = (oracle._u8(x) for x in (a, codes, scales, codebooks))
    a_scale = np.ascontiguousarray(a_scale, dtype=np.float32)
    y = np.empty((M, N), dtype=np.float32)
    bound = np.empty((M, N), dtype=np.float64)
    lib = oracle._load()
    lib.orc_gemm2(oracle._p(a, oracle.ctypes.c_uint8), oracle._p(a_scale, oracle.ctypes.c_float),
                  oracle._p(codes, oracle.ctypes.c_uint8), oracle._p(scales, oracle.ctypes.c_uint8),
                  oracle._p(codebooks, oracle.ctypes.c_uint8), M, N, K,
                  oracle._p(y, oracle.ctypes.c_float), oracle._p(bound, oracle.ctypes.c_double))
    return y, bound


def shortlist(s: np.ndarray, L: int = SHORTLIST) -> np.ndarray:
    """int32 [M, L]: per row of s the L highest entries in descending order,
    equal values -> lower index first (step 3)."""
    s = np.asarray(s, dtype=np.float32)
    M, N = s.shape
    out = np.empty((M, min(L, N)), dtype=np.int32)
    for m in range(M):
        # lexsort: last key is primary; descending value, then ascending index
        order = np.lexsort((np.arange(N), -s[m].astype(np.float64)))
        out[m] = order[:out.shape[1]]
    return out


def rescore(a, a_scale, head8, row_scale, rows, M: int, N: int, K: int):
    """(logits fp32 [M, R], bound fp64 [M, R]) of the FP8 head on rows [M, R]."""
    a, head8 = oracle._u8(a), oracle._u8(head8)
    a_scale = np.ascontiguousarray(a_scale, dtype=np.float32)
    row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    R = rows.shape[1]
    logits = np.empty((M, R), dtype=np.float32)
    bound = np.empty((M, R), dtype=np.float64)
    oracle._load().orc_rescore8(oracle._p(a, oracle.ctypes.c_uint8), oracle._p(a_scale, oracle.ctypes.c_float),
                                oracle._p(head8, oracle.ctypes.c_uint8),
                                oracle._p(row_scale, oracle.ctypes.c_float), M, N, K,
                                oracle._p(rows, oracle.ctypes.c_int32), R,
                                oracle._p(logits, oracle.ctypes.c_float),
                                oracle._p(bound, oracle.ctypes.c_double))
    return logits, bound


def pick(rows: np.ndarray, logits: np.ndarray) -> np.ndarray:
    """int32 [M]: the row of each token's highest rescored logit, ties -> the
    one earlier in the shortlist (step 5)."""
    rows = np.asarray(rows)
    logits = np.asarray(logits, dtype=np.float32)
    out = np.empty(rows.shape[0], dtype=np.int32)
    for m in range(rows.shape[0]):
        best = 0
        for i in range(1, rows.shape[1]):
            if logits[m, i] > logits[m, best]:
                best = i
        out[m] = rows[m, best]
    return out


def draft_head(a, a_scale, codes, scales, codebooks, head8, row_scale, M: int, N: int, K: int):
    """The whole step: (shortlist [M, 16], rescored logits [M, 16], picked
    token [M], 2-bit scores [M, N])."""
    s, _ = scores(a, a_scale, codes, scales, codebooks, M, N, K)
    rows = shortlist(s)
    logits, _ = rescore(a, a_scale, head8, row_scale, rows, M, N, K)
    return rows, logits, pick(rows, logits), s
