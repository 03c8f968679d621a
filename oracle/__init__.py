"""CPU oracle for the 3.25-bit codebook-quantised matmul.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library never does.  It shares
no code with the CUDA path.

The arithmetic lives in ``cbq_oracle.c`` (plain C, fp64, one loop per
definition; see its header for the format and the passages it follows, from
"Hibana: Fast Agentic Inference on Unified-Memory Devices", section
"Model surgery / Three-bit weights").  This module compiles it with gcc and
wraps it with numpy arrays.  ``brute.py`` holds an independent exact-rational
restatement for tiny shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cbq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcbq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = configure(ctypes.CDLL(build()))
        return _lib


def configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    if True:
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e8m0_value.argtypes = [ctypes.c_uint8]
        lib.orc_e8m0_value.restype = ctypes.c_double
        lib.orc_e4m3_round.argtypes = [ctypes.c_double]
        lib.orc_e4m3_round.restype = ctypes.c_uint8
        lib.orc_group_offset.argtypes = [i64, i64, i64, i64]
        lib.orc_group_offset.restype = i64
        lib.orc_code.argtypes = [u8p, i64, i64, i64, i64]
        lib.orc_code.restype = ctypes.c_int
        lib.orc_set_code.argtypes = [u8p, i64, i64, i64, i64, ctypes.c_int]
        lib.orc_set_code.restype = None
        lib.orc_gemm_rows.argtypes = [u8p, f32p, u8p, u8p, u8p, i64, i64, i64, i64p, i64, f32p,
                                      f64p]
        lib.orc_gemm_rows.restype = None
        lib.orc_group_scale.argtypes = [f32p]
        lib.orc_group_scale.restype = ctypes.c_uint8
        lib.orc_unpack.argtypes = [u8p, u8p, u8p, i64, i64, f32p]
        lib.orc_unpack.restype = None
        lib.orc_gemm.argtypes = [u8p, f32p, u8p, u8p, u8p, i64, i64, i64, f32p, f64p]
        lib.orc_gemm.restype = None
        lib.orc_grouped_gemm.argtypes = [u8p, f32p, u8p, u8p, u8p, i64, i32p, i64,
                                         i64, i64, i64, f32p, f64p, i64p]
        lib.orc_grouped_gemm.restype = None
        lib.orc_pack.argtypes = [f32p, i64, i64, u8p, u8p, u8p]
        lib.orc_pack.restype = None
        lib.orc_group_offset2.argtypes = [i64, i64, i64, i64]
        lib.orc_group_offset2.restype = i64
        lib.orc_code2.argtypes = [u8p, i64, i64, i64, i64]
        lib.orc_code2.restype = ctypes.c_int
        lib.orc_gemm2.argtypes = [u8p, f32p, u8p, u8p, u8p, i64, i64, i64, f32p, f64p]
        lib.orc_gemm2.restype = None
        lib.orc_rescore8.argtypes = [u8p, f32p, u8p, f32p, i64, i64, i64, i32p, i64, f32p, f64p]
        lib.orc_rescore8.restype = None
        lib.orc_num_threads.argtypes = []
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        lib.orc_set_num_threads.restype = None
    return lib


def _p(arr: np.ndarray, ctype):
    assert arr.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return arr.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.uint8)


# ---- formats ---------------------------------------------------------------

def e4m3_value(b: int) -> float:
    return _load().orc_e4m3_value(int(b))


def e8m0_value(s: int) -> float:
    return _load().orc_e8m0_value(int(s))


def e4m3_round(x: float) -> int:
    return int(_load().orc_e4m3_round(float(x)))


def e4m3_table() -> np.ndarray:
    """fp64 value of each of the 256 E4M3 bytes."""
    return np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


# ---- bitstream ---------------------------------------------------------------

def group_offset(N: int, K: int, n: int, g: int) -> int:
    """Byte offset of group (n, g) in the code stream (128-row tiles,
    k-tile-major inside a tile; see cbq_oracle.c)."""
    return int(_load().orc_group_offset(N, K, n, g))


def code_at(codes: np.ndarray, N: int, K: int, n: int, k: int) -> int:
    codes = _u8(codes)
    return int(_load().orc_code(_p(codes, ctypes.c_uint8), N, K, n, k))


def codes_from_indices(idx: np.ndarray) -> np.ndarray:
    """Pack an [N, K] array of codes 0..7 into the code stream (3KN/8 bytes,
    returned with shape [N, 3K/8] for convenience; the bytes are in tile
    order, not row order)."""
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    N, K = idx.shape
    out = np.zeros(N * (K // 32) * 12, dtype=np.uint8)
    lib = _load()
    p = _p(out, ctypes.c_uint8)
    for n in range(N):
        for k in range(K):
            lib.orc_set_code(p, N, K, n, k, int(idx[n, k]))
    return out.reshape(N, K // 32 * 12)


def indices_from_codes(codes: np.ndarray, N: int, K: int) -> np.ndarray:
    codes = _u8(codes)
    lib = _load()
    p = _p(codes, ctypes.c_uint8)
    out = np.empty((N, K), dtype=np.int64)
    for n in range(N):
        for k in range(K):
            out[n, k] = lib.orc_code(p, N, K, n, k)
    return out


# ---- unpack / gemm / grouped -----------------------------------------------

def unpack(codes, scales, codebooks, N: int, K: int) -> np.ndarray:
    codes, scales, codebooks = _u8(codes), _u8(scales), _u8(codebooks)
    W = np.empty((N, K), dtype=np.float32)
    _load().orc_unpack(_p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                       _p(codebooks, ctypes.c_uint8), N, K, _p(W, ctypes.c_float))
    return W


def gemm(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int):
    """Return (y fp32 [M, N], bound fp64 [M, N])."""
    a, codes, scales, codebooks = _u8(a), _u8(codes), _u8(scales), _u8(codebooks)
    a_scale = np.ascontiguousarray(a_scale, dtype=np.float32)
    y = np.empty((M, N), dtype=np.float32)
    bound = np.empty((M, N), dtype=np.float64)
    _load().orc_gemm(_p(a, ctypes.c_uint8), _p(a_scale, ctypes.c_float),
                     _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                     _p(codebooks, ctypes.c_uint8), M, N, K,
                     _p(y, ctypes.c_float), _p(bound, ctypes.c_double))
    return y, bound


def gemm_rows(a, a_scale, codes, scales, codebooks, M: int, N: int, K: int, rows):
    """y and bound [M, len(rows)] for the listed output rows of the N-row matrix."""
    a, codes, scales, codebooks = _u8(a), _u8(codes), _u8(scales), _u8(codebooks)
    a_scale = np.ascontiguousarray(a_scale, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    y = np.empty((M, len(rows)), dtype=np.float32)
    bound = np.empty((M, len(rows)), dtype=np.float64)
    _load().orc_gemm_rows(_p(a, ctypes.c_uint8), _p(a_scale, ctypes.c_float),
                          _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                          _p(codebooks, ctypes.c_uint8), M, N, K, _p(rows, ctypes.c_int64),
                          len(rows), _p(y, ctypes.c_float), _p(bound, ctypes.c_double))
    return y, bound


def expert(codes, scales, codebooks, e: int, N: int, K: int):
    """(codes, scales, codebooks) of expert e in a stack of packed experts."""
    cb = 3 * K * N // 8
    flat = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    return (flat[e * cb:(e + 1) * cb], np.ascontiguousarray(scales)[e * N:(e + 1) * N],
            np.ascontiguousarray(codebooks)[e * N:(e + 1) * N])


def grouped_gemm(a, a_scale, codes, scales, codebooks, E: int, topk_idx,
                 M: int, N: int, K: int):
    """Return (y fp32 [M, topk, N], bound fp64 [M, topk, N], read_count int64 [E])."""
    a, codes, scales, codebooks = _u8(a), _u8(codes), _u8(scales), _u8(codebooks)
    a_scale = np.ascontiguousarray(a_scale, dtype=np.float32)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    topk = topk_idx.shape[1]
    y = np.empty((M, topk, N), dtype=np.float32)
    bound = np.empty((M, topk, N), dtype=np.float64)
    reads = np.zeros(E, dtype=np.int64)
    _load().orc_grouped_gemm(_p(a, ctypes.c_uint8), _p(a_scale, ctypes.c_float),
                             _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8),
                             _p(codebooks, ctypes.c_uint8), E,
                             _p(topk_idx, ctypes.c_int32), topk, M, N, K,
                             _p(y, ctypes.c_float), _p(bound, ctypes.c_double),
                             _p(reads, ctypes.c_int64))
    return y, bound, reads


def pack(W: np.ndarray):
    """Quantise fp32 W [N, K] -> (codes [N, 3K/8], scales [N, K/32], codebooks [N, 8])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    codes = np.zeros((N, K // 32 * 12), dtype=np.uint8)
    scales = np.zeros((N, K // 32), dtype=np.uint8)
    cbs = np.zeros((N, 8), dtype=np.uint8)
    _load().orc_pack(_p(W, ctypes.c_float), N, K, _p(codes, ctypes.c_uint8),
                     _p(scales, ctypes.c_uint8), _p(cbs, ctypes.c_uint8))
    return codes, scales, cbs


def group_scale(w32: np.ndarray) -> int:
    w32 = np.ascontiguousarray(w32, dtype=np.float32)
    assert w32.size == 32
    return int(_load().orc_group_scale(_p(w32, ctypes.c_float)))


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def packed_bytes(N: int, K: int) -> int:
    """Bytes of one packed matrix: 3 bits per weight plus one byte per 32
    weights plus an 8-byte codebook per row."""
    return 3 * K * N // 8 + K * N // 32 + 8 * N
