"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, rejects bad arguments before touching the device, and its
host quantiser matches the oracle's byte for byte."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from bit_codebook_quantized_gb300 import ops, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_codebook_quantized_gb300 import build
    build.build()
    return ops.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "cbq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cbq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert set(names) == set(ops.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_packed_sizes_closed_form(L):
    for N, K in [(1, 128), (2048, 2048), (12288, 4096), (5120, 25600), (151936, 2048), (0, 0)]:
        c, s, b = ops.packed_sizes(N, K)
        assert (c, s, b) == (3 * K * N // 8, K * N // 32, 8 * N)
        assert c + s + b == oracle.packed_bytes(N, K)
    with pytest.raises(ops.CbqError):
        ops.packed_sizes(16, 96)
    with pytest.raises(ops.CbqError):
        ops.packed_sizes(-1, 128)


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4, -5):
        assert ops.status_str(s) and ops.status_str(s) != "unknown status"
    assert ops.status_str(7) == "unknown status"


def test_argument_errors_before_device(L):
    w = ops._Weight(16, 16, 16)
    p = ctypes.byref(w)
    # K not a multiple of 128, M out of range, bad path, bad topk / E
    assert L.cbq_gemm(16, 16, p, 1, 8, 96, 16, None) == ops.EINVAL
    assert L.cbq_gemm(16, 16, p, 65, 8, 128, 16, None) == ops.EINVAL
    assert L.cbq_gemm(16, 16, p, -1, 8, 128, 16, None) == ops.EINVAL
    assert L.cbq_gemm_path(16, 16, p, 1, 8, 128, 16, None, 0, None, 7) == ops.EINVAL
    assert L.cbq_gemm_ws(16, 16, p, 1, 8, 96, 16, None, 0, None) == ops.EINVAL
    n = ctypes.c_size_t(7)
    assert L.cbq_gemm_workspace_size(1, 8, 96, ctypes.byref(n)) == ops.EINVAL
    assert L.cbq_gemm_workspace_size(1, 8, 128, None) == ops.EINVAL
    assert L.cbq_gemm_workspace_size(0, 8, 128, ctypes.byref(n)) == ops.OK and n.value == 0
    assert L.cbq_grouped_gemm(16, 16, p, 0, 16, 1, 1, 8, 128, 16, None) == ops.EINVAL
    assert L.cbq_grouped_gemm(16, 16, p, 4, 16, 9, 1, 8, 128, 16, None) == ops.EINVAL
    assert L.cbq_grouped_gemm(16, 16, p, 4, 16, 5, 1, 8, 128, 16, None) == ops.EINVAL
    # grouped stream-K needs a workspace; workspace sizes of valid shapes only
    assert L.cbq_grouped_gemm_path(16, 16, p, 4, 16, 2, 1, 8, 128, 16, None, ops.PATH_STREAMK) == ops.EINVAL
    assert L.cbq_grouped_gemm_ws(16, 16, p, 4, 16, 2, 1, 8, 128, 16, None, 0, None, 4) == ops.EINVAL
    assert L.cbq_grouped_gemm_ws(16, 16, p, 4, 16, 9, 1, 8, 128, 16, None, 0, None, 0) == ops.EINVAL
    assert L.cbq_grouped_workspace_size(4, 2, 1, 8, 96, ctypes.byref(n)) == ops.EINVAL
    assert L.cbq_grouped_workspace_size(0, 1, 1, 8, 128, ctypes.byref(n)) == ops.EINVAL
    assert L.cbq_grouped_workspace_size(4, 2, 1, 8, 128, None) == ops.EINVAL
    assert L.cbq_grouped_workspace_size(4, 2, 0, 8, 128, ctypes.byref(n)) == ops.OK and n.value == 0
    assert L.cbq_unpack(p, 8, 100, 16, None) == ops.EINVAL
    # expert budget: k in [1, B], B <= E <= 4096, T >= 1, outputs present and aligned
    assert L.cbq_select_budget(16, 4, 12, 0, 4, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(16, 4, 12, 5, 4, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(16, 4, 12, 2, 13, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(16, 4, 4097, 2, 4, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(16, 0, 12, 2, 4, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(None, 4, 12, 2, 4, 16, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(16, 4, 12, 2, 4, None, 16, None) == ops.EINVAL
    assert L.cbq_select_budget(18, 4, 12, 2, 4, 16, 16, None) == ops.EINVAL   # logits not 4-byte aligned
    # empty problems are no-ops that succeed without a device
    assert L.cbq_gemm(0, 0, None, 0, 8, 128, 0, None) == ops.OK
    assert L.cbq_gemm(0, 0, None, 4, 0, 128, 0, None) == ops.OK
    assert L.cbq_unpack(None, 0, 128, None, None) == ops.OK
    assert L.cbq_pack(None, 0, 128, None, None, None) == ops.OK
    assert L.cbq_pack(None, 4, 128, None, None, None) == ops.EINVAL


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU answer")
def test_no_gpu_is_reported(L):
    w = ops._Weight(16, 16, 16)
    st = L.cbq_gemm(16, 16, ctypes.byref(w), 1, 8, 128, 16, None)
    assert st == ops.EDEVICE


def test_pack_rejects_non_finite(L):
    W = np.zeros((2, 128), np.float32)
    W[1, 5] = np.nan
    with pytest.raises(ops.CbqError):
        ops.pack(W)


@pytest.mark.parametrize("N,K,seed", [(5, 128, 1), (9, 256, 2), (3, 512, 3)])
def test_host_pack_matches_oracle_bytes(L, N, K, seed):
    W = synth.gen_dense_weights_fp32(N, K, seed)
    W[0, :32] = 0.0                                  # an all-zero group
    W[1 % N, 40] = 3e-39                             # a subnormal weight
    got = ops.pack(W)
    want = oracle.pack(W)
    for g_, w_ in zip(got, want):
        assert np.array_equal(g_, w_)


def test_host_pack_matches_oracle_on_few_valued_rows(L):
    """Rows built from 8 values (many exact ties in the Lloyd rounds) pack to
    the same bytes as the oracle."""
    rng = synth.rng_for(77)
    N, K = 3, 256
    vals = [-1.0, -0.5, -0.25, 0.0, 0.125, 0.25, 0.5, 1.0]
    W = np.empty((N, K), np.float32)
    for n in range(N):
        u = np.repeat(vals, K // 8)
        rng.shuffle(u)
        u[0::32] = [1.0, -1.0] * (K // 64)
        W[n] = u * np.ldexp(1.0, np.repeat(rng.integers(100, 150, K // 32), 32) - 127)
    codes, scales, cbs = ops.pack(W)
    ocodes, oscales, ocbs = oracle.pack(W)
    assert np.array_equal(codes, ocodes) and np.array_equal(scales, oscales)
    assert np.array_equal(cbs, ocbs)


def test_missing_library_fails_loudly():
    # the binding raises at once when the shared library is absent (no
    # fallback, no hang in the error path)
    import subprocess
    import sys
    code = ("from bit_codebook_quantized_gb300 import ops\n"
            "ops.LIB_PATH = '/nonexistent/libcbq.so'\n"
            "try:\n    ops.lib()\nexcept ops.CbqError as e:\n    print('raised', e.status)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120,
                       cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert r.returncode == 0, r.stderr
    assert "raised -2" in r.stdout


def test_auto_path_choice(L):
    # host-only decision table (no device access)
    # without a workspace (cbq_gemm): only the kernels that need no scratch
    assert L.cbq_gemm_auto_path(1, 12288, 4096, 0) == ops.PATH_GEMV
    assert L.cbq_gemm_auto_path(8, 12288, 4096, 0) == ops.PATH_GEMV
    assert L.cbq_gemm_auto_path(1, 151936, 2048, 0) == ops.PATH_MMA
    assert L.cbq_gemm_auto_path(16, 25600, 5120, 0) == ops.PATH_MMA
    assert L.cbq_gemm_auto_path(64, 151936, 2048, 0) == ops.PATH_MMA
    # with one (cbq_gemm_ws): the stream-K kernel wherever its plan fits (the
    # plan here sees no device, i.e. one CTA holding every k-tile); at M = 64
    # with K = 25600 its resident activations do not fit
    for M, N, K in [(1, 12288, 4096), (8, 12288, 4096), (16, 25600, 5120),
                    (1, 151936, 2048), (64, 151936, 2048), (64, 300, 1024)]:
        assert L.cbq_gemm_auto_path(M, N, K, 1) == ops.PATH_STREAMK, (M, N, K)
    assert L.cbq_gemm_auto_path(64, 5120, 25600, 1) == ops.PATH_MMA
    # small matrices at up to 8 rows: the GEMV kernel either way
    for ws in (0, 1):
        assert L.cbq_gemm_auto_path(1, 2048, 2048, ws) == ops.PATH_GEMV
        assert L.cbq_gemm_auto_path(8, 4096, 8192, ws) == ops.PATH_GEMV
    assert L.cbq_gemm_auto_path(16, 2048, 2048, 1) == ops.PATH_STREAMK
    for ws in (0, 1):
        assert L.cbq_gemm_auto_path(0, 16, 128, ws) == ops.EINVAL
        assert L.cbq_gemm_auto_path(4, 16, 100, ws) == ops.EINVAL
        assert L.cbq_gemm_auto_path(65, 16, 128, ws) == ops.EINVAL


def test_workspace_size_covers_counters_and_partials(L):
    # a fixed area of 65536 4-byte tile counters, 64 4-byte token maxima and a
    # finished-CTA count (512 bytes after the counters; the same for every
    # shape), then two partial tiles of 128 x ntok fp32 per CTA (the plan here
    # sees no device: 1 CTA); the gate-up call adds M x F fp32 products
    fixed = 65536 * 4 + 512
    n = ctypes.c_size_t()
    assert L.cbq_gemm_workspace_size(8, 12288, 4096, ctypes.byref(n)) == ops.OK
    assert n.value == fixed + 2 * 1 * 128 * 16 * 4
    assert L.cbq_gemm_workspace_size(64, 300, 1024, ctypes.byref(n)) == ops.OK
    assert n.value == fixed + 2 * 1 * 128 * 64 * 4
    assert L.cbq_gate_up_workspace_size(8, 6144, 4096, ctypes.byref(n)) == ops.OK
    assert n.value == fixed + 2 * 1 * 128 * 16 * 4 + 8 * 6144 * 4
    assert L.cbq_gemm_workspace_size(64, 5120, 25600, ctypes.byref(n)) == ops.OK
    assert n.value == 0                       # no kernel with a workspace takes it
    # grouped: the same layout, planned for min(E, M topk) used experts
    assert L.cbq_grouped_workspace_size(128, 8, 64, 1536, 2048, ctypes.byref(n)) == ops.OK
    assert n.value == fixed + 2 * 1 * 128 * 64 * 4
    assert L.cbq_grouped_workspace_size(5000, 8, 64, 1536, 2048, ctypes.byref(n)) == ops.EINVAL


def test_draft_head_sizes(L):
    # the 2-bit head: KN/4 code bytes, KN/32 scale bytes, 4N codebook bytes
    c, sc, cb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert L.cbq_head2_sizes(151936, 2048, ctypes.byref(c), ctypes.byref(sc), ctypes.byref(cb)) == ops.OK
    assert (c.value, sc.value, cb.value) == (2048 * 151936 // 4, 2048 * 151936 // 32, 4 * 151936)
    assert L.cbq_head2_sizes(100, 96, ctypes.byref(c), ctypes.byref(sc), ctypes.byref(cb)) == ops.EINVAL
    # the draft-head workspace: the stream-K scratch (fixed area + two partial
    # tiles per CTA; 1 CTA without a device), the scores M x N fp32 and the
    # chunk lists M x ceil(N / 1024) x 16 words, each part rounded to 256 bytes
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    n = ctypes.c_size_t()
    for M, N, K in [(1, 151936, 2048), (8, 1030, 256), (64, 262144, 128)]:
        assert L.cbq_draft_head_workspace_size(M, N, K, ctypes.byref(n)) == ops.OK
        ntok = 16 if M <= 16 else (32 if M <= 32 else 64)
        want = r256(65536 * 4 + 512 + 2 * 128 * ntok * 4) + r256(M * N * 4) + r256(M * (-(-N // 1024)) * 16 * 8)
        assert n.value == want, (M, N, K)
    for M, N, K in [(0, 64, 128), (65, 64, 128), (1, 15, 128), (1, 262145, 128), (1, 64, 96), (1, 64, 0)]:
        assert L.cbq_draft_head_workspace_size(M, N, K, ctypes.byref(n)) == ops.EINVAL, (M, N, K)


def test_library_pack_matches_the_hand_worked_lloyd_row(golden_dir):
    # the library's quantiser (its own code) on the hand-worked Lloyd row
    from tests.test_oracle import lloyd_golden_row
    W, cb, sc = lloyd_golden_row(golden_dir)
    codes, scales, cbs = ops.pack(W)
    assert bytes(cbs.ravel()) == cb
    assert scales.ravel().tolist() == sc
