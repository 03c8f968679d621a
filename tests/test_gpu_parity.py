"""GPU parity: the CUDA kernels against the CPU oracle on the same seeded
inputs.  Bit-exact for unpack and for one-hot activations; fp32 results
within |y - y_ref| <= 1e-3 * |a_scale| * sum|a*w| + 1e-6 elsewhere."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from bit_codebook_quantized_gb300 import ops, synth
from tests.gpu_util import Case, assert_close, ensure_built, sample_rows

pytestmark = pytest.mark.gpu

PATHS = [ops.PATH_GEMV, ops.PATH_MMA, ops.PATH_STREAMK]
GROUPED_PATHS = [ops.PATH_GEMV, ops.PATH_MMA, ops.PATH_STREAMK]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


# ---- unpack ------------------------------------------------------------------

@pytest.mark.parametrize("N,K,lo,hi", [(37, 384, 120, 127), (300, 4096, 0, 254), (1, 128, 1, 1)])
def test_unpack_bit_exact(N, K, lo, hi):
    pw = synth.gen_weights(N, K, seed=N + K, scale_lo=lo, scale_hi=hi)
    # include negative, subnormal and zero codebook entries
    pw.codebooks[0] = [0x80, 0x00, 0x01, 0x07, 0x08, 0xB8, 0x7E, 0xFE][:8]
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N, K)
    W = ops.unpack(w)
    torch.cuda.synchronize()
    ref = oracle.unpack(pw.codes, pw.scales, pw.codebooks, N, K)
    assert np.array_equal(W.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ---- small shapes, every M, both kernels ---------------------------------------

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 16, 24, 33, 64])
def test_gemm_small(path, M):
    # N = 200: 12 full 16-row slabs + a ragged slab, and 1 full + 1 ragged 128-row tile
    # K = 640: 5 chunks of 128, i.e. a ragged last pipeline stage
    c = Case(M, 200, 640, seed=1000 + M)
    y = c.run(path)
    yref, b = c.oracle()
    assert_close(y, yref, b, f"path {path} M {M}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("N,K", [(16, 128), (1, 128), (129, 256), (2048, 2048), (40, 25600)])
def test_gemm_shapes(path, N, K):
    c = Case(3, N, K, seed=N * 7 + K)
    y = c.run(path)
    yref, b = c.oracle()
    assert_close(y, yref, b, f"path {path} N {N} K {K}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("lo,hi", [(100, 150), (0, 3)])
def test_one_hot_is_bit_exact(path, lo, hi):
    # (0, 3): E8M0 0 (2^-127) and weights that are fp32 subnormals
    N, K = 150, 512
    c = Case(8, N, K, seed=5, scale_lo=lo, scale_hi=hi)
    ks = [0, 1, 31, 32, 100, 255, 256, 511]
    c.a[:] = 0
    for m, k in enumerate(ks):
        c.a[m, k] = 0x38                      # E4M3 1.0
    c.s[:] = 1.0
    y = c.run(path)
    W = oracle.unpack(c.pw.codes, c.pw.scales, c.pw.codebooks, N, K)
    for m, k in enumerate(ks):
        assert np.array_equal(y[m].view(np.uint32), W[:, k].view(np.uint32)), (m, k)


@pytest.mark.parametrize("path", PATHS)
def test_zero_codes_and_zero_codebook(path):
    c = Case(4, 70, 384, seed=9)
    c.pw.codes[:] = 0
    y = c.run(path)
    yref, b = c.oracle()
    assert_close(y, yref, b, "all-zero codes")
    c2 = Case(4, 70, 384, seed=9)
    c2.pw.codebooks[:] = 0
    assert np.all(c2.run(path) == 0)


@pytest.mark.parametrize("path", PATHS)
def test_a_scale_linearity(path):
    c = Case(5, 64, 256, seed=17)
    y1 = c.run(path)
    a, s, w = c.device()
    y2 = ops.gemm(a, s * 2, w, path=path).cpu().numpy()
    assert np.array_equal(y2, 2 * y1)


def test_streamk_many_parts_deterministic():
    # K = 25600 over one 40-row tile: ~150 SMs share the tile's 200 k-tiles,
    # the last to arrive sums every part; two runs agree bit for bit
    c = Case(5, 40, 25600, seed=77)
    y1 = c.run(ops.PATH_STREAMK)
    y2 = c.run(ops.PATH_STREAMK)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    yref, b = c.oracle()
    assert_close(y1, yref, b, "many parts")
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("M,N,K", [(3, 150000, 128), (2, 150000, 256), (5, 40000, 256)])
def test_streamk_fewer_k_tiles_than_mma_groups(M, N, K):
    # one or two k-tiles per row and up to 15 units per CTA: each of the three
    # MMA groups steps through the resident activation slots modulo K / 128
    c = Case(M, N, K, seed=N + K + M)
    yref, b = c.oracle()
    assert_close(c.run(ops.PATH_STREAMK), yref, b, f"M {M} N {N} K {K}")
    assert ops.device_status() == ops.OK


def test_streamk_shape_sequence_on_one_stream():
    # tile counters are back to zero after every call, whatever the shape; a
    # call with many tiles (129, and 96 at the decode shape) after calls that
    # wrote partial tiles into the same workspace finds its counters at zero
    cases = [Case(1, 300, 1024, seed=81), Case(16, 1000, 384, seed=82), Case(64, 129, 2048, seed=83),
             Case(2, 16461, 512, seed=84), Case(1, 12288, 1024, seed=85)]
    for c in cases + cases[::-1]:
        yref, b = c.oracle()
        assert_close(c.run(ops.PATH_STREAMK), yref, b, f"M {c.M} N {c.N} K {c.K}")
    assert ops.device_status() == ops.OK


def test_streamk_rejects_what_does_not_fit():
    # 64 token columns x 53 k-tiles of resident activations per SM do not fit
    c = Case(64, 5120, 25600, seed=5)
    a, s, w = c.device()
    with pytest.raises(ops.CbqError):
        ops.gemm(a, s, w, path=ops.PATH_STREAMK)
    rows = sample_rows(c.N, 24, seed=6)
    yref, b = c.oracle_rows(rows)
    assert_close(c.run(ops.PATH_AUTO)[:, rows], yref, b, "auto falls back to the tile kernel")


def test_auto_path_matches_both_kernels():
    for M in (1, 4, 5, 8, 16):
        c = Case(M, 96, 256, seed=40 + M)
        yref, b = c.oracle()
        assert_close(c.run(ops.PATH_AUTO), yref, b, f"auto M {M}")


def test_empty_and_zero_k():
    a = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(4, device="cuda")
    pw = synth.gen_weights(8, 128, 1)
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, 8, 0)
    y = torch.full((4, 8), 7.0, device="cuda")
    ops.gemm(a, s, w, out=y)                 # K = 0 -> y = 0
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    w0 = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, 0, 128)
    ops.gemm(a, s, w0, out=y)                # N = 0 -> nothing happens
    assert ops.device_status() == ops.OK


# ---- full workload sizes, every element ----------------------------------------

FULL = ["gemv_2048", "decode_4096x12288_m1", "decode_4096x12288_m2", "decode_4096x12288_m4",
        "decode_4096x12288_m8", "verify_up_5120x25600_m16", "verify_down_25600x5120_m16",
        "vocab_head_2048x151936_m1", "vocab_head_2048x151936_m8", "vocab_head_2048x151936_m64"]

_full_cache = {}


def full_case(name):
    """The workload's seeded case and its oracle result (computed once)."""
    if name not in _full_cache:
        wl = synth.workloads()[name]
        c = Case(wl.M, wl.N, wl.K, seed=zlib.crc32(name.encode()) % 1000, a_scale=wl.a_scale,
                 half_normal=wl.half_normal)
        _full_cache.clear()                  # keep one workload's arrays at a time
        _full_cache[name] = (c, c.oracle())
    return _full_cache[name]


@pytest.mark.parametrize("path", [ops.PATH_AUTO, ops.PATH_MMA, ops.PATH_GEMV])
@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name, path):
    """Every output of the workload against the oracle: the automatic choice
    with a workspace (the stream-K kernel where it fits), the tile kernel,
    and the GEMV kernel on the workloads it is chosen for without one."""
    c, (yref, b) = full_case(name)
    if path == ops.PATH_GEMV and c.M > 8:
        pytest.skip("the GEMV kernel is chosen only up to 8 token rows")
    try:
        y = c.run(path)
    except ops.CbqError as e:
        assert path == ops.PATH_MMA and e.status == ops.EINVAL   # activations do not fit
        return
    assert_close(y, yref, b, f"{name} path {path}")
    assert ops.device_status() == ops.OK


# ---- grouped (MoE verify round) ---------------------------------------------------

def _grouped_case(E, N, K, M, budget, topk, seed):
    pw = synth.gen_weights(E * N, K, seed)
    a = synth.gen_activations(M, K, seed + 1)
    s = synth.gen_a_scale(M, seed + 2, "uniform")
    idx = synth.gen_moe_routing(M, E, budget, topk, seed + 3)
    return pw, a, s, idx


def _run_grouped(pw, a, s, idx, E, N, K, path=ops.PATH_AUTO):
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N, K)
    y = ops.grouped_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(s).cuda(), w, E,
                         torch.from_numpy(idx).cuda(), path=path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("path", GROUPED_PATHS)
@pytest.mark.parametrize("E,N,K,M,budget,topk", [(12, 80, 256, 6, 4, 2), (16, 33, 384, 64, 16, 8),
                                                  (5, 16, 128, 1, 1, 1), (6, 300, 640, 20, 3, 2)])
def test_grouped_small(path, E, N, K, M, budget, topk):
    pw, a, s, idx = _grouped_case(E, N, K, M, budget, topk, seed=E + N + M)
    y = _run_grouped(pw, a, s, idx, E, N, K, path)
    yref, b, reads = oracle.grouped_gemm(a, s, pw.codes, pw.scales, pw.codebooks, E, idx, M, N, K)
    assert_close(y, yref, b, "grouped")
    assert ops.device_status() == ops.OK


_grouped_full = {}


@pytest.mark.parametrize("path", GROUPED_PATHS)
def test_grouped_full_size_every_element(path):
    wl = synth.workloads()["moe_verify_e128_2048x1536_m64"]
    E, N, K, M = wl.experts, wl.N, wl.K, wl.M
    if not _grouped_full:
        pw, a, s, idx = _grouped_case(E, N, K, M, wl.budget, wl.topk, seed=321)
        yref, b, reads = oracle.grouped_gemm(a, s, pw.codes, pw.scales, pw.codebooks, E, idx, M, N, K)
        _grouped_full["case"] = (pw, a, s, idx, yref, b)
    pw, a, s, idx, yref, b = _grouped_full["case"]
    y = _run_grouped(pw, a, s, idx, E, N, K, path)
    assert_close(y, yref, b, f"grouped full size path {path}")
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("path", GROUPED_PATHS)
def test_grouped_routing_errors_are_reported(path):
    E, N, K, M = 4, 16, 128, 2
    pw, a, s, idx = _grouped_case(E, N, K, M, 4, 2, seed=8)
    bad = idx.copy()
    bad[1, 0] = 9                              # outside [0, E)
    _run_grouped(pw, a, s, bad, E, N, K, path)
    assert ops.device_status() == ops.EROUTING
    dup = idx.copy()
    dup[0, 1] = dup[0, 0]                      # one token lists an expert twice
    _run_grouped(pw, a, s, dup, E, N, K, path)
    assert ops.device_status() == ops.EROUTING
    assert ops.device_status() == ops.OK       # the status is cleared once read
