"""Failure handling on the GPU without a fault: a kernel's bounded waits are
made to run out (a wait limit of a few nanoseconds), the kernel reports
CBQ_ETIMEOUT through cbq_device_status and returns, and the next normal call
on the same workspace is exact.  Also: cbq_gemm takes no device memory."""
import ctypes

import numpy as np
import pytest
import torch

from bit_codebook_quantized_gb300 import ops, synth
from tests.gpu_util import Case, assert_close, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("M,N,K", [(8, 12288, 4096), (16, 1000, 25600)])
def test_streamk_gives_up_then_the_next_call_is_exact(M, N, K):
    c = Case(M, N, K, seed=91 + M)
    a, s, w = c.device()
    y = torch.full((M, N), 3.0, device="cuda")
    ops.set_wait_limit(2)                    # the first wait not already satisfied gives up
    try:
        ops.gemm(a, s, w, out=y, path=ops.PATH_STREAMK)
        torch.cuda.synchronize()
    finally:
        ops.set_wait_limit(0)                # back to the default
    assert ops.device_status() == ops.ETIMEOUT
    assert ops.device_status() == ops.OK     # read once, then cleared
    y2 = ops.gemm(a, s, w, path=ops.PATH_STREAMK)   # the same cached workspace
    torch.cuda.synchronize()
    yref, b = c.oracle()
    assert_close(y2.cpu().numpy(), yref, b, "after a give-up")
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("path", [ops.PATH_GEMV, ops.PATH_MMA])
def test_gemv_and_tile_kernel_give_up_then_the_next_call_is_exact(path):
    c = Case(5, 3000, 2048, seed=95 + path)
    a, s, w = c.device()
    ops.set_wait_limit(2)
    try:
        ops.gemm(a, s, w, path=path)
        torch.cuda.synchronize()
    finally:
        ops.set_wait_limit(0)
    assert ops.device_status() == ops.ETIMEOUT
    y = ops.gemm(a, s, w, path=path)
    torch.cuda.synchronize()
    yref, b = c.oracle()
    assert_close(y.cpu().numpy(), yref, b, f"path {path} after a give-up")
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("path", [ops.PATH_MMA, ops.PATH_STREAMK])
def test_grouped_gives_up_then_the_next_call_is_exact(path):
    E, N, K, M = 12, 200, 512, 16
    pw = synth.gen_weights(E * N, K, 41)
    a = synth.gen_activations(M, K, 42)
    s = synth.gen_a_scale(M, 43, "uniform")
    idx = synth.gen_moe_routing(M, E, 6, 4, 44)
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N, K)
    da, ds, di = torch.from_numpy(a).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(idx).cuda()
    ops.set_wait_limit(2)
    try:
        ops.grouped_gemm(da, ds, w, E, di, path=path)
        torch.cuda.synchronize()
    finally:
        ops.set_wait_limit(0)
    assert ops.device_status() == ops.ETIMEOUT
    y = ops.grouped_gemm(da, ds, w, E, di, path=path)
    torch.cuda.synchronize()
    import oracle
    yref, b, _ = oracle.grouped_gemm(a, s, pw.codes, pw.scales, pw.codebooks, E, idx, M, N, K)
    assert_close(y.cpu().numpy(), yref, b, "grouped after a give-up")
    assert ops.device_status() == ops.OK


def test_cbq_gemm_takes_no_device_memory():
    # the verify-round up-projection shape, through the C entry point itself
    # (no workspace) on a fresh stream
    M, N, K = 16, 25600, 5120
    c = Case(M, N, K, seed=5)
    a, s, w = c.device()
    y = torch.empty((M, N), device="cuda")
    stream = torch.cuda.Stream()
    wt = w.struct()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc = ops.lib().cbq_gemm(a.data_ptr(), s.data_ptr(), ctypes.byref(wt), M, N, K, y.data_ptr(),
                                ctypes.c_void_p(stream.cuda_stream))
        assert rc == ops.OK
    stream.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    rows = np.arange(0, N, 97)
    yref, b = c.oracle_rows(rows)
    assert_close(y.cpu().numpy()[:, rows], yref, b, "cbq_gemm")
    assert ops.device_status() == ops.OK
