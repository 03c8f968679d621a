"""The allocation-free entry point (cbq_gemm_noalloc): the stream-K kernel on
the library's static device scratch.  Collected last; passes alone and after
the other GPU tests (its counters start at zero either way)."""
import numpy as np
import pytest
import torch

from bit_codebook_quantized_gb300 import ops
from tests.gpu_util import Case, assert_close, ensure_built, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("M,N,K", [(1, 200, 640), (8, 129, 256), (16, 1000, 384), (64, 300, 1024),
                                   (5, 40, 25600)])
def test_noalloc_matches_oracle(M, N, K):
    c = Case(M, N, K, seed=300 + M + N)
    a, s, w = c.device()
    y = torch.full((M, N), 7.0, device="cuda")
    ops.gemm_noalloc(a, s, w, y)
    torch.cuda.synchronize()
    yref, b = c.oracle()
    assert_close(y.cpu().numpy(), yref, b, f"noalloc M {M} N {N} K {K}")
    assert ops.device_status() == ops.OK


def test_noalloc_equals_streamk_bitwise_and_allocates_nothing():
    c = Case(8, 12288, 4096, seed=11)
    a, s, w = c.device()
    y1 = ops.gemm(a, s, w, path=ops.PATH_STREAMK)
    y2 = torch.empty_like(y1)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        ops.gemm_noalloc(a, s, w, y2)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == before
    assert free1 >= free0                      # no device memory taken by the calls
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    rows = sample_rows(c.N, 32, seed=12)
    yref, b = c.oracle_rows(rows)
    assert_close(y2.cpu().numpy()[:, rows], yref, b, "noalloc full size")


def test_noalloc_rejects_what_the_static_buffer_cannot_take():
    c = Case(64, 5120, 25600, seed=5)          # activations do not fit next to the ring
    a, s, w = c.device()
    y = torch.empty((64, 5120), device="cuda")
    with pytest.raises(ops.CbqError):
        ops.gemm_noalloc(a, s, w, y)
    a0 = torch.zeros((4, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.CbqError):          # K == 0 has nothing to stream
        ops.gemm_noalloc(a0, s[:4], ops.PackedWeights(w.codes, w.scales, w.codebooks, 8, 0), y)
