"""GPU parity of the two-bit draft head (cbq_gemm2_ws, cbq_draft_head) against
the oracle.  The 2-bit scores are compared element by element within the
stated fp32 tolerance.  The shortlist and the pick are decisions taken on
floating-point values, so each is compared exactly against the oracle's rule
applied to the GPU's own values (the scores from cbq_gemm2_ws -- the same
kernel and plan as inside cbq_draft_head, so bit-identical -- and the GPU's
FP8 logits); the FP8 logits are compared with the oracle's rescoring of the
same rows within the tolerance."""
import numpy as np
import pytest
import torch

from bit_codebook_quantized_gb300 import ops, synth
from oracle import draft_head as dh
from tests.gpu_util import assert_close, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _case(M, N, K, seed, zero_codebooks=False):
    h2 = synth.gen_head2(N, K, seed)
    if zero_codebooks:
        h2.codebooks[:] = 0
    h8, rs = synth.gen_head8(N, K, seed + 1)
    a = synth.gen_activations(M, K, seed + 2)
    s = synth.gen_a_scale(M, seed + 3, "uniform")
    return h2, h8, rs, a, s


def _device(h2, h8, rs, a, s):
    w = ops.PackedWeights.from_host(h2.codes, h2.scales, h2.codebooks, h2.N, h2.K)
    return (w, torch.from_numpy(h8).cuda(), torch.from_numpy(rs).cuda(), torch.from_numpy(a).cuda(),
            torch.from_numpy(s).cuda())


def _check_head(M, N, K, seed, zero_codebooks=False):
    h2, h8, rs, a, s = _case(M, N, K, seed, zero_codebooks)
    w, dh8, drs, da, ds = _device(h2, h8, rs, a, s)
    y = ops.gemm2(da, ds, w)
    rows, logits, pick = ops.draft_head(da, ds, w, dh8, drs)
    torch.cuda.synchronize()
    assert ops.device_status() == ops.OK
    y, rows, logits, pick = y.cpu().numpy(), rows.cpu().numpy(), logits.cpu().numpy(), pick.cpu().numpy()
    # scores: every element against the oracle
    yref, b = dh.scores(a, s, h2.codes, h2.scales, h2.codebooks, M, N, K)
    assert_close(y, yref, b, f"2-bit scores {M}x{N}x{K}")
    # the shortlist: the oracle's rule on the GPU's scores, exactly
    assert np.array_equal(rows, dh.shortlist(y)), "shortlist"
    # the FP8 logits of those rows; the pick on the GPU's logits, exactly
    lref, lb = dh.rescore(a, s, h8, rs, rows, M, N, K)
    assert_close(logits, lref, lb, "FP8 logits")
    assert np.array_equal(pick, dh.pick(rows, logits)), "pick"
    return rows


@pytest.mark.parametrize("M,N,K", [(1, 200, 640), (3, 130, 256), (16, 1000, 384), (64, 300, 1024), (8, 16, 128),
                                   (2, 1024, 128), (2, 1030, 256), (1, 16 * 1024 + 7, 128), (4, 40000, 256),
                                   (2, 100000, 256), (1, 150000, 128), (1, 262144, 128)])
def test_draft_head_small(M, N, K):
    _check_head(M, N, K, seed=M + N + K)


def test_draft_head_all_scores_equal():
    # all-zero codebooks: every 2-bit score is 0, so the shortlist is rows 0..15
    rows = _check_head(2, 500, 256, seed=3, zero_codebooks=True)
    assert rows.tolist() == [list(range(16))] * 2


@pytest.mark.parametrize("name", sorted(synth.draft_head_workloads()))
def test_draft_head_full_size(name):
    wl = synth.draft_head_workloads()[name]
    _check_head(wl.M, wl.N, wl.K, seed=77)


def test_draft_head_gives_up_then_the_next_call_is_exact():
    # the 2-bit matmul gives up (its scores are then incomplete); the
    # shortlist kernels still read in-bounds rows (a word always carries a
    # real row), and the next call on the same workspace is exact
    M, N, K = 2, 3000, 512
    h2, h8, rs, a, s = _case(M, N, K, 5)
    w, dh8, drs, da, ds = _device(h2, h8, rs, a, s)
    ops.set_wait_limit(2)                      # the first wait not already satisfied gives up
    try:
        ops.draft_head(da, ds, w, dh8, drs)
        torch.cuda.synchronize()
    finally:
        ops.set_wait_limit(0)
    assert ops.device_status() == ops.ETIMEOUT
    _check_head(M, N, K, seed=5)


def test_draft_head_rejects_bad_arguments():
    L = ops.lib()
    import ctypes
    n = ctypes.c_size_t()
    assert L.cbq_draft_head_workspace_size(1, 15, 128, ctypes.byref(n)) == ops.EINVAL     # N < 16
    assert L.cbq_draft_head_workspace_size(1, 64, 96, ctypes.byref(n)) == ops.EINVAL      # K % 128
    assert L.cbq_draft_head_workspace_size(65, 64, 128, ctypes.byref(n)) == ops.EINVAL    # M > 64
    assert L.cbq_draft_head_workspace_size(1, 262145, 128, ctypes.byref(n)) == ops.EINVAL  # N > 256 chunks
    assert L.cbq_draft_head_workspace_size(1, 262144, 128, ctypes.byref(n)) == ops.OK
    h2, h8, rs, a, s = _case(1, 64, 128, 1)
    w, dh8, drs, da, ds = _device(h2, h8, rs, a, s)
    out = torch.empty(64, 16, dtype=torch.int32, device="cuda")
    wt = w.struct()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    assert L.cbq_draft_head(da.data_ptr(), ds.data_ptr(), ctypes.byref(wt), dh8.data_ptr() + 1, drs.data_ptr(), 1,
                            64, 128, out.data_ptr(), out.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                            None) == ops.EINVAL                                          # head8 misaligned
    assert L.cbq_draft_head(da.data_ptr(), ds.data_ptr(), ctypes.byref(wt), dh8.data_ptr(), drs.data_ptr(), 1,
                            64, 128, out.data_ptr(), out.data_ptr(), out.data_ptr(), ws.data_ptr(), 1024,
                            None) == ops.EINVAL                                          # workspace too small
