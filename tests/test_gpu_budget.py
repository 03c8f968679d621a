"""GPU parity of cbq_select_budget (the shared expert budget of a verify
round) against the oracle, exact: every decision is a comparison of the same
fp32 logits or an integer sum.  Then the chosen routing drives the grouped
matmul."""
import numpy as np
import pytest
import torch

import oracle
from bit_codebook_quantized_gb300 import ops, synth
from oracle import budget as ob
from tests.gpu_util import assert_close, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _logits(T, E, seed, ties):
    rng = synth.rng_for(seed)
    x = rng.standard_normal((T, E))
    if ties:
        x = np.round(x * 2)
    return x.astype(np.float32)


@pytest.mark.parametrize("T,E,k,B", [(1, 12, 2, 4), (6, 12, 2, 4), (64, 128, 8, 24), (64, 4096, 8, 64),
                                     (33, 100, 3, 3), (5, 17, 1, 17), (70, 257, 8, 31), (16, 256, 4, 40)])
@pytest.mark.parametrize("ties", [False, True])
def test_budget_matches_the_oracle(T, E, k, B, ties):
    logits = _logits(T, E, T * 1000 + E + k + B, ties)
    budget, topk = ops.select_budget(torch.from_numpy(logits).cuda(), k, B)
    torch.cuda.synchronize()
    want_budget, want_topk = ob.select_budget(logits, k, B)
    assert budget.cpu().tolist() == want_budget
    assert topk.cpu().tolist() == want_topk
    assert ops.device_status() == ops.OK


def test_budget_non_finite_logits_match_the_oracle():
    # NaN ranks below every value, -0 equals +0, infinities order normally;
    # a row of NaNs still yields k distinct budget experts
    logits = _logits(40, 96, 9, True)
    logits[0, [3, 7, 50]] = np.nan
    logits[1, :] = np.nan
    logits[2, [0, 1]] = [np.inf, -np.inf]
    logits[3, :] = 0.0
    logits[3, ::2] = -0.0
    budget, topk = ops.select_budget(torch.from_numpy(logits).cuda(), 8, 20)
    torch.cuda.synchronize()
    want_budget, want_topk = ob.select_budget(logits, 8, 20)
    assert budget.cpu().tolist() == want_budget
    assert topk.cpu().tolist() == want_topk
    assert ops.device_status() == ops.OK


def test_budget_rejects_bad_arguments():
    x = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    for k, B in [(0, 4), (5, 4), (2, 17), (9, 12)]:
        with pytest.raises(ops.CbqError):
            ops.select_budget(x, k, B)
    with pytest.raises(ops.CbqError):
        ops.select_budget(torch.zeros((2, 4097), dtype=torch.float32, device="cuda"), 2, 4)


def test_budget_routing_drives_the_grouped_matmul():
    # a verify round: router logits -> budget and routing -> one grouped call
    E, N, K, M, k, B = 16, 80, 256, 12, 2, 5
    logits = _logits(M, E, 5, False)
    pw = synth.gen_weights(E * N, K, 11)
    a = synth.gen_activations(M, K, 12)
    s = synth.gen_a_scale(M, 13, "uniform")
    budget, topk = ops.select_budget(torch.from_numpy(logits).cuda(), k, B)
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N, K)
    y = ops.grouped_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(s).cuda(), w, E, topk)
    torch.cuda.synchronize()
    idx = topk.cpu().numpy()
    assert set(np.unique(idx)) <= set(budget.cpu().tolist())
    yref, bound, reads = oracle.grouped_gemm(a, s, pw.codes, pw.scales, pw.codebooks, E, idx, M, N, K)
    assert_close(y.cpu().numpy(), yref, bound, "budget routing")
    assert ops.device_status() == ops.OK
