"""GPU parity of the fused gate-up epilogue (cbq_gemm_gate_up) against the
oracle (oracle/gate_up.py), through the C ABI.

Tolerance, derived from the arithmetic: the matmul outputs g, u agree with
the oracle's within eps = 1e-3 * B + 1e-6 (B = |a_scale| sum|a w|, the
matmul tolerance); |d SiLU / dg| <= 1.1, so h = SiLU(g) u moves by at most
dh = 1.1 (|u| + eps_u) eps_g + (|SiLU(g)| + 1.1 eps_g) eps_u.  The dequantised
output E4M3(q) * s must then lie within half an E4M3 step of h / s (times s)
plus dh of the oracle's h; the largest |h| of a token (when it leads the
next by more than 2 dh) must be coded as +-448 exactly, and the scale must
be within max(dh) / 448 of the oracle's."""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_codebook_quantized_gb300 import ops, synth
from oracle import gate_up as og
from tests.gpu_util import Case, ensure_built

pytestmark = pytest.mark.gpu

E4M3 = np.array([oracle.e4m3_value(b) for b in range(256)])


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def half_step(x):
    """Half the E4M3 spacing at magnitude |x| (subnormal spacing 2^-9 below 2^-6)."""
    ax = np.maximum(np.abs(x), 1e-300)
    e = np.floor(np.log2(ax))
    return np.where(ax < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))


def check_gate_up(q, s, a, a_scale, pw, M, F, K, what):
    qr, sr, hr, y, bound = og.gate_up(a, a_scale, pw.codes, pw.scales, pw.codebooks, M, 2 * F, K)
    eps = 1e-3 * bound + 1e-6
    gi = np.array([og.rows_of_feature(F, f)[0] for f in range(F)])
    ui = np.array([og.rows_of_feature(F, f)[1] for f in range(F)])
    g, u = y[:, gi].astype(np.float64), y[:, ui].astype(np.float64)
    eg, eu = eps[:, gi], eps[:, ui]
    silu_g = np.vectorize(og.silu)(g)
    dh = 1.1 * (np.abs(u) + eu) * eg + (np.abs(silu_g) + 1.1 * eg) * eu + 1e-6 * np.abs(hr)
    s = np.asarray(s, np.float64)
    assert np.all(np.abs(s - sr) <= dh.max(axis=1) / 448.0 + 1e-6 * sr), f"{what}: scale"
    d = E4M3[q.astype(np.int64)] * s[:, None]
    x_hi = (np.abs(hr) + dh) / s[:, None]
    lim = half_step(x_hi) * s[:, None] + dh
    bad = np.abs(d - hr) > lim
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside; first {np.argwhere(bad)[0]}: "
                           f"got {d[bad][0]!r} want {hr[bad][0]!r} lim {lim[bad][0]!r}")
    for m in range(M):
        order = np.argsort(-np.abs(hr[m]))
        if F > 1 and abs(hr[m, order[0]]) - abs(hr[m, order[1]]) > 2 * dh[m].max():
            assert q[m, order[0]] in (0x7E, 0xFE), f"{what}: token {m} max not coded as 448"


@pytest.mark.parametrize("M,F,K", [(3, 100, 640), (1, 64, 128), (16, 200, 384), (33, 70, 256)])
def test_gate_up_small(M, F, K):
    c = Case(M, 2 * F, K, seed=700 + M + F)
    c.a[M - 1] = 0                              # an all-zero token: scale 1, codes +-0
    a, s, w = c.device()
    h, hs = ops.gate_up(a, s, w)
    torch.cuda.synchronize()
    q, sc = h.cpu().numpy(), hs.cpu().numpy()
    assert sc[M - 1] == 1.0 and np.all((q[M - 1] & 0x7F) == 0)
    check_gate_up(q, sc, c.a, c.s, c.pw, M, F, K, f"gate-up M {M} F {F} K {K}")
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("name,M", [("decode_4096x12288_m8", 8), ("decode_4096x12288_m1", 1),
                                    ("verify_up_5120x25600_m16", 16)])
def test_gate_up_full_size(name, M):
    wl = synth.workloads()[name]
    c = Case(M, wl.N, wl.K, seed=77 + M, a_scale=wl.a_scale, half_normal=wl.half_normal)
    a, s, w = c.device()
    h, hs = ops.gate_up(a, s, w)
    h2, hs2 = ops.gate_up(a, s, w)              # twice in a row: the workspace maxima were cleared
    torch.cuda.synchronize()
    assert torch.equal(h, h2) and torch.equal(hs, hs2)
    check_gate_up(h.cpu().numpy(), hs.cpu().numpy(), c.a, c.s, c.pw, M, wl.N // 2, wl.K, name)
    assert ops.device_status() == ops.OK


@pytest.mark.parametrize("M,F,K", [(3, 100, 640), (16, 1100, 384)])
def test_gate_up_gives_up_then_the_next_call_is_exact(M, F, K):
    # quantised by the matmul's last CTA (M F <= 8192) and by the separate
    # kernel (M F > 8192): after a forced give-up every CTA still counts
    # itself, so the per-token maxima and the count of finished CTAs are back
    # to zero and the next call on the same workspace is exact
    c = Case(M, 2 * F, K, seed=800 + M + F)
    a, s, w = c.device()
    ops.set_wait_limit(2)                      # the first wait not already satisfied gives up
    try:
        ops.gate_up(a, s, w)
        torch.cuda.synchronize()
    finally:
        ops.set_wait_limit(0)
    assert ops.device_status() == ops.ETIMEOUT
    h, hs = ops.gate_up(a, s, w)
    torch.cuda.synchronize()
    check_gate_up(h.cpu().numpy(), hs.cpu().numpy(), c.a, c.s, c.pw, M, F, K, f"after a give-up, M {M} F {F}")
    assert ops.device_status() == ops.OK


def test_gate_up_rejects_bad_arguments():
    c = Case(2, 128, 128, seed=3)
    a, s, w = c.device()
    L = ops.lib()
    import ctypes
    wt = w.struct()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    h = torch.empty((2, 64), dtype=torch.uint8, device="cuda")
    hs = torch.empty(2, device="cuda")
    args = lambda M, F, K, wsb: (a.data_ptr(), s.data_ptr(), ctypes.byref(wt), M, F, K, h.data_ptr(),  # noqa: E731
                                 hs.data_ptr(), ws.data_ptr(), wsb, None)
    assert L.cbq_gemm_gate_up(*args(2, 64, 100, ws.numel())) == ops.EINVAL     # K % 128
    assert L.cbq_gemm_gate_up(*args(0, 64, 128, ws.numel())) == ops.EINVAL     # M
    assert L.cbq_gemm_gate_up(*args(2, 64, 128, 1024)) == ops.EINVAL           # workspace too small
    assert L.cbq_gemm_gate_up(*args(2, 64, 128, ws.numel())) == ops.OK
    torch.cuda.synchronize()
    assert ops.device_status() == ops.OK
