"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the C oracle (on the CPU), builds it, and checks that at
least one pin from test_oracle.py-style checks fails on it."""
import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import brute
from bit_codebook_quantized_gb300 import synth

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "cbq_oracle.c")).read()

MUTANTS = {
    "e4m3_bias": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    "e4m3_subnormal": ("ldexp((double)m, -9)", "ldexp((double)m, -8)"),
    "e4m3_sign": ("return sign ? -v : v;", "return v;"),
    "code_bit_order": ("code |= bit << i;", "code |= bit << (2 - i);"),
    "code_group_offset": ("return tile_base + c * R * 48 + (n % 128) * W + (g % 4) * 12;",
                          "return tile_base + c * 128 * 48 + (n % 128) * W + (g % 4) * 12;"),
    "row_major_groups": ("return tile_base + c * R * 48 + (n % 128) * W + (g % 4) * 12;",
                         "return (n * (K / 32) + g) * 12;"),
    "partial_ktile_width": ("int64_t W = (G - 4 * c < 4) ? 12 * (G - 4 * c) : 48;",
                            "int64_t W = 48;"),
    "e8m0_bias": ("return ldexp(1.0, (int)s - 127);", "return ldexp(1.0, (int)s - 128);"),
    "dropped_abs_sign": ("acc += p;", "acc += fabs(p);"),
    "no_a_scale": ("y[m * N + n] = (float)((double)a_scale[m] * acc);", "y[m * N + n] = (float)acc;"),
    "reversed_k": ("double p = orc_e4m3_value(a[m * K + k]) *", "double p = orc_e4m3_value(a[m * K + (K - 1 - k)]) *"),
    "scale_of_next_group": ("scales[n * (K / 32) + k / 32]);", "scales[n * (K / 32) + (k / 32 + 1) % (K / 32)]);"),
    "pack_floor_log2": ("s = 127 + ((f == 0.5) ? ex - 1 : ex);", "s = 127 + ex - 1;"),
    "pack_tie_upper": ("if (fabs(u[k] - orc_e4m3_value(cb[c])) <\n                    fabs",
                       "if (fabs(u[k] - orc_e4m3_value(cb[c])) <=\n                    fabs"),
    "round_half_away": ("double r = nearbyint(sig);", "double r = floor(sig + 0.5);"),
    "lloyd_15_rounds": ("for (int it = 0; it < 16; it++)", "for (int it = 0; it < 15; it++)"),
    "lloyd_one_round": ("for (int it = 0; it < 16; it++)", "for (int it = 0; it < 1; it++)"),
    "lloyd_start_floor": ("cen[i] = sorted[(int64_t)((i + 0.5) * (double)K / 8.0)];",
                          "cen[i] = sorted[(int64_t)(i * (double)K / 8.0)];"),
    "lloyd_empty_reset": ("if (cnt[c] > 0)\n                    cen[c] = sum[c] / (double)cnt[c];",
                          "if (cnt[c] > 0)\n                    cen[c] = sum[c] / (double)cnt[c];\n"
                          "                else\n                    cen[c] = 0.0;"),
}


def _build(src: str, tag: str) -> ctypes.CDLL:
    d = tempfile.mkdtemp(prefix=f"orc_{tag}_")
    c = os.path.join(d, "m.c")
    so = os.path.join(d, "m.so")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC", c, "-o", so,
                    "-lm"], check=True)
    return oracle.configure(ctypes.CDLL(so))


def _pins_pass() -> bool:
    """A compact set of the oracle pins; False as soon as one fails."""
    import torch
    # E4M3 table vs torch
    ref = torch.tensor(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        v = oracle.e4m3_value(b)
        if b in (0x7F, 0xFF):
            if not math.isnan(v):
                return False
        elif v != ref[b] or math.copysign(1, v) != math.copysign(1, ref[b]):
            return False
    for sbyte in range(255):
        if oracle.e8m0_value(sbyte) != math.ldexp(1.0, sbyte - 127):
            return False
    # bit layout golden row (codes 0..7 repeated -> 88 c6 fa)
    idx = np.tile(np.arange(8), 4).reshape(1, 32)
    if bytes(oracle.codes_from_indices(idx).ravel()) != bytes.fromhex("88c6fa" * 4):
        return False
    g = np.frombuffer(bytes.fromhex("000000c0010000000000000000"[:24]), dtype=np.uint8)
    if oracle.code_at(g, 1, 32, 0, 10) != 7:
        return False
    # tile order of groups (hand-worked golden offsets)
    for N_, K_, n_, g_, off in [(130, 256, 129, 5, 12444), (130, 256, 5, 4, 6384),
                                (300, 384, 299, 5, 41052), (2, 96, 1, 2, 60)]:
        if oracle.group_offset(N_, K_, n_, g_) != off:
            return False
    # exact rationals on a tiny gemm
    M, N, K = 2, 3, 64
    pw = synth.gen_weights(N, K, 5, 100, 140)
    rng = synth.rng_for(6)
    a = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 1
    s = np.array([1.5, -0.75], np.float32)
    y, _ = oracle.gemm(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    ex = brute.gemm_exact(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    for m in range(M):
        for n in range(N):
            r = np.float32(float(ex[m][n]))
            if abs(float(y[m, n]) - float(r)) > float(np.spacing(np.abs(r))):
                return False
    # pack: scale rule and nearest assignment
    w = np.zeros(32, np.float32)
    w[3] = 4.0
    if oracle.group_scale(w) != 129:
        return False
    w[3] = 3.0
    if oracle.group_scale(w) != 129:
        return False
    # a two-valued row: duplicate centroids, every assignment is a tie
    W2 = np.where(np.arange(128) % 2 == 0, -1.0, 1.0).astype(np.float32).reshape(1, 128)
    c2, _, _ = oracle.pack(W2)
    if set(oracle.indices_from_codes(c2, 1, 128).ravel().tolist()) != {0, 4}:
        return False
    W = synth.gen_dense_weights_fp32(3, 128, 8)
    codes, scales, cbs = oracle.pack(W)
    cbv = torch.tensor(cbs).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ids = oracle.indices_from_codes(codes, 3, 128)
    for n in range(3):
        u = W[n].astype(np.float64) / np.ldexp(1.0, np.repeat(scales[n].astype(np.int64), 32) - 127)
        d = np.abs(u[:, None] - cbv[n][None, :])
        if not np.array_equal(ids[n], np.argmax(d == d.min(axis=1)[:, None], axis=1)):
            return False
    # E4M3 rounding ties go to the even mantissa
    if oracle.e4m3_round(1.0625) != 0x38 or oracle.e4m3_round(1.1875) != 0x3A:
        return False
    # the hand-worked Lloyd row (quantile start, 16 rounds, empty cluster kept)
    from tests.test_oracle import lloyd_golden_row
    Wl, cbl, scl = lloyd_golden_row(os.path.join(os.path.dirname(os.path.dirname(__file__)), "tests", "golden"))
    _, sl, bl = oracle.pack(Wl)
    if bytes(bl.ravel()) != cbl or sl.ravel().tolist() != scl:
        return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    # the anchor may appear in both gemm loops (all rows / listed rows): mutate every copy
    assert SRC.count(old) >= 1, f"mutation anchor for {name} missing"
    lib = _build(SRC.replace(old, new), name)
    saved = oracle._lib
    oracle._lib = lib
    try:
        assert not _pins_pass(), f"pins did not catch mutant {name}"
    finally:
        oracle._lib = saved
