"""Pins for the CPU oracle, checked against things other than itself:
library conversions (torch float8), hand-derived golden fixtures, closed
forms, exact rational brute force, invariants.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from bit_codebook_quantized_gb300 import synth


def _torch_e4m3(b):
    t = torch.tensor(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _lib_weights(pw):
    """w[n, k] from library conversions and Python big-int bit extraction."""
    N, K = pw.N, pw.K
    W = np.empty((N, K), dtype=np.float64)
    cbv = _torch_e4m3(pw.codebooks)
    flat = bytes(pw.codes.reshape(-1))
    for n in range(N):
        for g in range(K // 32):
            o = brute.group_offset(N, K, n, g)
            G = int.from_bytes(flat[o:o + 12], "little")
            sc = math.ldexp(1.0, int(pw.scales[n, g]) - 127)
            for j in range(32):
                W[n, 32 * g + j] = cbv[n, (G >> (3 * j)) & 7] * sc
    return W


# ---- number formats ----------------------------------------------------------

def test_e4m3_all_bytes_match_torch():
    ours = oracle.e4m3_table()
    ref = _torch_e4m3(np.arange(256))
    for b in range(256):
        if b in (0x7F, 0xFF):
            assert math.isnan(ours[b]) and math.isnan(ref[b])
        else:
            assert ours[b] == ref[b], hex(b)
            assert math.copysign(1.0, ours[b]) == math.copysign(1.0, ref[b]), hex(b)


def test_e4m3_golden(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "e4m3_values.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        b, v = line.split()[:2]
        b, v = int(b, 16), float(v)
        got = oracle.e4m3_value(b)
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(b)
            if b not in (0x7F, 0xFF):
                assert brute.e4m3(b) == v
        n += 1
    assert n == 14


def test_e8m0():
    for s in range(255):
        assert oracle.e8m0_value(s) == math.ldexp(1.0, s - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_e4m3_round_matches_torch_cast():
    rng = synth.rng_for(7)
    x = np.concatenate([
        rng.standard_normal(20000) * 3,
        rng.standard_normal(5000) * 1e-2,
        rng.uniform(-500, 500, 5000),
        np.ldexp(rng.uniform(-1, 1, 5000), -7),
    ]).astype(np.float32)
    ref = synth.to_e4m3_bytes(x)           # torch RNE (inputs clipped to 448)
    ours = np.array([oracle.e4m3_round(float(v)) for v in x], dtype=np.uint8)
    # +0 / -0 may differ only for values that round to zero
    both_zero = ((ours & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert np.all((ours == ref) | both_zero)


def test_e4m3_round_ties_and_saturation():
    r = oracle.e4m3_round
    assert r(1.0) == 0x38 and r(-1.0) == 0xB8
    assert r(1.0625) == 0x38          # halfway 1.0 / 1.125 -> even mantissa (0)
    assert r(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> even mantissa (2)
    assert r(2.0 ** -10) == 0x00      # half of the smallest subnormal -> 0
    assert r(3 * 2.0 ** -10) == 0x02  # halfway 2^-9 / 2^-8 -> even (2)
    assert r(460.0) == 0x7E and r(1e9) == 0x7E and r(-1e9) == 0xFE
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        v = oracle.e4m3_value(b)
        assert oracle.e4m3_value(r(v)) == v


# ---- bitstream ----------------------------------------------------------------

def test_bit_layout_golden(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "bit_layout.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, codes, hexbytes = [p.strip() for p in line.split(";")]
        idx = np.array([int(c) for c in codes.split()], dtype=np.int64).reshape(1, 32)
        want = bytes(int(h, 16) for h in hexbytes.split())
        got = oracle.codes_from_indices(idx)
        assert bytes(got.ravel()) == want, name
        for k in range(32):
            assert oracle.code_at(np.frombuffer(want, dtype=np.uint8), 1, 32, 0, k) == idx[0, k]
        n += 1
    assert n == 6


def test_bitstream_roundtrip_vs_bigint():
    rng = synth.rng_for(11)
    for N, K in [(5, 128), (130, 256)]:
        idx = rng.integers(0, 8, size=(N, K))
        packed = oracle.codes_from_indices(idx).reshape(-1)
        assert packed.size == 3 * K * N // 8
        seen = set()
        for n in range(N):
            for g in range(K // 32):
                G = sum(int(idx[n, 32 * g + j]) << (3 * j) for j in range(32))
                o = brute.group_offset(N, K, n, g)
                assert bytes(packed[o:o + 12]) == G.to_bytes(12, "little")
                seen.add(o)
        assert len(seen) == N * K // 32            # every group has its own 12 bytes
        assert np.array_equal(oracle.indices_from_codes(packed, N, K), idx)


def test_tile_layout_golden(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "tile_layout.txt")):
        if line.startswith("#") or not line.strip():
            continue
        N, K, row, g, off = map(int, line.split()[:5])
        assert oracle.group_offset(N, K, row, g) == off, line
        assert brute.group_offset(N, K, row, g) == off, line
        n += 1
    assert n == 12


# ---- footprint -----------------------------------------------------------------

def test_footprint_closed_form(golden_dir):
    n = 0
    for line in open(os.path.join(golden_dir, "footprint.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, K, N, c, s, b, tot = line.split()
        K, N, c, s, b, tot = map(int, (K, N, c, s, b, tot))
        pw = synth.gen_weights(1, K, seed=0)  # one row gives the per-row sizes
        assert pw.codes.nbytes * N == c and pw.scales.nbytes * N == s
        assert pw.codebooks.nbytes * N == b
        assert oracle.packed_bytes(N, K) == tot == c + s + b
        # 3 + 8/32 bits per weight, codebooks aside
        assert (c + s) * 8 == 3.25 * K * N
        n += 1
    assert n == 6


# ---- gemm against exact rationals ----------------------------------------------

SHAPES = [(1, 1, 32), (1, 3, 32), (2, 2, 64), (1, 8, 64), (4, 8, 64), (3, 5, 96), (4, 2, 32)]


def _random_case(M, N, K, seed, scale_lo=100, scale_hi=140):
    rng = synth.rng_for(seed)
    pw = synth.gen_weights(N, K, seed, scale_lo, scale_hi)
    # codebooks: any finite E4M3 byte, signs and subnormals included
    cb = rng.integers(0, 256, size=(N, 8), dtype=np.uint8)
    cb[(cb & 0x7F) == 0x7F] = 0x3F
    pw.codebooks = cb
    a = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x01
    a_scale = rng.uniform(-2, 2, size=M).astype(np.float32)
    return pw, a, a_scale


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_vs_exact_rationals(M, N, K):
    pw, a, a_scale = _random_case(M, N, K, seed=100 + M * 31 + N * 7 + K)
    y, bound = oracle.gemm(a, a_scale, pw.codes, pw.scales, pw.codebooks, M, N, K)
    exact = brute.gemm_exact(a, a_scale, pw.codes, pw.scales, pw.codebooks, M, N, K)
    for m in range(M):
        for n in range(N):
            e = float(exact[m][n])
            ref32 = np.float32(e)
            # one fp32 rounding (the oracle rounds a_scale*sum in double first)
            assert abs(float(y[m, n]) - float(ref32)) <= float(np.spacing(np.abs(ref32))), (m, n)
            absum = abs(float(a_scale[m])) * sum(
                abs(float(brute.e4m3(int(a[m][k])) * brute.weight(pw.codes, pw.scales,
                                                                  pw.codebooks, N, K, n, k)))
                for k in range(K))
            assert bound[m, n] == pytest.approx(absum, rel=1e-12, abs=0)


def test_unpack_matches_library_decode():
    pw = synth.gen_weights(16, 256, seed=3, scale_lo=110, scale_hi=140)
    W = oracle.unpack(pw.codes, pw.scales, pw.codebooks, pw.N, pw.K)
    ref = _lib_weights(pw)
    assert np.array_equal(W.astype(np.float64), ref)
    assert np.array_equal(np.signbit(W), np.signbit(ref))


def test_one_hot_activation_returns_weight_column():
    N, K = 12, 128
    pw = synth.gen_weights(N, K, seed=5)
    W = _lib_weights(pw)
    for k in (0, 1, 31, 32, 77, 127):
        a = np.zeros((1, K), dtype=np.uint8)
        a[0, k] = 0x38                       # E4M3 1.0
        y, _ = oracle.gemm(a, np.ones(1, np.float32), pw.codes, pw.scales, pw.codebooks, 1, N, K)
        assert np.array_equal(y[0].astype(np.float64), W[:, k])


def test_linearity_in_a():
    M, N, K = 3, 10, 256
    pw = synth.gen_weights(N, K, seed=9)
    a = synth.gen_activations(M, K, seed=10)
    s = synth.gen_a_scale(M, seed=11, mode="uniform")
    y1, b1 = oracle.gemm(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    y2, _ = oracle.gemm(a, 2 * s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    assert np.array_equal(y2, 2 * y1)        # scaling by 2 is exact
    # disjoint K supports: y(a1 + a2) = y(a1) + y(a2)
    a1 = a.copy(); a1[:, K // 2:] = 0
    a2 = a.copy(); a2[:, :K // 2] = 0
    ya1, _ = oracle.gemm(a1, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    ya2, _ = oracle.gemm(a2, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    assert np.all(np.abs((ya1.astype(np.float64) + ya2) - y1) <= 1e-6 * b1 + 1e-30)


def test_all_zero_codes_closed_form():
    M, N, K = 2, 6, 192
    pw = synth.gen_weights(N, K, seed=13, scale_lo=110, scale_hi=135)
    pw.codes[:] = 0
    a = synth.gen_activations(M, K, seed=14)
    s = synth.gen_a_scale(M, seed=15, mode="uniform")
    y, bound = oracle.gemm(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    av = _torch_e4m3(a)
    cb0 = _torch_e4m3(pw.codebooks[:, 0])
    gsum = av.reshape(M, K // 32, 32).sum(axis=2)                       # [M, G]
    sc = np.ldexp(1.0, pw.scales.astype(np.int64) - 127)                # [N, G]
    ref = s[:, None].astype(np.float64) * cb0[None, :] * (gsum @ sc.T)  # [M, N]
    assert np.all(np.abs(y - ref) <= 1e-6 * bound + 1e-30)
    pw.codebooks[:] = 0
    y0, _ = oracle.gemm(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    assert np.all(y0 == 0)


def test_grouped_equals_per_expert_gemm_and_reads_only_budget():
    E, N, K, M, budget, topk = 12, 16, 64, 6, 4, 2
    pw = synth.gen_weights(E * N, K, seed=21)
    a = synth.gen_activations(M, K, seed=22)
    s = synth.gen_a_scale(M, seed=23, mode="uniform")
    idx = synth.gen_moe_routing(M, E, budget, topk, seed=24)
    y, bound, reads = oracle.grouped_gemm(a, s, pw.codes, pw.scales, pw.codebooks, E, idx, M, N, K)
    used = set(int(e) for e in idx.ravel())
    assert len(used) <= budget
    assert set(np.nonzero(reads)[0].tolist()) == used
    for t in range(M):
        for j in range(topk):
            e = int(idx[t, j])
            ce, se, be = oracle.expert(pw.codes, pw.scales, pw.codebooks, e, N, K)
            ye, _ = oracle.gemm(a[t:t + 1], s[t:t + 1], ce, se, be, 1, N, K)
            assert np.array_equal(y[t, j], ye[0])
            ex = brute.gemm_exact(a[t:t + 1], s[t:t + 1], ce, se, be, 1, N, K)[0]
            for n in range(3):
                assert abs(float(y[t, j, n]) - float(np.float32(float(ex[n])))) <= \
                    float(np.spacing(np.float32(abs(float(ex[n])))))


def test_moe_routing_generator_properties():
    idx = synth.gen_moe_routing(64, 128, 24, 8, seed=3)
    assert idx.shape == (64, 8)
    assert len(set(idx.ravel().tolist())) <= 24
    for row in idx:
        assert len(set(row.tolist())) == 8


# ---- pack ---------------------------------------------------------------------

def test_group_scale_closed_form():
    w = np.zeros(32, np.float32)
    assert oracle.group_scale(w) == 127
    for e in range(-20, 20):
        w = np.zeros(32, np.float32)
        w[5] = -(2.0 ** e)                       # power of two: ceil(log2) = e
        assert oracle.group_scale(w) == 127 + e
        w[5] = 2.0 ** e * 1.0001                 # just above: e + 1
        assert oracle.group_scale(w) == 128 + e
        w[5] = 2.0 ** e * 0.75                   # in (2^(e-1), 2^e): e
        assert oracle.group_scale(w) == 127 + e
    w = np.full(32, 1e-45, np.float32)           # ~2^-149 -> clamp to 0
    assert oracle.group_scale(w) == 0
    w = np.full(32, 3e38, np.float32)            # ~2^128 -> 255 clamps to 254
    assert oracle.group_scale(w) == 254


def test_pack_nearest_assignment_is_optimal():
    W = synth.gen_dense_weights_fp32(6, 256, seed=31)
    codes, scales, cbs = oracle.pack(W)
    idx = oracle.indices_from_codes(codes, 6, 256)
    cbv = _torch_e4m3(cbs)
    assert np.all(np.diff(cbv, axis=1) >= 0)     # sorted codebooks
    for n in range(6):
        sc = np.ldexp(1.0, np.repeat(scales[n].astype(np.int64), 32) - 127)
        u = W[n].astype(np.float64) / sc
        assert np.all(np.abs(u) <= 1.0)
        d = np.abs(u[:, None] - cbv[n][None, :])          # [K, 8]
        best = d.min(axis=1)
        assert np.array_equal(d[np.arange(256), idx[n]], best)
        # ties go to the lower index
        first = np.argmax(d == best[:, None], axis=1)
        assert np.array_equal(idx[n], first)


def test_pack_is_exact_on_representable_weights():
    """Rows built from 8 distinct E4M3 values, each used K/8 times, every group
    holding a +-1.0 (so the scale rule recovers the group scale), pack to
    exactly themselves."""
    rng = synth.rng_for(41)
    N, K = 4, 256
    vals = np.array([-1.0, -0.5, -0.25, 0.0, 0.125, 0.25, 0.5, 1.0])
    W = np.empty((N, K), np.float32)
    for n in range(N):
        firsts = np.array([1.0, -1.0] * (K // 64))
        rest = np.concatenate([np.full(K // 8 - (K // 64), 1.0), np.full(K // 8 - (K // 64), -1.0)]
                              + [np.full(K // 8, v) for v in vals[1:-1]])
        rng.shuffle(rest)
        u = np.empty(K)
        u[0::32] = firsts
        mask = np.ones(K, bool); mask[0::32] = False
        u[mask] = rest
        s = rng.integers(110, 141, size=K // 32)
        W[n] = u * np.ldexp(1.0, np.repeat(s, 32) - 127)
    codes, scales, cbs = oracle.pack(W)
    back = oracle.unpack(codes, scales, cbs, N, K)
    assert np.array_equal(back, W)


def test_pack_ties_go_to_the_lower_index():
    """A row holding only -1 and +1: the quantile start puts four centroids on
    each value, every assignment is an exact tie, and ties go to the lowest
    index, so the codes are exactly 0 (for -1) and 4 (for +1)."""
    W = np.where(synth.rng_for(3).permutation(256) < 128, -1.0, 1.0).astype(np.float32)
    W = W.reshape(1, 256)
    codes, scales, cbs = oracle.pack(W)
    idx = oracle.indices_from_codes(codes, 1, 256)
    assert np.all(scales == 127)
    assert list(cbs[0]) == [0xB8] * 4 + [0x38] * 4
    assert np.array_equal(idx[0], np.where(W[0] < 0, 0, 4))


def test_gemm_rows_equals_full_gemm_rows():
    M, N, K = 3, 300, 256
    pw = synth.gen_weights(N, K, seed=51)
    a = synth.gen_activations(M, K, seed=52)
    s = synth.gen_a_scale(M, seed=53, mode="uniform")
    y, b = oracle.gemm(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K)
    rows = np.array([0, 1, 127, 128, 255, 256, 299])
    yr, br = oracle.gemm_rows(a, s, pw.codes, pw.scales, pw.codebooks, M, N, K, rows)
    assert np.array_equal(yr, y[:, rows]) and np.array_equal(br, b[:, rows])


def lloyd_golden_row(golden_dir):
    """The hand-worked Lloyd row of tests/golden/lloyd_row.txt: (W [1, 128],
    codebook bytes, scale bytes)."""
    from fractions import Fraction
    vals, cb, sc, inside = [], None, None, False
    for line in open(os.path.join(golden_dir, "lloyd_row.txt")):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        if line == "values":
            inside = True
        elif line == "end":
            inside = False
        elif inside:
            v, n = line.split()
            vals += [Fraction(v)] * int(n)
        elif line.startswith("codebook"):
            cb = bytes(int(x, 16) for x in line.split()[1:])
        elif line.startswith("scales"):
            sc = [int(x) for x in line.split()[1:]]
    S = sorted(vals)
    assert len(S) == 128
    row = [S[4 * j + g] for g in range(4) for j in range(32)]
    W = np.array([float(v) for v in row], np.float32).reshape(1, 128)
    assert all(Fraction(float(w)) == v for w, v in zip(W[0], row))   # exact in fp32
    return W, cb, sc


def test_pack_lloyd_fit_hand_worked_row(golden_dir):
    """Step 3 of the packer (quantile start, 16 rounds, empty cluster kept):
    a row whose fit still moves one point per round through round 16; the
    sorted E4M3 codebook and the scale bytes equal the hand-worked ones."""
    W, cb, sc = lloyd_golden_row(golden_dir)
    codes, scales, cbs = oracle.pack(W)
    assert bytes(cbs.ravel()) == cb
    assert scales.ravel().tolist() == sc
