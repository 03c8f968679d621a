"""Pins of the two-bit draft-head oracle (CPU): hand-worked bit layouts, group
offsets, shortlists and picks (tests/golden/draft_head.txt), the footprint
closed form, exact rationals on tiny shapes, one-hot and linearity of the
FP8 rescoring -- and planted mistakes in copies of the oracle that each fail
a pin."""
import ctypes
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import draft_head as dh
from bit_codebook_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "draft_head.txt")


def _golden():
    groups, offsets, shortlists, picks = [], [], [], []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = (x.strip() for x in line.split("->"))
        kind, *args = lhs.split()
        if kind == "group":
            groups.append(([int(c) for c in args[0].split(",")], bytes.fromhex(rhs)))
        elif kind == "offset":
            offsets.append((tuple(int(x) for x in args), int(rhs)))
        elif kind == "shortlist":
            shortlists.append((int(args[0]), [float(x) for x in args[1].split(",")],
                               [int(x) for x in rhs.split(",")]))
        elif kind == "pick":
            picks.append(([int(x) for x in args[0].split(",")], [float(x) for x in args[1].split(",")], int(rhs)))
    return groups, offsets, shortlists, picks


def _e4m3_exact(b: int) -> Fraction:
    """E4M3 from the format rule, as an exact rational (NaN bytes excluded)."""
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def _code_from_bytes(codes: np.ndarray, off: int, j: int) -> int:
    """Code j of the 64-bit little-endian group starting at byte off."""
    v = int.from_bytes(bytes(codes[off:off + 8]), "little")
    return (v >> (2 * j)) & 3


def _exact_scores(a, a_scale, codes, scales, cbs, M, N, K):
    out = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                off = oracle._load().orc_group_offset2(N, K, n, k // 32)
                c = _code_from_bytes(codes, off, k % 32)
                w = _e4m3_exact(int(cbs[n * 4 + c])) * Fraction(2) ** (int(scales[n * (K // 32) + k // 32]) - 127)
                acc += _e4m3_exact(int(a[m, k])) * w
            out[m][n] = Fraction(float(a_scale[m])) * acc
    return out


def _tiny_head(N, K, seed):
    rng = synth.rng_for(seed)
    codes = rng.integers(0, 256, size=K * N // 4, dtype=np.uint8)
    scales = rng.integers(118, 131, size=N * (K // 32), dtype=np.uint8)
    cbs = rng.integers(0, 256, size=N * 4, dtype=np.uint8)
    cbs[(cbs & 0x7F) == 0x7F] = 0x38
    return codes, scales, cbs


def _head_pins_pass(shortlist_fn=dh.shortlist, pick_fn=dh.pick) -> bool:
    lib = oracle._load()
    groups, offsets, shortlists, picks = _golden()
    # bit layout of a group
    for codes, raw in groups:
        buf = np.frombuffer(raw, dtype=np.uint8).copy()
        if [lib.orc_code2(buf.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), 1, 32, 0, k) for k in range(32)] \
                != codes:
            return False
    # tile order of groups
    for (N, K, n, g), off in offsets:
        if lib.orc_group_offset2(N, K, n, g) != off:
            return False
    # footprint: 2 + 8/32 bits per weight, 4 codebook bytes per row
    c, s, b = dh.footprint_bytes(200, 416)
    if Fraction(8 * (c + s), 200 * 416) != Fraction(9, 4) or b != 800:
        return False
    # exact rationals, ragged tile and partial k-tile (N = 130, K = 160)
    M, N, K = 2, 130, 160
    codes, scales, cbs = _tiny_head(N, K, 3)
    rng = synth.rng_for(4)
    a = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x30
    asc = np.array([1.25, -0.5], np.float32)
    y, bound = dh.scores(a, asc, codes, scales, cbs, M, N, K)
    ex = _exact_scores(a, asc, codes, scales, cbs, M, N, [K][0])
    for m in range(M):
        for n in (0, 1, 64, 127, 128, 129):
            r = np.float32(float(ex[m][n]))
            if abs(float(y[m, n]) - float(r)) > float(np.spacing(np.abs(r))):
                return False
    # FP8 rescoring: one-hot activations give row_scale * w8 exactly;
    # doubling a_scale doubles the logits exactly
    Nh, Kh = 5, 64
    head8 = synth.rng_for(5).integers(0, 256, size=(Nh, Kh), dtype=np.uint8)
    head8[(head8 & 0x7F) == 0x7F] = 0x40
    rs = np.array([0.5, 2.0, 1.0, 0.25, 4.0], np.float32)
    a1 = np.zeros((1, Kh), np.uint8)
    a1[0, 7] = 0x38                                            # 1.0
    rows = np.array([[4, 0, 2]], np.int32)
    lg, _ = dh.rescore(a1, np.ones(1, np.float32), head8, rs, rows, 1, Nh, Kh)
    for i, n in enumerate(rows[0]):
        if lg[0, i] != np.float32(float(rs[n]) * float(_e4m3_exact(int(head8[n, 7])))):
            return False
    a2 = synth.rng_for(6).integers(0, 120, size=(1, Kh), dtype=np.uint8)
    l1, _ = dh.rescore(a2, np.array([1.5], np.float32), head8, rs, rows, 1, Nh, Kh)
    l2, _ = dh.rescore(a2, np.array([3.0], np.float32), head8, rs, rows, 1, Nh, Kh)
    if not np.array_equal(l2, 2 * l1):
        return False
    # shortlist and pick
    for L, sc, want in shortlists:
        if shortlist_fn(np.array([sc], np.float32), L)[0].tolist() != want:
            return False
    for rws, lgs, want in picks:
        if int(pick_fn(np.array([rws]), np.array([lgs], np.float32))[0]) != want:
            return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _head_pins_pass()


def test_shortlist_invariants():
    rng = synth.rng_for(11)
    s = np.round(rng.standard_normal((3, 500)) * 4).astype(np.float32)   # many ties
    rows = dh.shortlist(s)
    for m in range(3):
        v = s[m, rows[m]]
        assert len(set(rows[m].tolist())) == 16
        assert np.all(np.diff(v) <= 0)                                    # descending
        for i in range(15):                                               # equal -> lower id first
            if v[i] == v[i + 1]:
                assert rows[m, i] < rows[m, i + 1]
        assert np.all(np.delete(s[m], rows[m]) <= v[-1])                  # nothing better left out


C_MUTANTS = {
    "code2_bit_order": ("        int pos = 2 * j + i;", "        int pos = 2 * j + (1 - i);"),
    "offset2_tile_base": ("    int64_t tile_base = 128 * t * (K / 4);", "    int64_t tile_base = 128 * t * (K / 2);"),
    "offset2_partial_ktile": ("    int64_t W = (G - 4 * c < 4) ? 8 * (G - 4 * c) : 32;",
                              "    int64_t W = 32;"),
    "codebook2_stride": ("    return orc_e4m3_value(codebooks[n * 4 + c]) *", "    return orc_e4m3_value(codebooks[n * 8 + c]) *"),
    "rescore_no_row_scale": ("(double)((n >= 0 && n < N) ? row_scale[n] : 0.0f)", "(double)((n >= 0 && n < N) ? 1.0f : 0.0f)"),
}


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_pins_catch_c_mutant(name):
    from tests.test_oracle_mutations import SRC, _build
    old, new = C_MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name}"
    lib = _build(SRC.replace(old, new), name)
    saved = oracle._lib
    oracle._lib = lib
    try:
        assert not _head_pins_pass(), f"pins did not catch mutant {name}"
    finally:
        oracle._lib = saved


def _shortlist_ties_upper(s, L=16):
    s = np.asarray(s, np.float32)
    return np.array([np.lexsort((-np.arange(s.shape[1]), -s[m].astype(np.float64)))[:min(L, s.shape[1])]
                     for m in range(s.shape[0])], np.int32)


def _pick_ties_later(rows, logits):
    out = np.empty(rows.shape[0], np.int32)
    for m in range(rows.shape[0]):
        best = 0
        for i in range(1, rows.shape[1]):
            if logits[m, i] >= logits[m, best]:
                best = i
        out[m] = rows[m, best]
    return out


def test_pins_catch_python_mutants():
    assert not _head_pins_pass(shortlist_fn=_shortlist_ties_upper)
    assert not _head_pins_pass(pick_fn=_pick_ties_later)
