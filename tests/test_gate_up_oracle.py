"""The fused gate-up epilogue's oracle (oracle/gate_up.py) against a
hand-worked example, identities of SiLU, the quantisation's fixed points and
the block layout; planted mistakes fail the pins.  CPU only."""
import math
import os

import numpy as np
import pytest

from bit_codebook_quantized_gb300 import synth
from oracle import gate_up as og


def _golden(golden_dir):
    out = {}
    for line in open(os.path.join(golden_dir, "gate_up.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, *v = line.split()
            out[k] = v
    return out


def test_hand_worked_example(golden_dir):
    g = _golden(golden_dir)
    y = np.array([[float(v) for v in g["y"]]], np.float32)
    q, s, h = og.gate_up_from_y(y)
    assert h[0] == pytest.approx([float(v) for v in g["h"]], rel=1e-15)
    assert s[0] == pytest.approx(float(g["s"][0]), rel=1e-15)
    assert bytes(q[0]) == bytes(int(v, 16) for v in g["q"])


def test_silu_identities():
    # SiLU(x) - SiLU(-x) = x; SiLU(0) = 0; SiLU(x) ~ x for large x, ~ 0 for very negative x
    for x in [0.0, 1e-8, 0.3, 1.0, 2.5, 7.0, 30.0, 100.0]:
        assert og.silu(x) - og.silu(-x) == pytest.approx(x, rel=1e-14, abs=1e-300)
    assert og.silu(0.0) == 0.0
    assert og.silu(60.0) == pytest.approx(60.0, rel=1e-24)
    assert og.silu(-800.0) == 0.0
    # the derivative at 0 is 1/2: SiLU(x) / x -> sigmoid(0)
    assert og.silu(1e-9) / 1e-9 == pytest.approx(0.5, rel=1e-8)


def test_block_layout():
    # hand-listed (gate, up) rows: F = 100 -> blocks of 64 and 36 features
    F = 100
    assert og.rows_of_feature(F, 0) == (0, 64)
    assert og.rows_of_feature(F, 63) == (63, 127)
    assert og.rows_of_feature(F, 64) == (128, 164)
    assert og.rows_of_feature(F, 99) == (163, 199)
    rows = sorted(r for f in range(F) for r in og.rows_of_feature(F, f))
    assert rows == list(range(2 * F))          # every row used once


def test_quantisation_fixed_points():
    rng = synth.rng_for(3)
    y = (rng.standard_normal((5, 2 * 150)) * 3).astype(np.float32)
    y[4] = 0.0                                  # an all-zero token
    q, s, h = og.gate_up_from_y(y)
    for m in range(4):
        f = int(np.argmax(np.abs(h[m])))
        assert q[m, f] in (0x7E, 0xFE)          # the largest |h| lands on +-448
        assert s[m] == np.max(np.abs(h[m])) / 448.0
        # every code is the E4M3 value nearest h / s (the E4M3 table, by search)
        table = np.array([og.oracle.e4m3_value(b) if (b & 0x7F) != 0x7F else np.inf for b in range(256)])
        for f in range(0, 150, 7):
            x = h[m, f] / s[m]
            best = np.min(np.abs(table - x))
            assert abs(table[q[m, f]] - x) == best
    assert s[4] == 1.0 and np.all((q[4] & 0x7F) == 0)
    # scaling every up value by 2 doubles h and s and keeps the codes
    y2 = y.copy()
    F = 150
    for f in range(F):
        y2[:, og.rows_of_feature(F, f)[1]] *= 2
    q2, s2, _ = og.gate_up_from_y(y2)
    assert np.array_equal(q2, q) and np.allclose(s2[:4], 2 * s[:4], rtol=0, atol=0)


def _run_mutant(src_edit, golden_dir):
    """Load a copy of oracle/gate_up.py with one planted mistake and run the pins on it."""
    import types
    src = open(og.__file__).read()
    old, new = src_edit
    assert old in src
    mod = types.ModuleType("gate_up_mutant")
    exec(compile(src.replace(old, new), "gate_up_mutant", "exec"), mod.__dict__)
    g = _golden(golden_dir)
    y = np.array([[float(v) for v in g["y"]]], np.float32)
    try:
        q, s, h = mod.gate_up_from_y(y)
        ok = bytes(q[0]) == bytes(int(v, 16) for v in g["q"]) and \
            abs(h[0][0] - float(g["h"][0])) < 1e-12 and abs(s[0] - float(g["s"][0])) < 1e-15
        ok = ok and mod.rows_of_feature(100, 64) == (128, 164)
        ok = ok and abs(mod.silu(2.0) - mod.silu(-2.0) - 2.0) < 1e-14
    except Exception:
        ok = False
    return ok


MUTANTS = {
    "sigmoid_not_silu": ("return x / (1.0 + math.exp(-x))", "return 1.0 / (1.0 + math.exp(-x))"),
    "silu_of_up": ("h[m, f] = silu(float(y[m, gr])) * float(y[m, ur])",
                   "h[m, f] = float(y[m, gr]) * silu(float(y[m, ur]))"),
    "full_block_in_ragged_tail": ("R = min(BLOCK, F - BLOCK * b)", "R = BLOCK"),
    "int8_range": ("E4M3_MAX = 448.0", "E4M3_MAX = 127.0"),
    "scale_by_mean": ("amax = float(np.max(np.abs(h[m]))) if F else 0.0",
                      "amax = float(np.mean(np.abs(h[m]))) if F else 0.0"),
}


def test_pins_pass_on_the_real_oracle(golden_dir):
    assert _run_mutant(("BLOCK = 64", "BLOCK = 64"), golden_dir)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, golden_dir):
    assert not _run_mutant(MUTANTS[name], golden_dir), name
