"""Adaptive draft length ("Hibana: Fast Agentic Inference on Unified-Memory
Devices", section "Adaptive speculation / Adaptive draft length"): the oracle
against the page's closed form and against cases with a closed-form answer,
then the library entry point against the oracle.  Host only (no GPU)."""
import ctypes
import math
from fractions import Fraction

import pytest

from bit_codebook_quantized_gb300 import ops
from oracle import draft

QS = [i / 20 for i in range(21)]
CS = [0.0, 0.01, 0.05, 0.1, 0.2, 0.3, 0.45, 0.5, 0.55, 0.7, 1.0, 2.0]
DMAX = [1, 2, 3, 4, 8, 16, 32, 63]


# ---- the oracle against the page ---------------------------------------------

def test_sum_equals_the_closed_form():
    # E[N_d] summed term by term vs (1 - q^(d+1)) / (1 - q) in exact rationals
    for q in QS:
        for d in range(0, 33):
            exact = draft.expected_tokens_exact(Fraction(q), d)
            assert draft.expected_tokens(q, d) == pytest.approx(float(exact), rel=1e-14, abs=0)


def test_no_acceptance_drafts_one():
    for c in CS:
        for dmax in DMAX:
            assert draft.draft_length(0.0, c, dmax)[0] == 1


def test_free_drafts_take_the_longest():
    # c = 0: E[N_d] grows with d for any q > 0, so d* = dmax (exactly); in
    # double precision once q^d drops below the sum's last bit the longer
    # drafts tie and the shorter one is kept, so check there only where q^dmax
    # stays well above it
    for q in QS[1:]:
        for dmax in DMAX:
            assert draft.draft_length_exact(Fraction(q), Fraction(0), dmax)[0] == dmax
            if q ** dmax > 1e-12:
                assert draft.draft_length(q, 0.0, dmax)[0] == dmax


def test_full_acceptance_closed_form():
    # q = 1: E[N_d] / T(d) = (d + 1) / (1 + c (d - 1)) grows with d iff c < 1/2,
    # is constant (a tie: the shorter draft) at c = 1/2, falls for c > 1/2
    for dmax in DMAX:
        assert draft.draft_length(1.0, 0.3, dmax)[0] == dmax
        assert draft.draft_length(1.0, 0.5, dmax)[0] == 1
        assert draft.draft_length(1.0, 0.6, dmax)[0] == 1
        d, e, r = draft.draft_length(1.0, 0.3, dmax)
        assert e == dmax + 1 and r == pytest.approx((dmax + 1) / (1 + 0.3 * (dmax - 1)), rel=1e-15)


def test_double_rule_equals_the_exact_rule():
    for q in QS:
        for c in CS:
            for dmax in DMAX:
                d_exact, r_exact = draft.draft_length_exact(Fraction(q), Fraction(c), dmax)
                # skip near-ties, where double rounding may pick either length
                others = [draft.expected_tokens_exact(Fraction(q), d) / (1 + Fraction(c) * (d - 1))
                          for d in range(1, dmax + 1) if d != d_exact]
                if others and min(abs(float(r_exact - o)) for o in others) < 1e-12 * float(r_exact):
                    continue
                assert draft.draft_length(q, c, dmax)[0] == d_exact


def test_higher_acceptance_never_shortens_the_draft():
    # the page's point that frequent acceptance warrants longer drafts:
    # E[N_(d+1)] / E[N_d] grows with q, so d* is non-decreasing in q (exact
    # rationals, no rounding)
    for c in CS:
        for dmax in DMAX:
            ds = [draft.draft_length_exact(Fraction(i, 40), Fraction(c), dmax)[0] for i in range(41)]
            assert ds == sorted(ds)


# ---- the library against the oracle -------------------------------------------

@pytest.mark.parametrize("dmax", DMAX)
def test_library_matches_the_oracle(dmax):
    for q in QS + [0.123456789, 0.987654321]:
        for c in CS + [0.0333]:
            assert ops.draft_length(q, c, dmax) == draft.draft_length(q, c, dmax), (q, c, dmax)


def test_library_rejects_bad_arguments():
    for q, c, dmax in [(-0.1, 0.1, 8), (1.1, 0.1, 8), (math.nan, 0.1, 8), (0.5, -0.1, 8),
                       (0.5, math.inf, 8), (0.5, math.nan, 8), (0.5, 0.1, 0), (0.5, 0.1, 64),
                       (0.5, 0.1, 2**31 - 1)]:
        with pytest.raises(ops.CbqError):
            ops.draft_length(q, c, dmax)
    assert ops.lib().cbq_draft_length(0.5, 0.1, 8, None, None, None) == ops.EINVAL
    d = ctypes.c_int32(0)
    assert ops.lib().cbq_draft_length(0.5, 0.1, 8, ctypes.byref(d), None, None) == ops.OK
    assert d.value == draft.draft_length(0.5, 0.1, 8)[0]


# ---- the pins catch plausible mistakes planted in a copy of the oracle ----------

def _pins_pass(mod):
    """The closed-form-answer pins above, run against an oracle module `mod`."""
    try:
        for q in QS:
            for d in range(0, 9):
                exact = mod.expected_tokens_exact(Fraction(q), d)
                assert mod.expected_tokens(q, d) == pytest.approx(float(exact), rel=1e-14, abs=0)
        for dmax in (2, 8):
            assert mod.draft_length(0.0, 0.1, dmax)[0] == 1
            assert mod.draft_length(1.0, 0.3, dmax)[0] == dmax
            assert mod.draft_length(1.0, 0.5, dmax)[0] == 1
            assert mod.draft_length(1.0, 0.6, dmax)[0] == 1
    except AssertionError:
        return False
    return True


def _mutant(**over):
    import types
    m = types.ModuleType("draft_mutant")
    for name in ("expected_tokens", "round_time", "draft_length", "expected_tokens_exact", "draft_length_exact"):
        setattr(m, name, getattr(draft, name))
    for name, fn in over.items():
        setattr(m, name, fn)
    # draft_length looks its helpers up in its own module: rebind it to the mutant's
    def draft_length(q, c, dmax, _m=m, _ties_longer=over.get("_ties_longer", False)):
        best = None
        for d in range(1, dmax + 1):
            e = _m.expected_tokens(q, d)
            r = e / _m.round_time(c, d)
            if best is None or r > best[2] or (_ties_longer and r == best[2]):
                best = (d, e, r)
        return best
    m.draft_length = draft_length
    return m


def test_pins_catch_planted_mistakes():
    assert _pins_pass(_mutant())                                   # the oracle as it is
    mutants = {
        "the target-produced token left out": _mutant(expected_tokens=lambda q, d: draft.expected_tokens(q, d) - 1.0),
        "one term too few": _mutant(expected_tokens=lambda q, d: draft.expected_tokens(q, d - 1) if d > 0 else 0.0),
        "round time 1 + c d": _mutant(round_time=lambda c, d: 1.0 + c * d),
        "ties to the longer draft": _mutant(_ties_longer=True),
        "q^(d+1) summed as q^d": _mutant(expected_tokens=lambda q, d: sum(q ** j for j in range(1, d + 2))),
    }
    for what, m in mutants.items():
        assert not _pins_pass(m), what
