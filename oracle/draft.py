"""Oracle for the adaptive draft length -- TEST INFRASTRUCTURE ONLY (tests may
import it; the library never does; no code is shared with it).

"Hibana: Fast Agentic Inference on Unified-Memory Devices", section
"Adaptive speculation / Adaptive draft length": a round drafts d tokens; each
drafted token is accepted with probability q (tracked per request); the round
yields the drafted tokens accepted before the first rejection plus one token
the target model produces itself, so the
expected tokens per round are E[N_d] = sum_{j=0..d} q^j = (1 - q^(d+1)) / (1 - q);
a round takes T(d) = 1 + c (d - 1) relative to a round with d = 1, c being the
added cost of one more draft token; the chosen length is
d* = argmax_{1 <= d <= dmax} E[N_d] / T(d).

Readings where the page is silent: ties go to the shorter draft (the first
maximum in increasing d); q = 1 uses the sum (E[N_d] = d + 1).  Floating point
decides an integer here, so ``draft_length`` takes that decision in double
precision with the sum accumulated in increasing j, the precision and order
the library uses; ``draft_length_exact`` is the same rule in exact rationals.
"""
from __future__ import annotations

from fractions import Fraction


def expected_tokens(q: float, d: int) -> float:
    """E[N_d] = sum_{j=0..d} q^j, summed in increasing j in double precision."""
    total, power = 0.0, 1.0
    for _ in range(d + 1):
        total += power
        power *= q
    return total


def round_time(c: float, d: int) -> float:
    """T(d) = 1 + c (d - 1)."""
    return 1.0 + c * (d - 1)


def draft_length(q: float, c: float, dmax: int):
    """(d*, E[N_d*], E[N_d*] / T(d*)) with ties to the shorter draft."""
    best = None
    for d in range(1, dmax + 1):
        e = expected_tokens(q, d)
        r = e / round_time(c, d)
        if best is None or r > best[2]:
            best = (d, e, r)
    return best


def expected_tokens_exact(q: Fraction, d: int) -> Fraction:
    """The page's closed form (1 - q^(d+1)) / (1 - q), and d + 1 at q = 1."""
    if q == 1:
        return Fraction(d + 1)
    return (1 - q ** (d + 1)) / (1 - q)


def draft_length_exact(q: Fraction, c: Fraction, dmax: int):
    best = None
    for d in range(1, dmax + 1):
        r = expected_tokens_exact(q, d) / (1 + c * (d - 1))
        if best is None or r > best[1]:
            best = (d, r)
    return best
