"""Oracle for the shared expert budget of a verify round -- TEST INFRASTRUCTURE
ONLY (tests may import it; the library never does; no code is shared).

"Hibana: Fast Agentic Inference on Unified-Memory Devices", section
"Adaptive speculation / Expert sharing": checking a round of drafted tokens has
to read every expert chosen by at least one of them; limiting the whole round
to one common set of experts cuts the bytes read, and a token whose choice
falls outside the set takes its best expert inside it instead.  The page
illustrates this on a small example only, so the rule here is a proposal, each
step the plainest reading and every decision a comparison or an integer sum
(so two implementations agree exactly):

1. each token ranks the experts by its router logit (higher first, equal
   logits -> lower expert id) and takes its own top-k;
2. expert e scores sum over tokens of (k - r) where r is e's rank (0-based)
   in that token's own top-k (a first choice counts k, a k-th choice 1);
3. the budget is the B experts with the highest score (ties -> lower id);
4. each token's final choices are its top-k among the budget experts, in
   its own rank order (the same comparison as step 1).
"""
from __future__ import annotations

import math

import numpy as np


def _rank_key(row, e):
    """Sort key of expert e in a token's ranking: higher logit first, equal
    logits -> lower id (float32 values compared exactly, -0 equal to +0).  The
    page says nothing of non-finite logits; the reading taken here is that a
    NaN logit ranks below every other value, NaNs among themselves by id."""
    v = float(row[e])
    return (1, 0.0, e) if math.isnan(v) else (0, -v, e)


def _ranked(row, experts):
    return sorted(experts, key=lambda e: _rank_key(row, e))


def own_topk(logits: np.ndarray, k: int) -> list[list[int]]:
    T, E = logits.shape
    return [_ranked(logits[t], range(E))[:k] for t in range(T)]


def scores(logits: np.ndarray, k: int) -> list[int]:
    E = logits.shape[1]
    s = [0] * E
    for choices in own_topk(logits, k):
        for r, e in enumerate(choices):
            s[e] += k - r
    return s


def select_budget(logits: np.ndarray, k: int, B: int):
    """(budget as ascending expert ids [B], topk_idx [T][k] in rank order)."""
    T, E = logits.shape
    assert 1 <= k <= B <= E and T >= 1
    s = scores(logits, k)
    budget = sorted(sorted(range(E), key=lambda e: (-s[e], e))[:B])
    topk = [_ranked(logits[t], budget)[:k] for t in range(T)]
    return budget, topk
