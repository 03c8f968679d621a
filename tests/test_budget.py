"""Shared expert budget of a verify round ("Hibana: Fast Agentic Inference on
Unified-Memory Devices", section "Adaptive speculation / Expert sharing"):
the oracle against a hand-worked example, invariants and an independent
restatement; planted mistakes fail the pins.  CPU only."""
import numpy as np

from bit_codebook_quantized_gb300 import synth
from oracle import budget as ob


def _example():
    # Worked by hand: k = 2, B = 2.  Own top-2: t0 -> e0, e1; t1 -> e2, e3;
    # t2 -> e3, e1.  Scores (k - rank): e0 2, e1 1 + 1 = 2, e2 2, e3 1 + 2 = 3,
    # e4 0.  Budget: e3, then the lowest id of the tied e0, e1, e2 -> {0, 3}.
    # Choices inside it: t0 (e0 = 5, e3 = 0) -> [0, 3]; t1 (e3 = 4) -> [3, 0];
    # t2 (e3 = 5) -> [3, 0].
    logits = np.array([[5, 4, 0, 0, 0], [0, 0, 5, 4, 0], [0, 4, 0, 5, 0]], dtype=np.float32)
    return logits, 2, 2, [0, 3], [[0, 3], [3, 0], [3, 0]]


def test_hand_worked_example():
    logits, k, B, budget, topk = _example()
    assert ob.select_budget(logits, k, B) == (budget, topk)


def _random_logits(T, E, seed, ties=False):
    rng = synth.rng_for(seed)
    x = rng.standard_normal((T, E))
    if ties:
        x = np.round(x * 2)                       # few distinct values: many equal logits
    return x.astype(np.float32)


def test_full_budget_keeps_every_choice():
    for seed, (T, E, k) in enumerate([(6, 12, 2), (64, 128, 8), (9, 40, 5)]):
        logits = _random_logits(T, E, seed, ties=seed % 2 == 1)
        budget, topk = ob.select_budget(logits, k, E)
        assert budget == list(range(E))
        assert topk == ob.own_topk(logits, k)


def test_shared_choices_make_the_budget():
    # every token's own top-k is the same set S: with B = k the budget is S
    # and no choice is replaced
    rng = synth.rng_for(7)
    T, E, k = 10, 30, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    S = [3, 11, 17, 25]
    logits[:, S] += 10.0
    budget, topk = ob.select_budget(logits, k, k)
    assert budget == S
    assert topk == ob.own_topk(logits, k)


def test_invariants_and_independent_restatement():
    for seed, (T, E, k, B) in enumerate([(6, 12, 2, 4), (64, 128, 8, 24), (33, 100, 3, 3), (5, 17, 1, 17),
                                         (64, 300, 8, 40)]):
        for ties in (False, True):
            logits = _random_logits(T, E, 100 + seed, ties)
            budget, topk = ob.select_budget(logits, k, B)
            # the same rule through numpy sorts: lexsort keys (id, -logit) -> logit desc, id asc
            own = [list(np.lexsort((np.arange(E), -logits[t].astype(np.float64)))[:k]) for t in range(T)]
            score = np.zeros(E, np.int64)
            for t in range(T):
                for r, e in enumerate(own[t]):
                    score[e] += k - r
            want_budget = sorted(np.lexsort((np.arange(E), -score))[:B].tolist())
            assert budget == want_budget
            assert len(budget) == B and budget == sorted(set(budget))
            bset = set(budget)
            for t in range(T):
                ch = topk[t]
                assert len(set(ch)) == k and set(ch) <= bset
                key = [(-float(logits[t, e]), e) for e in ch]
                assert key == sorted(key)                          # in rank order
                worst = key[-1]
                for e in bset - set(ch):                           # nothing better left out
                    assert (-float(logits[t, e]), e) > worst


def test_pins_catch_planted_mistakes():
    logits, k, B, budget, topk = _example()

    def run(score_fn=None, tie_high=False):
        T, E = logits.shape
        own = ob.own_topk(logits, k)
        s = [0] * E
        for choices in own:
            for r, e in enumerate(choices):
                s[e] += score_fn(r) if score_fn else k - r
        order = sorted(range(E), key=lambda e: (-s[e], -e if tie_high else e))
        b = sorted(order[:B])
        return b

    assert run() == budget                                         # the rule as stated
    assert run(score_fn=lambda r: 1) != budget                     # plain votes
    assert run(score_fn=lambda r: k - r + 1) != budget             # rank weight off by one
    assert run(tie_high=True) != budget                            # ties to the higher id


def test_non_finite_and_signed_zero_logits():
    # Worked by hand, k = 3: row [1, NaN, 3, NaN, -inf, -0.0, +0.0]; NaN ranks
    # below every value (NaNs by id), -0 equals +0 (lower id first):
    # order 2 (3), 0 (1), 5 (-0), 6 (+0), 4 (-inf), 1 (NaN), 3 (NaN).
    row = np.array([[1, np.nan, 3, np.nan, -np.inf, -0.0, 0.0]], dtype=np.float32)
    assert ob.own_topk(row, 7) == [[2, 0, 5, 6, 4, 1, 3]]
    # the numpy restatement agrees: lexsort puts NaN last and keeps id order in ties
    assert list(np.lexsort((np.arange(7), -row[0].astype(np.float64)))) == [2, 0, 5, 6, 4, 1, 3]
    # a token whose logits are all NaN still gets k distinct in-budget choices
    x = _random_logits(8, 20, 3)
    x[2, :] = np.nan
    budget, topk = ob.select_budget(x, 4, 6)
    assert len(topk[2]) == 4 and len(set(topk[2])) == 4 and set(topk[2]) <= set(budget)
