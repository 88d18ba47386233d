"""Pins for the oracle's exact top-k with forced pages.

What fixes the answer: with distinct scores the top-k is the unique k-subset
of candidates with the largest score sum (checked by enumerating every
subset); with ties, the rule of the Day 10·2 page (确定性红线: equal scores go
to the lower block index) and the stable sort of the SALS QSI top-k give an
order-by-(score desc, index asc) characterisation, checked here as
invariants on inputs full of ties.
"""

import itertools

import numpy as np
import pytest

from oracle import select


def test_distinct_scores_match_best_subset(rng):
    for trial in range(40):
        P = int(rng.integers(1, 13))
        n_sink, n_recent = int(rng.integers(0, 3)), int(rng.integers(0, 3))
        n_sel = n_sink + n_recent + int(rng.integers(0, 6))
        scores = rng.permutation(P).astype(float) + rng.random(P) * 0.5
        sel = select.select_pages(scores, P, n_sel, n_sink, n_recent)
        forced = set(range(min(n_sink, P))) | set(range(max(P - n_recent, 0), P))
        cand = [p for p in range(P) if p not in forced]
        k = min(max(n_sel - len(forced), 0), len(cand))
        best = max(itertools.combinations(cand, k), key=lambda c: sum(scores[p] for p in c))
        assert sel == sorted(forced | set(best))


def _check_invariants(scores, P, n_sel, n_sink, n_recent, sel):
    forced = set(range(min(n_sink, P))) | set(range(max(P - n_recent, 0), P))
    cand = [p for p in range(P) if p not in forced]
    assert sel == sorted(set(sel)), "ascending and unique"
    assert forced <= set(sel)
    assert len(sel) == min(max(n_sel, len(forced)), P)
    chosen = [p for p in sel if p not in forced]
    rest = [p for p in cand if p not in set(sel)]
    for s in chosen:
        for u in rest:
            assert scores[s] > scores[u] or (scores[s] == scores[u] and s < u)


def test_ties_go_to_lower_index(rng):
    for trial in range(200):
        P = int(rng.integers(0, 40))
        n_sink, n_recent = int(rng.integers(0, 3)), int(rng.integers(0, 3))
        n_sel = n_sink + n_recent + int(rng.integers(0, 12))
        scores = rng.integers(0, 3, size=max(P, 1)).astype(float)
        sel = select.select_pages(scores, P, n_sel, n_sink, n_recent)
        _check_invariants(scores, P, n_sel, n_sink, n_recent, sel)


def test_all_equal_scores_pick_lowest_candidates():
    P = 20
    sel = select.select_pages(np.zeros(P), P, 6, 1, 2)
    assert sel == [0, 1, 2, 3, 18, 19]


def test_short_sequence_selects_every_page():
    for P in range(0, 9):
        assert select.select_pages(np.arange(P, dtype=float), P, 8, 1, 1) == list(range(P))


def test_sketch_tail_only_forcing():
    # SALS: the tail block is forced and never a candidate
    scores = np.array([5.0, 1.0, 4.0, 3.0, np.nan])
    assert select.select_pages(scores, 5, 3, 0, 1) == [0, 2, 4]


def test_dominant_needle_page_always_selected(rng):
    for trial in range(30):
        P = int(rng.integers(5, 60))
        scores = rng.standard_normal(P)
        needle = int(rng.integers(1, P - 1))
        scores[needle] = scores.max() + 1.0
        sel = select.select_pages(scores, P, 3, 1, 1)
        assert needle in sel


def test_planted_mistake_is_caught(rng, monkeypatch):
    """Reversing the tie rule must fail the tie invariant."""

    def upper_wins(scores, P, n_sel, n_sink, n_recent):
        forced = select.forced_pages(P, n_sink, n_recent)
        cand = [p for p in range(P) if p not in set(forced)]
        ranked = sorted(cand, key=lambda p: (-float(scores[p]), -p))
        return sorted(set(forced) | set(ranked[: max(n_sel - len(forced), 0)]))

    monkeypatch.setattr(select, "select_pages", upper_wins)
    with pytest.raises(AssertionError):
        test_ties_go_to_lower_index(rng)


# ---- adaptive (top-p) budget: SequenceO1 close reading §3.2 / §4.2 -----------

def _mass(scores, pages, tau):
    mx = max(scores)
    w = {p: np.exp(tau * (scores[p] - mx)) for p in range(len(scores))}
    return sum(w[p] for p in pages) / sum(w.values())


def test_top_p_count_is_the_smallest_subset_reaching_p(rng):
    """Brute force over every subset of a few candidates: the top-p count is
    the fewest pages whose softmax mass reaches p, and the chosen pages carry
    the largest mass among subsets of that size."""
    for trial in range(150):
        n = int(rng.integers(1, 9))
        scores = rng.standard_normal(n) * float(rng.choice([0.3, 1.0, 4.0]))
        tau = float(rng.choice([1.0, 0.5, 2.0]))
        p = float(rng.uniform(0.05, 0.99))
        sel = select.select_pages_top_p(scores, n, n, 0, 0, p, 0, tau)
        m_star = min(len(c) for r in range(1, n + 1) for c in itertools.combinations(range(n), r)
                     if _mass(scores, c, tau) >= p)
        assert len(sel) == m_star
        best = max(_mass(scores, c, tau) for c in itertools.combinations(range(n), m_star))
        assert _mass(scores, sel, tau) == pytest.approx(best, rel=1e-12)


def test_top_p_uniform_scores_closed_form():
    # equal weights: the count is ceil(p * n); ties keep the lowest indices
    for n, p, k in [(10, 0.45, 5), (10, 0.91, 10), (7, 0.2, 2), (100, 0.805, 81)]:
        sel = select.select_pages_top_p(np.zeros(n), n, n, 0, 0, p, 0, 1.0)
        assert sel == list(range(k))


def test_top_p_one_dominant_page_floor_and_cap():
    scores = np.array([0.0] * 30)
    scores[17] = 12.0  # e^12 against 29: above 99.9 % of the mass
    assert select.select_pages_top_p(scores, 30, 30, 0, 0, 0.99, 0, 1.0) == [17]
    # the floor keeps at least min_pages candidates (the §4.2 listing keeps one)
    assert select.select_pages_top_p(scores, 30, 30, 0, 0, 0.99, 3, 1.0) == [0, 1, 17]
    # p = 1 takes every candidate within the budget; the budget caps the count
    assert len(select.select_pages_top_p(scores, 30, 30, 0, 0, 1.0, 0, 1.0)) == 30
    assert len(select.select_pages_top_p(np.zeros(30), 30, 6, 1, 2, 0.9, 0, 1.0)) == 6


def test_top_p_forced_pages_and_off_switch(rng):
    for trial in range(50):
        P = int(rng.integers(1, 60))
        n_sink, n_recent = int(rng.integers(0, 3)), int(rng.integers(0, 3))
        n_sel = n_sink + n_recent + int(rng.integers(0, 20))
        scores = rng.standard_normal(P) * 3
        fixed = select.select_pages(scores, P, n_sel, n_sink, n_recent)
        assert select.select_pages_top_p(scores, P, n_sel, n_sink, n_recent, 0.0, 0, 1.0) == fixed
        adapt = select.select_pages_top_p(scores, P, n_sel, n_sink, n_recent, 0.8, 1, 1.0)
        forced = set(select.forced_pages(P, n_sink, n_recent))
        assert forced <= set(adapt) and set(adapt) <= set(fixed) and adapt == sorted(adapt)


def test_top_p_temperature_is_a_score_scale(rng):
    for trial in range(30):
        P = int(rng.integers(2, 40))
        s = rng.standard_normal(P)
        a = select.select_pages_top_p(s, P, P, 0, 0, 0.7, 0, 0.5)
        b = select.select_pages_top_p(s * 0.5, P, P, 0, 0, 0.7, 0, 1.0)
        assert a == b
