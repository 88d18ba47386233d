"""Exact top-k page selection with forced pages, fp64 scores.

Sources:
  * "SALS长序列推理优化", QSI Top-k 计算实现: the top-k must be exact (no
    approximate algorithm); it is built from a *stable* descending sort, so
    among equal scores the earlier block stays first; the fixed tail block
    indices are appended after the top-k (QSI step 5).
  * "Day 10·2 sparse top-k 块选择", 确定性红线 and top-k 补满: equal scores
    go to the lower block index, no randomness; when fewer than k blocks
    remain, selection simply stops.
  * "Quest 完全拆解", 三段式 kernel: Top-K filtering outputs page ids that
    index the sparse load of the attention kernel.

Reading: forced pages (sinks [0, n_sink) and the last n_recent pages) are
outside the candidate set and count toward the budget of n_sel pages; the
remaining k_top = n_sel - |forced| slots go to the candidates in order of
(score descending, page index ascending).  The result is the union, in
ascending page order.
"""

from __future__ import annotations

import math


def forced_pages(P: int, n_sink: int, n_recent: int) -> list[int]:
    f = set(range(min(n_sink, P))) | set(range(max(P - n_recent, 0), P))
    return sorted(f)


def select_pages(scores, P: int, n_sel: int, n_sink: int, n_recent: int) -> list[int]:
    """Selected logical pages of one (batch, kv-head), ascending.

    scores: indexable by page id (only candidate pages are read).
    """
    forced = forced_pages(P, n_sink, n_recent)
    fset = set(forced)
    cand = [p for p in range(P) if p not in fset]
    k_top = max(n_sel - len(forced), 0)
    ranked = sorted(cand, key=lambda p: (-float(scores[p]), p))
    return sorted(fset | set(ranked[:k_top]))


def top_p_count(cand_scores, top_p: float, tau: float) -> int:
    """Smallest k such that the k best candidates hold at least top_p of the
    softmax mass of all candidates.

    Source: "SequenceO1" close reading, §3.2 (STCA's relative threshold:
    keep the leading items whose cumulative importance reaches the fraction
    p of the total, p typically 0.8 to 0.95) and §4.2 (softmax of the sketch
    scores, sorted descending, cumulative sum, at least one item kept).
    cand_scores must already be in selection order (score descending, index
    ascending); the weights are exp(tau * (s - max s)) in fp64.  Returns
    len(cand_scores) when the running sum never reaches top_p * total (fp64
    rounding at p = 1).
    """
    s = [float(x) for x in cand_scores]
    if not s:
        return 0
    mx = max(s)
    w = [math.exp(tau * (x - mx)) for x in s]
    total = math.fsum(w)
    acc = 0.0
    for j, x in enumerate(w):
        acc += x
        if acc >= top_p * total:
            return j + 1
    return len(s)


def select_pages_top_p(scores, P: int, n_sel: int, n_sink: int, n_recent: int, top_p: float,
                       min_pages: int, tau: float) -> list[int]:
    """Selected logical pages with the adaptive (top-p) budget, ascending.

    The candidates are ranked as in select_pages; the fixed budget's k_top =
    n_sel - |forced| (at most the candidates) caps the count; within it the
    count is the top-p count of top_p_count, but at least min_pages
    candidates (SequenceO1 §4.2 keeps at least one).  top_p <= 0 turns the
    adaptive budget off (the fixed budget, as select_pages).
    """
    if top_p <= 0.0:
        return select_pages(scores, P, n_sel, n_sink, n_recent)
    forced = forced_pages(P, n_sink, n_recent)
    fset = set(forced)
    cand = [p for p in range(P) if p not in fset]
    k_budget = min(max(n_sel - len(forced), 0), len(cand))
    ranked = sorted(cand, key=lambda p: (-float(scores[p]), p))
    k_p = top_p_count([scores[p] for p in ranked], top_p, tau)
    k_top = min(k_budget, max(k_p, min(min_pages, k_budget)))
    return sorted(fset | set(ranked[:k_top]))
