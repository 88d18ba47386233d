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
