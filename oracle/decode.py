"""One decode step of query-aware sparse-page attention, end to end, fp64.

For each (batch b, kv-head h) unit: build the page metadata from the K
pool, score every candidate page against the query, pick the exact top-k
plus the forced pages, and run exact attention of the group's query rows
over the selected pages.  Everything is recomputed from the raw K/V pool:
the oracle never reads metadata or indices produced elsewhere (except in
``attend_selection``, which takes a selection as an argument so that a
selection made elsewhere can be checked for its attention result).

Selectors
  quest   page score = group max of sum_i max(q_i m_i, q_i M_i)
          ("Quest 完全拆解", 核心机制); forced = sinks + recent pages.
  sketch  block score = LSE of dequantised int4 sketch logits over the
          block's tokens ("SALS长序列推理优化", QSI); forced = the tail
          block holding token L_b - 1 (n_sink = 0, n_recent = 1).
  probe   page score = largest q . k over n_probe uniformly sampled tokens
          of the page, max over the group ("Day 10·2 sparse top-k", §1-§2).
  all     every page (dense attention baseline).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import attention, probe, quest, select, sketch


@dataclass
class StepParams:
    page_size: int
    n_sel: int
    n_sink: int
    n_recent: int
    selector: str  # "quest" | "sketch" | "all"
    head_dim: int
    softmax_scale: float = 0.0  # 0 -> 1/sqrt(head_dim)
    top_p: float = 0.0  # adaptive budget: 0 = off (the fixed budget)
    min_pages: int = 0  # adaptive budget: fewest candidate pages kept
    n_probe: int = 8  # probe selector: sampled tokens per page
    meta_dtype: str = "f16"  # Quest over int8 keys: the stored metadata type (the query's)

    @property
    def tau(self) -> float:
        """Temperature of the page-score softmax of the adaptive budget: the
        sketch block score is already a log attention mass (1); the Quest
        bound is on the unscaled dot product, so it takes the softmax scale."""
        return 1.0 if self.selector == "sketch" else self.scale  # Quest and probe: dot products

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.head_dim)


@dataclass
class StepInputs:
    """Plain arrays: q [B][Hq][d]; pools [P_phys][Hkv][S][d]; scales [P_phys][Hkv][S] or None."""

    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: np.ndarray | None
    v_scale: np.ndarray | None
    page_table: np.ndarray
    seq_lens: np.ndarray
    proj: np.ndarray | None = None

    @property
    def group(self) -> int:
        return self.q.shape[1] // self.k_pool.shape[1]


def _group_rows(inp: StepInputs, b: int, h: int):
    G = inp.group
    return inp.q[b, h * G : (h + 1) * G]


def unit_quest_scores(inp: StepInputs, prm: StepParams, b: int, h: int) -> np.ndarray:
    """Scores of all pages [0, P_b) of unit (b, h) (forced pages included)."""
    L = int(inp.seq_lens[b])
    P = quest.num_pages(L, prm.page_size)
    m = np.empty((P, inp.k_pool.shape[-1]))
    M = np.empty_like(m)
    for p in range(P):
        phys = int(inp.page_table[b][p])
        t0, t1 = quest.page_token_range(p, prm.page_size, L)
        keys = np.asarray(inp.k_pool[phys, h, : t1 - t0]).astype(np.float64)
        if inp.k_scale is not None:  # int8 codes: dequantised, stored rounded outward
            keys = keys * np.asarray(inp.k_scale[phys, h, : t1 - t0]).astype(np.float64)[:, None]
            m[p] = quest.round_outward(keys.min(axis=0), prm.meta_dtype, down=True)
            M[p] = quest.round_outward(keys.max(axis=0), prm.meta_dtype, down=False)
            continue
        m[p] = keys.min(axis=0)
        M[p] = keys.max(axis=0)
    q_rows = np.asarray(_group_rows(inp, b, h)).astype(np.float64)
    return quest.group_scores(q_rows, m, M)


def unit_sketch_blocks(inp: StepInputs, prm: StepParams, b: int, h: int, blocks):
    """(codes [n][S][d_s], scales [n]) of the given full blocks of unit (b, h)."""
    codes, scales = [], []
    for p in blocks:
        phys = int(inp.page_table[b][p])
        if inp.k_scale is not None:
            kd = sketch.dequant(inp.k_pool[phys, h], inp.k_scale[phys, h])
        else:
            kd = np.asarray(inp.k_pool[phys, h]).astype(np.float32)
        c, s = sketch.build_sketch(kd, inp.proj)
        codes.append(c)
        scales.append(s)
    return codes, scales


def unit_sketch_scores(inp: StepInputs, prm: StepParams, b: int, h: int) -> np.ndarray:
    """Block scores of unit (b, h); the tail block (holding token L_b - 1) is NaN."""
    L = int(inp.seq_lens[b])
    P = quest.num_pages(L, prm.page_size)
    out = np.full(P, np.nan)
    if P == 0:
        return out
    blocks = list(range(P - 1))
    codes, scales = unit_sketch_blocks(inp, prm, b, h, blocks)
    qc, sq = sketch.index_query(_group_rows(inp, b, h), inp.proj)
    if blocks:
        out[: P - 1] = sketch.block_scores(qc, sq, codes, scales, prm.head_dim)
    return out


def unit_probe_scores(inp: StepInputs, prm: StepParams, b: int, h: int) -> np.ndarray:
    """Probe scores of all pages [0, P_b) of unit (b, h) (forced pages included)."""
    L = int(inp.seq_lens[b])
    P = quest.num_pages(L, prm.page_size)
    q_rows = np.asarray(_group_rows(inp, b, h)).astype(np.float64)
    out = np.empty(P)
    for p in range(P):
        phys = int(inp.page_table[b][p])
        if inp.k_scale is not None:
            keys = np.asarray(inp.k_pool[phys, h]).astype(np.float64) * \
                np.asarray(inp.k_scale[phys, h]).astype(np.float64)[:, None]
        else:
            keys = np.asarray(inp.k_pool[phys, h]).astype(np.float64)
        pos = probe.probe_positions(p, prm.page_size, L, prm.n_probe)
        out[p] = probe.probe_score(q_rows, keys, pos, p * prm.page_size)
    return out


def unit_scores(inp: StepInputs, prm: StepParams, b: int, h: int) -> np.ndarray:
    if prm.selector == "quest":
        return unit_quest_scores(inp, prm, b, h)
    if prm.selector == "sketch":
        return unit_sketch_scores(inp, prm, b, h)
    if prm.selector == "probe":
        return unit_probe_scores(inp, prm, b, h)
    raise ValueError(prm.selector)


def unit_selection(inp: StepInputs, prm: StepParams, b: int, h: int, scores=None) -> list[int]:
    L = int(inp.seq_lens[b])
    P = quest.num_pages(L, prm.page_size)
    if prm.selector == "all":
        return list(range(P))
    if scores is None:
        scores = unit_scores(inp, prm, b, h)
    if prm.top_p > 0.0:
        return select.select_pages_top_p(scores, P, prm.n_sel, prm.n_sink, prm.n_recent, prm.top_p,
                                         prm.min_pages, prm.tau)
    return select.select_pages(scores, P, prm.n_sel, prm.n_sink, prm.n_recent)


def attend_selection(inp: StepInputs, prm: StepParams, b: int, h: int, pages):
    """Attention of the group's query rows over the given logical pages."""
    L = int(inp.seq_lens[b])
    k = attention.gather_tokens(inp.k_pool, inp.k_scale, inp.page_table[b], pages, L, prm.page_size, h)
    v = attention.gather_tokens(inp.v_pool, inp.v_scale, inp.page_table[b], pages, L, prm.page_size, h)
    q_rows = np.asarray(_group_rows(inp, b, h)).astype(np.float64)
    return attention.attend(q_rows, k, v, prm.scale)


def decode_step(inp: StepInputs, prm: StepParams, units=None):
    """Selections, outputs and lse for the given (b, h) units (default: all).

    Returns dict(sel={(b, h): [pages]}, scores={(b, h): [P_b]},
                 out={(b, h): [G][d]}, lse={(b, h): [G]}).
    """
    B, Hq, d = inp.q.shape
    Hkv = inp.k_pool.shape[1]
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hkv)]
    res = {"sel": {}, "scores": {}, "out": {}, "lse": {}}
    for b, h in units:
        sc = None if prm.selector == "all" else unit_scores(inp, prm, b, h)
        sel = unit_selection(inp, prm, b, h, sc)
        out, lse = attend_selection(inp, prm, b, h, sel)
        res["sel"][(b, h)] = sel
        res["scores"][(b, h)] = sc
        res["out"][(b, h)] = out
        res["lse"][(b, h)] = lse
    return res
