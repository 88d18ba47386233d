"""Exact softmax attention over a set of pages, fp64.

Sources: "SALS长序列推理优化", Sparse Flash Attention Antiquant (SFAA):
ordinary attention over the selected K/V, with int8 K and V dequantised by
their scales; "Quest 完全拆解", 三段式 kernel (Approximate attention loads
only the chosen pages into a FlashAttention-style kernel); "Day 10·2"
确定性红线: the softmax is renormalised over the selected blocks only.
The scale is 1/sqrt(d) ("SequenceO1" close reading §3.1).

Only tokens t < L_b of each page take part.  An empty token set gives a
zero output and lse = -inf.
"""

from __future__ import annotations

import math

import numpy as np

from .quest import page_token_range


def gather_tokens(pool, scale, page_table_row, pages, seq_len, page_size, h):
    """K (or V) rows of kv-head h for the valid tokens of the given pages, fp64."""
    rows = []
    for p in pages:
        phys = int(page_table_row[p])
        t0, t1 = page_token_range(p, page_size, seq_len)
        x = np.asarray(pool[phys, h, : t1 - t0, :]).astype(np.float64)
        if scale is not None:
            x = x * np.asarray(scale[phys, h, : t1 - t0]).astype(np.float64)[:, None]
        rows.append(x)
    if not rows:
        return np.zeros((0, np.asarray(pool).shape[-1]))
    return np.concatenate(rows, axis=0)


def attend(q_rows, k, v, scale):
    """softmax(q k^T * scale) v and the log-sum-exp of each row.

    q_rows [G][d], k/v [T][d] (fp64).  Returns (out [G][d], lse [G]).
    """
    q = np.asarray(q_rows, dtype=np.float64)
    G, d = q.shape
    if k.shape[0] == 0:
        return np.zeros((G, d)), np.full(G, -np.inf)
    z = np.einsum("gd,td->gt", q, k) * scale
    mx = z.max(axis=1, keepdims=True)
    w = np.exp(z - mx)
    den = w.sum(axis=1, keepdims=True)
    out = np.einsum("gt,td->gd", w / den, v)
    lse = mx[:, 0] + np.log(den[:, 0])
    return out, lse


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def lse_combine(parts):
    """Merge (out, lse) results of disjoint token sets into the result of their union.

    Each part is (out [G][d], lse [G]).  This is the reduction step that
    turns split rows back into one (SALS, AICPU Tiling challenge 2).
    """
    lses = np.stack([p[1] for p in parts])  # [n][G]
    outs = np.stack([p[0] for p in parts])  # [n][G][d]
    mx = lses.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    w = np.exp(lses - safe)  # [n][G]
    den = w.sum(axis=0)
    lse = np.where(den > 0, safe + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    out = np.einsum("ng,ngd->gd", w, outs) / np.where(den > 0, den, 1.0)[:, None]
    return out, lse
