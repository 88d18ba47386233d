"""Quest page metadata and page criticality bound, fp64.

Source: "Quest 完全拆解：查询感知的页级稀疏注意力" (pinghaoyang.com.cn),
sections 核心机制 (the per-dimension bound U_i = max(q_i m_i, q_i M_i) and
its two-case proof) and 关键性估计算法 (incremental M_i <- max(M_i, k_i),
m_i <- min(m_i, k_i) on insert; score = sum_i max(q_i M_i, q_i m_i) at
attention time).  GQA handling follows the same page's "GQA 下的并集放大"
section: one selection shared by the query heads of a kv-head group; the
group score is the largest per-head bound, so the bound still holds for
every query head of the group.

Quantised keys (the same page, 与量化、GQA、多页并行的兼容性: the min/max
metadata can be taken from the quantised KV directly): for int8 codes with a
per-token fp16 scale, m and M are the min and max of the dequantised keys
code * scale (exact in fp32), stored in a 16-bit type rounded outward (m
down, M up), so that the stored interval still contains every key and the
bound stays an upper bound (page_minmax_dequant).
"""

from __future__ import annotations

import numpy as np


def page_token_range(p: int, page_size: int, seq_len: int) -> tuple[int, int]:
    """Logical token range [t0, t1) of page p that holds valid tokens."""
    t0 = p * page_size
    return t0, min(t0 + page_size, seq_len)


def num_pages(seq_len: int, page_size: int) -> int:
    return -(-seq_len // page_size)


def page_minmax(k_pool, page_table, seq_lens, page_size):
    """Per-channel min m and max M of K over the valid tokens of each page.

    k_pool: [P_phys][Hkv][S][d] (any real dtype; values are exact in fp64).
    Returns an fp64 array [P_phys][Hkv][2][d] (index 0 = m, 1 = M) with NaN
    in pages that no sequence uses.
    """
    k_pool = np.asarray(k_pool)
    P_phys, Hkv, S, d = k_pool.shape
    out = np.full((P_phys, Hkv, 2, d), np.nan)
    for b, L in enumerate(seq_lens):
        for p in range(num_pages(int(L), page_size)):
            phys = int(page_table[b][p])
            t0, t1 = page_token_range(p, page_size, int(L))
            keys = k_pool[phys, :, : t1 - t0, :].astype(np.float64)  # [Hkv][n][d]
            out[phys, :, 0, :] = keys.min(axis=1)
            out[phys, :, 1, :] = keys.max(axis=1)
    return out


def minmax_append(meta_page, k_new, slot):
    """Incremental update of one page's (m, M) on inserting key k_new.

    meta_page: fp64 [2][d] (m, M); slot: the token's index inside its page.
    The first token of a page starts the page's statistics.
    """
    k_new = np.asarray(k_new, dtype=np.float64)
    if slot == 0:
        return np.stack([k_new.copy(), k_new.copy()])
    return np.stack([np.minimum(meta_page[0], k_new), np.maximum(meta_page[1], k_new)])


def head_bound(q_head, m, M):
    """sum_i max(q_i m_i, q_i M_i) for one query head over pages.

    q_head: [d]; m, M: [P][d].  Returns [P] fp64.
    """
    q = np.asarray(q_head, dtype=np.float64)[None, :]
    return np.sum(np.maximum(q * m, q * M), axis=-1)


def group_scores(q_group, m, M):
    """Page score for a kv-head group: the largest per-head bound.

    q_group: [G][d] query rows of the group; m, M: [P][d].  Returns [P].
    """
    per_head = np.stack([head_bound(qh, m, M) for qh in np.asarray(q_group, dtype=np.float64)])
    return per_head.max(axis=0)


def round_outward(x, dtype: str, down: bool):
    """x (values exact in fp32) rounded toward -inf (down) or +inf (up) to
    the 16-bit type dtype ("f16" or "bf16"), returned as fp64."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        y = x.astype(np.float16)  # round to nearest
        if down:
            y = np.where(y.astype(np.float32) > x, np.nextafter(y, np.float16(-np.inf)), y)
        else:
            y = np.where(y.astype(np.float32) < x, np.nextafter(y, np.float16(np.inf)), y)
        return y.astype(np.float64)
    # bf16: the upper half of the fp32 bit pattern; cutting the low half
    # rounds toward zero, one step of the kept half away from zero fixes the
    # other direction
    u = x.view(np.uint32)
    t = u & np.uint32(0xFFFF0000)
    v = t.view(np.float32)
    bump = (v > x) if down else (v < x)
    t = np.where(bump, t + np.uint32(0x10000), t)
    return t.view(np.float32).astype(np.float64)


def page_minmax_dequant(codes, scales, page_table, seq_lens, page_size, meta_dtype):
    """Quest metadata of int8 keys with per-token scales, as stored.

    codes: [P_phys][Hkv][S][d] int8; scales: [P_phys][Hkv][S] fp16.
    Returns fp64 [P_phys][Hkv][2][d] (m rounded down, M rounded up to
    meta_dtype), NaN in unused pages.
    """
    deq = np.asarray(codes).astype(np.float64) * np.asarray(scales).astype(np.float64)[..., None]
    exact = page_minmax(deq, page_table, seq_lens, page_size)
    out = exact.copy()
    used = ~np.isnan(exact[:, :, 0, 0])
    out[used, 0] = round_outward(exact[used, 0], meta_dtype, down=True)
    out[used, 1] = round_outward(exact[used, 1], meta_dtype, down=False)
    return out
