"""Read-ratio and algorithmic-byte model of one decode step.

Source: "Quest 完全拆解", 三段式 kernel 与内存流水: per layer the step
reads 2ML/S bytes of metadata plus 2M*K*S bytes of the top-K pages,
against 2ML for the whole cache, i.e. a read ratio of 1/S + K/PageNum,
where M is the bytes of one K (or V) vector, L the sequence length, S the
page size and K the number of pages selected.  The same page works the
example S = 16, 64K context (4096 pages), K = 256 -> 1/16 + 1/16 = 1/8.
The KV sizes of its 背景与问题定义 section (2 * layers * L * heads * d * 2 B)
and of the SequenceO1 close reading §1 (2 * 32 * 8 * 128 * 2 B per token)
are the same product.
"""

from __future__ import annotations


def read_ratio(page_size: int, seq_len: int, k_pages: int) -> float:
    """Bytes read by the sparse step over bytes read by dense attention."""
    return 1.0 / page_size + k_pages * page_size / seq_len


def kv_cache_bytes(n_layers: int, seq_len: int, n_kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    return 2 * n_layers * seq_len * n_kv_heads * head_dim * elem_bytes


def step_bytes(seq_lens, n_kv_heads, num_q_heads, head_dim, page_size, kv_bytes,
               selector, sel_tokens, candidate_pages, sketch_dim=16, scale_bytes=0,
               q_bytes=2, sel_pages=0):
    """Algorithmic HBM bytes of one select + attend step.

    seq_lens: per-sequence lengths.  sel_tokens: total valid tokens attended,
    summed over every (batch, kv-head) unit.  candidate_pages: total pages
    scored, summed over units.  kv_bytes: bytes of one K or V element.
    scale_bytes: bytes of one per-token K (or V) scale (int8 pools), else 0.

    Counted: metadata of every scored page, K and V (and their scales) of
    every attended token, the query, the output and lse (fp32), and the
    int32 page ids written and read back (sel_pages = pages selected,
    summed over units).
    """
    B = len(seq_lens)
    if selector == "quest":
        meta = candidate_pages * 2 * head_dim * kv_bytes
    elif selector == "sketch":
        meta = candidate_pages * (page_size * sketch_dim // 2 + 4)
    else:
        meta = 0
    kv = sel_tokens * 2 * (head_dim * kv_bytes + scale_bytes)
    q = B * num_q_heads * head_dim * q_bytes
    out = B * num_q_heads * (head_dim + 1) * 4
    idx = sel_pages * 4 * 2
    return meta + kv + q + out + idx
