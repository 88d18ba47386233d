"""SALS-style low-rank int4 index key and block log-sum-exp score.

Source: "SALS长序列推理优化" (CANN learning hub), section Quant Sals Indexer
(QSI): the index query is the group-mean of the query heads (query length
1); the index key is a low-rank projection of K quantised to int4; the
score is computed in the listed order (1) query x key matrix product,
(2) dequantisation, (3) block-level log-sum-exp over every block except the
fixed tail blocks, (4) exact top-k, (5) append the tail indices.  The
formulas themselves are missing from the page's text; the reading used
here (all of it stated, none of it from the page's symbols):

  * projection P (d x d_s) is fixed, random and shared by all heads
    ("SequenceO1" close reading, Sketch Attention §3.1 / §5.3);
  * k~_t = sum_i deq(k_t)_i P_ij, computed in fp32, one product and one
    add per step, i = 0..d-1 in order, no fused multiply-add;
  * per (block, kv-head): scale sk = max|k~| / 7 (1 when the block is all
    zero) and codes clip(rint(k~ / sk), -7, 7), round half to even, fp32;
  * index query: qbar = (sum_g q_g) / G, q~ = P^T qbar (same fp32 rule),
    sq = max|q~| / 127 (1 if zero), qc = clip(rint(q~ / sq), -127, 127);
  * dot_t = sum_j qc_j * kc_tj, an exact integer;
  * z_t = dot_t * sq * sk / sqrt(d)   (fp64 here);
  * s_b = max_t z_t + ln sum_t exp(z_t - max z) over the block's tokens.

The int4/int8 codes are defined by the fp32 arithmetic above so that any
implementation following the same steps reproduces them bit for bit;
``project_fp64`` gives the exact projection for checking that the fp32
codes differ from exact rounding only next to a rounding boundary.
"""

from __future__ import annotations

import math

import numpy as np

F32 = np.float32


def dequant(codes, scales):
    """int8 codes [.., d] times their per-token fp16 scale [..] -> fp32 (exact)."""
    return np.asarray(codes).astype(F32) * np.asarray(scales).astype(F32)[..., None]


def project_fp32(x, proj):
    """x [T][d] fp32 times P [d][d_s] fp32, sequential over d, unfused, fp32."""
    x = np.asarray(x, dtype=F32)
    proj = np.asarray(proj, dtype=F32)
    acc = np.zeros((x.shape[0], proj.shape[1]), dtype=F32)
    for i in range(x.shape[1]):
        prod = x[:, i : i + 1] * proj[i : i + 1, :]  # fp32 product, rounded
        acc = acc + prod  # fp32 add, rounded
    return acc


def project_fp64(x, proj):
    return np.asarray(x, dtype=np.float64) @ np.asarray(proj, dtype=np.float64)


def quantise_block_int4(sk_rows):
    """Codes in [-7, 7] and one fp32 scale for a block's projected keys."""
    v = np.asarray(sk_rows, dtype=F32)
    amax = F32(np.max(np.abs(v))) if v.size else F32(0)
    scale = amax / F32(7.0) if amax > 0 else F32(1.0)
    codes = np.clip(np.rint(v / scale), -7, 7).astype(np.int8)
    return codes, F32(scale)


def index_query(q_group, proj):
    """Group-mean index query, projected and quantised to int8.

    q_group: [G][d] query rows (fp16/bf16 values).  Returns (qc int8 [d_s], sq fp32).
    """
    qg = np.asarray(q_group, dtype=F32)
    s = qg[0].copy()
    for g in range(1, qg.shape[0]):
        s = s + qg[g]
    qbar = s / F32(qg.shape[0])
    qt = project_fp32(qbar[None, :], proj)[0]
    amax = F32(np.max(np.abs(qt)))
    sq = amax / F32(127.0) if amax > 0 else F32(1.0)
    qc = np.clip(np.rint(qt / sq), -127, 127).astype(np.int8)
    return qc, F32(sq)


def int_dots(qc, codes):
    """Exact integer dot of the index query codes with each token's codes."""
    return np.asarray(codes, dtype=np.int64) @ np.asarray(qc, dtype=np.int64)


def block_lse(z):
    """log sum_t exp(z_t), written as max + log of the shifted sum (fp64)."""
    z = np.asarray(z, dtype=np.float64)
    mx = np.max(z)
    return float(mx + math.log(np.sum(np.exp(z - mx))))


def block_scores(qc, sq, codes_blocks, scales, head_dim):
    """Per-block LSE score of the dequantised integer logits.

    codes_blocks: [n_blocks][S][d_s] int codes, scales: [n_blocks] fp32.
    """
    inv = 1.0 / math.sqrt(head_dim)
    out = np.empty(len(codes_blocks))
    for i, (codes, sk) in enumerate(zip(codes_blocks, scales)):
        dots = int_dots(qc, codes)
        z = dots.astype(np.float64) * float(sq) * float(sk) * inv
        out[i] = block_lse(z)
    return out


def build_sketch(k_block_deq, proj):
    """Projected, quantised index key of one full block: (codes [S][d_s], scale)."""
    return quantise_block_int4(project_fp32(k_block_deq, proj))


def pack_int4(codes):
    """Pack codes [.., 2n] into bytes [.., n]: even index in the low nibble."""
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed):
    """Inverse of pack_int4 (two's-complement nibbles)."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out
