"""Probe-sampled block scores (a third page selector), fp64.

Source: "Day 10·2 sparse top-k 块选择", §1 (the three signals of block
selection: the probe) and §2 (the probe loop): a block's potential attention
score is the largest dot product of the query with a few keys sampled
uniformly inside the block, n_probe of them (8 by default), so that a needle
in the middle of a block is not missed the way the block's first token
alone would miss it.  The sample starts at the block's first token and
steps by (valid tokens in the block) // n_probe, at least 1, up to the
block's last valid token; a short block is therefore sampled at every
token.  Ties between blocks go to the lower block index (the same page,
确定性红线), which the common selection rule (select.py) already applies.

Readings: the page of this library is the page's block; under GQA the
score of a (batch, kv-head) unit's page is the largest over the group's
query heads (as for Quest); the page's reserved half budget for prefill
importance needs attention statistics of a prefill pass, which a decode
step does not have, so it is not part of this selector; its recency
insurance (the last block is always kept) is the forced recent page.
"""

from __future__ import annotations

import numpy as np


def probe_positions(block: int, page_size: int, seq_len: int, n_probe: int) -> list[int]:
    """Token positions sampled in block `block` (absolute token indices)."""
    p0 = block * page_size
    p_end = min(p0 + page_size, seq_len)
    if p_end <= p0:
        return []
    n_probe = max(n_probe, 1)
    step = max((p_end - p0) // n_probe, 1)
    return list(range(p0, p_end, step))


def probe_score(q_rows, keys, positions, p0: int) -> float:
    """max over the group's query rows and the sampled tokens of q . k (fp64).

    q_rows: [G][d]; keys: the block's [S][d] keys (token t at keys[t - p0])."""
    q = np.asarray(q_rows, dtype=np.float64)
    best = -np.inf
    for t in positions:
        k = np.asarray(keys[t - p0], dtype=np.float64)
        best = max(best, float(np.max(q @ k)))
    return best
