"""Pins for the Quest part of the oracle: metadata and the page bound.

What fixes the answer (Quest 完全拆解, 核心机制): the bound sum_i max(q_i m_i,
q_i M_i) is the largest q.k over the box [m, M] of the page, so it is at
least q.k for every token of the page, equals q.k when the page holds one
distinct key, and equals the maximum of q.x over the box's corners
(a linear function on a box peaks at a vertex).
"""

import itertools

import numpy as np
import pytest

from oracle import quest


def _rand_pages(rng, P, S, d, G=1, scale_chan=True):
    c = np.exp(0.5 * rng.standard_normal(d)) if scale_chan else np.ones(d)
    keys = rng.standard_normal((P, S, d)) * c
    q = rng.standard_normal((G, d))
    return q, keys


def test_bound_is_at_least_every_token_dot(rng):
    for trial in range(20):
        P, S, d, G = 7, int(rng.integers(1, 17)), 8 * int(rng.integers(1, 5)), int(rng.integers(1, 5))
        q, keys = _rand_pages(rng, P, S, d, G)
        m, M = keys.min(axis=1), keys.max(axis=1)
        s = quest.group_scores(q, m, M)
        for p in range(P):
            best = max(float(sum(q[g][i] * keys[p][t][i] for i in range(d))) for g in range(G) for t in range(S))
            assert s[p] >= best - 1e-9 * max(1.0, abs(best))


def test_bound_equals_box_corner_maximum(rng):
    for trial in range(30):
        d = int(rng.integers(1, 9))
        q = rng.standard_normal(d)
        lo = rng.standard_normal(d)
        hi = lo + np.abs(rng.standard_normal(d))
        corners = itertools.product(*[(lo[i], hi[i]) for i in range(d)])
        brute = max(sum(q[i] * c[i] for i in range(d)) for c in corners)
        s = quest.head_bound(q, lo[None], hi[None])[0]
        assert s == pytest.approx(brute, rel=1e-12, abs=1e-12)


def test_bound_tight_for_single_distinct_key(rng):
    d = 32
    for S in (1, 4, 16):
        k = rng.standard_normal(d)
        keys = np.repeat(k[None], S, axis=0)
        q = rng.standard_normal((3, d))
        s = quest.group_scores(q, keys.min(0)[None], keys.max(0)[None])[0]
        assert s == pytest.approx(max(float(q[g] @ k) for g in range(3)), rel=1e-12)


def test_group_score_is_max_over_heads(rng):
    q, keys = _rand_pages(rng, 5, 16, 16, G=4)
    m, M = keys.min(axis=1), keys.max(axis=1)
    per = [quest.head_bound(q[g], m, M) for g in range(4)]
    s = quest.group_scores(q, m, M)
    for p in range(5):
        assert s[p] == max(per[g][p] for g in range(4))


def test_page_minmax_brute_force(rng):
    S, Hkv, d = 4, 2, 3
    lens = [9, 4, 1]
    pages = [-(-L // S) for L in lens]
    n_phys = sum(pages) + 2  # two unused pages
    pool = rng.standard_normal((n_phys, Hkv, S, d)).astype(np.float16)
    perm = rng.permutation(n_phys)
    pt = np.full((3, 3), -1)
    off = 0
    for b in range(3):
        pt[b, : pages[b]] = perm[off : off + pages[b]]
        off += pages[b]
    mm = quest.page_minmax(pool, pt, lens, S)
    used = set()
    for b, L in enumerate(lens):
        for p in range(pages[b]):
            phys = int(pt[b, p])
            used.add(phys)
            n_valid = min(S, L - p * S)
            for h in range(Hkv):
                for i in range(d):
                    vals = [float(pool[phys, h, t, i]) for t in range(n_valid)]
                    assert mm[phys, h, 0, i] == min(vals)
                    assert mm[phys, h, 1, i] == max(vals)
    for phys in set(range(n_phys)) - used:
        assert np.isnan(mm[phys]).all()


def test_incremental_append_matches_page_statistics(rng):
    S, d = 16, 8
    keys = rng.standard_normal((37, d))
    meta = None
    for t, k in enumerate(keys):
        slot = t % S
        meta = quest.minmax_append(meta, k, slot)
        p0 = t - slot
        page = keys[p0 : t + 1]
        assert (meta[0] == page.min(axis=0)).all() and (meta[1] == page.max(axis=0)).all()


def test_planted_mistake_is_caught(rng, monkeypatch):
    """A bound that swaps m and M must fail the box-corner pin."""

    def swapped(q_head, m, M):
        q = np.asarray(q_head, dtype=np.float64)[None, :]
        return np.sum(np.maximum(q * M, q * m) * 0 + np.minimum(q * m, q * M), axis=-1)

    monkeypatch.setattr(quest, "head_bound", swapped)
    with pytest.raises(AssertionError):
        test_bound_equals_box_corner_maximum(rng)
