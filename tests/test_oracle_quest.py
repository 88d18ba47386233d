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


# ---- Quest over int8 keys (与量化、GQA、多页并行的兼容性) ---------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_round_outward_brackets_within_one_step(rng, dtype):
    import torch

    x = (rng.standard_normal(4000) * rng.choice([0.01, 1.0, 300.0], 4000)).astype(np.float32)
    lo = quest.round_outward(x, dtype, down=True)
    hi = quest.round_outward(x, dtype, down=False)
    assert np.all(lo <= x) and np.all(hi >= x)
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    # both ends are values of the 16-bit type, next to each other (or equal when x is one)
    for v in (lo, hi):
        back = torch.tensor(v, dtype=torch.float64).to(tdt).to(torch.float64).numpy()
        assert np.array_equal(back, v)
    exact = torch.tensor(x).to(tdt).to(torch.float32).numpy() == x
    assert np.all((lo == hi) == exact)
    nxt = torch.nextafter(torch.tensor(lo, dtype=torch.float32).to(tdt) if dtype == "f16" else
                          torch.tensor(lo, dtype=torch.float32).to(tdt),
                          torch.full(x.shape, float("inf")).to(tdt))
    assert np.all((hi == lo) | (hi == nxt.to(torch.float64).numpy()))


def test_dequant_metadata_bounds_every_dequantised_key(rng):
    """The bound over int8 keys with per-token scales stays an upper bound of
    q . k for every token of every page (the Quest invariant), and the stored
    interval is at most one step of the stored type wider than the exact one."""
    P_phys, Hkv, S, d = 9, 2, 16, 32
    codes = rng.integers(-127, 128, (P_phys, Hkv, S, d)).astype(np.int8)
    scales = (rng.random((P_phys, Hkv, S)) * 0.05 + 0.001).astype(np.float16)
    pt = np.array([[3, 1, 4, 0, 8, 2, 7, 5, 6]])
    L = 8 * S + 5
    for meta in ("f16", "bf16"):
        mm = quest.page_minmax_dequant(codes, scales, pt, [L], S, meta)
        deq = codes.astype(np.float64) * scales.astype(np.float64)[..., None]
        exact = quest.page_minmax(deq, pt, [L], S)
        used = ~np.isnan(exact[:, 0, 0, 0])
        assert np.all(mm[used, :, 0] <= exact[used, :, 0]) and np.all(mm[used, :, 1] >= exact[used, :, 1])
        q = rng.standard_normal((2, d))
        for p in range(9):
            phys = pt[0, p]
            n = min(S, L - p * S)
            for h in range(Hkv):
                bound = quest.group_scores(q, mm[phys, h, 0][None], mm[phys, h, 1][None])[0]
                assert bound >= (q @ deq[phys, h, :n].T).max() - 1e-12


def test_dequant_metadata_is_exact_when_representable():
    # unit scales and small codes: every key is a 16-bit value, nothing rounds
    codes = np.arange(-8, 8, dtype=np.int8).reshape(1, 1, 2, 8)
    scales = np.ones((1, 1, 2), np.float16)
    mm = quest.page_minmax_dequant(codes, scales, np.array([[0]]), [2], 2, "f16")
    assert np.array_equal(mm[0, 0, 0], np.minimum(codes[0, 0, 0], codes[0, 0, 1]).astype(np.float64))
    assert np.array_equal(mm[0, 0, 1], np.maximum(codes[0, 0, 0], codes[0, 0, 1]).astype(np.float64))
