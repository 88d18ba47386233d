"""Pins for the probe selector of the oracle (Day 10·2 sparse top-k, §1-§2).

What fixes the answer: the sampled positions follow the page's loop (start
at the block's first token, step (valid tokens) // n_probe, at least 1), so
a full 32-token block with 8 probes is sampled every 4 tokens and a short
block at every token; with at least as many probes as tokens the score is
the exact maximum of q . k over the block (brute force), which never exceeds
the Quest upper bound of the same page; a needle on a sampled token puts its
page on top.
"""

import numpy as np
import pytest

from oracle import decode, probe, quest, select
from synth import get_workload, make_inputs, scaled

from conftest import oracle_inputs


def test_probe_positions_closed_forms():
    assert probe.probe_positions(0, 32, 1000, 8) == [0, 4, 8, 12, 16, 20, 24, 28]
    assert probe.probe_positions(3, 32, 1000, 8) == [96 + 4 * j for j in range(8)]
    assert probe.probe_positions(3, 32, 96 + 5, 8) == [96, 97, 98, 99, 100]  # short: every token
    assert probe.probe_positions(3, 32, 96 + 20, 8) == [96 + 2 * j for j in range(10)]
    assert probe.probe_positions(1, 16, 1000, 8) == [16 + 2 * j for j in range(8)]
    assert probe.probe_positions(1, 16, 1000, 1) == [16]
    assert probe.probe_positions(1, 16, 1000, 0) == [16]  # n_probe < 1 counts as 1
    assert probe.probe_positions(2, 16, 1000, 64) == list(range(32, 48))
    assert probe.probe_positions(5, 16, 80, 8) == []  # past the end


def test_probe_with_every_token_is_the_block_max_and_below_the_bound(rng):
    for trial in range(20):
        d, S, G = 16, 16, int(rng.choice([1, 2, 4]))
        P = int(rng.integers(2, 9))
        L = (P - 1) * S + int(rng.integers(1, S + 1))
        k = rng.standard_normal((P, 1, S, d))
        q = rng.standard_normal((1, G, d))
        inp = decode.StepInputs(q, k, k, None, None, np.arange(P)[None, :], np.array([L]))
        prm_all = decode.StepParams(S, P, 0, 0, "probe", d, n_probe=S)
        got = decode.unit_scores(inp, prm_all, 0, 0)
        qb = quest.group_scores(q[0].astype(np.float64), *_minmax(k, L, S))
        for p in range(P):
            n = min(S, L - p * S)
            brute = max(float(q[0, g] @ k[p, 0, t]) for g in range(G) for t in range(n))
            assert got[p] == pytest.approx(brute, rel=1e-12)
            assert got[p] <= qb[p] + 1e-9
        # fewer probes: a subset of the tokens, so never above the full max
        part = decode.unit_scores(inp, decode.StepParams(S, P, 0, 0, "probe", d, n_probe=3), 0, 0)
        assert np.all(part <= got + 1e-12)


def _minmax(k, L, S):
    P = k.shape[0]
    m = np.empty((P, k.shape[-1]))
    M = np.empty_like(m)
    for p in range(P):
        n = min(S, L - p * S)
        m[p] = k[p, 0, :n].min(axis=0)
        M[p] = k[p, 0, :n].max(axis=0)
    return m, M


def test_needle_on_a_probe_is_selected(rng):
    d, S, P = 32, 32, 40
    k = rng.standard_normal((P, 1, S, d)) * 0.1
    q = rng.standard_normal((1, 1, d))
    k[23, 0, 8] = 5.0 * q[0, 0] / np.linalg.norm(q[0, 0]) * np.sqrt(d)  # token 8: a probe position
    inp = decode.StepInputs(q, k, k, None, None, np.arange(P)[None, :], np.array([P * S]))
    prm = decode.StepParams(S, 4, 1, 1, "probe", d)
    sc = decode.unit_scores(inp, prm, 0, 0)
    assert int(np.argmax(sc[1:P - 1])) + 1 == 23
    assert 23 in decode.unit_selection(inp, prm, 0, 0)
    # the same needle between two probes (token 9) is not seen by the probes
    k2 = k.copy()
    k2[23, 0, 9] = k2[23, 0, 8]
    k2[23, 0, 8] = k[22, 0, 8]
    inp2 = decode.StepInputs(q, k2, k2, None, None, np.arange(P)[None, :], np.array([P * S]))
    assert decode.unit_scores(inp2, prm, 0, 0)[23] < sc[23]


def test_probe_step_on_a_workload_finds_needles_on_probes():
    w = scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=4, seq_len=32 * 64 + 9,
               page_size=32, n_sel_pages=12, needles_per_head=0)
    inp = make_inputs(w)
    oi = oracle_inputs(inp)
    prm = decode.StepParams(32, 12, 1, 1, "probe", w.head_dim)
    res = decode.decode_step(oi, prm)
    for (b, h), sel in res["sel"].items():
        P = -(-int(oi.seq_lens[b]) // 32)
        assert len(sel) == 12 and sel[0] == 0 and sel[-1] == P - 1
        assert sel == select.select_pages(res["scores"][(b, h)], P, 12, 1, 1)
