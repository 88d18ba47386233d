"""The GPU parity checker has teeth: host-only checks of gpu_helpers.check_unit.

Buffers laid out as the library writes them are filled from the oracle
itself, on the CPU, for the Quest, sketch and probe selectors; check_unit
must accept them, and must reject each of a set of planted mistakes (a
lower-scoring page swapped into the selection, an output element moved by
more than the tolerance, a score off by more than the relative bar, a
non-(-1) pad entry, an lse off, a top-p count that the oracle's cumulative
mass does not allow).  No GPU is involved.
"""

import types

import numpy as np
import pytest
import torch

from oracle import decode, select
from synth import get_workload, make_inputs, scaled

from conftest import oracle_params
from gpu_helpers import TOL_OUT, check_unit, unit_inputs


def _fake_buffers(inp, prm):
    """What a correct GPU step leaves behind, computed by the oracle."""
    w = inp.workload
    B, Hkv, G, d, S = w.batch, w.num_kv_heads, w.group, w.head_dim, w.page_size
    MP = inp.page_table.shape[1]
    bufs = types.SimpleNamespace(
        scores=torch.full((B, Hkv, MP), -float("inf")),
        sel=torch.full((B, Hkv, w.n_sel_pages), -1, dtype=torch.int32),
        sel_cnt=torch.zeros((B, Hkv), dtype=torch.int32),
        out=torch.zeros((B, w.num_q_heads, d)),
        lse=torch.zeros((B, w.num_q_heads)))
    scores = {}
    for b in range(B):
        L = int(inp.seq_lens[b])
        P = -(-L // S)
        for h in range(Hkv):
            sub = unit_inputs(inp, b, h)
            sc = decode.unit_scores(sub, prm, 0, 0)
            scores[(b, h)] = sc
            lo = min(prm.n_sink, P)
            hi = max(P - prm.n_recent, lo)
            bufs.scores[b, h, lo:hi] = torch.from_numpy(np.asarray(sc[lo:hi], dtype=np.float64)).float()
            sel = decode.unit_selection(sub, prm, 0, 0, scores=sc)
            bufs.sel[b, h, :len(sel)] = torch.tensor(sel, dtype=torch.int32)
            bufs.sel_cnt[b, h] = len(sel)
            out, lse = decode.attend_selection(sub, prm, 0, 0, sel)
            bufs.out[b, h * G:(h + 1) * G] = torch.from_numpy(out).float()
            bufs.lse[b, h * G:(h + 1) * G] = torch.from_numpy(lse).float()
    return bufs, scores


def _case_inputs(selector):
    if selector == "sketch":
        w = scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=4, num_kv_heads=2,
                   seq_len=64 * 20, n_sel_pages=6)
        lens = [64 * 20, 64 * 3 + 5]  # 4 blocks: two pad entries
    else:
        w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=2, num_q_heads=4, num_kv_heads=2,
                   head_dim=64, seq_len=1200, seq_range=None, n_sel_pages=12, needles_per_head=2,
                   random_page_table=True, selector=selector)
        lens = [1200, 150]  # 10 pages: two pad entries
    return w, make_inputs(w, device="cpu", seq_lens=lens)


def _params(w, top_p=0.0):
    prm = oracle_params(w)
    if w.selector == "probe":
        prm.n_probe = 8
    prm.top_p = top_p
    return prm


@pytest.fixture(scope="module", params=["quest", "sketch", "probe"])
def case(request):
    w, inp = _case_inputs(request.param)
    prm = _params(w)
    bufs, scores = _fake_buffers(inp, prm)
    return w, inp, prm, bufs, scores


def _check_all(w, inp, prm, bufs):
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])


def _copy(bufs):
    return types.SimpleNamespace(**{k: v.clone() for k, v in vars(bufs).items()})


def test_oracle_filled_buffers_pass(case):
    w, inp, prm, bufs, _ = case
    _check_all(w, inp, prm, bufs)


def test_lower_scoring_page_swapped_in_is_caught(case):
    w, inp, prm, bufs, scores = case
    bad = _copy(bufs)
    b, h = 0, 1
    S = w.page_size
    P = -(-int(inp.seq_lens[b]) // S)
    cnt = int(bad.sel_cnt[b, h])
    sel = bad.sel[b, h, :cnt].tolist()
    forced = set(select.forced_pages(P, prm.n_sink, prm.n_recent))
    cand = [p for p in range(P) if p not in forced]
    worst = min((p for p in cand if p not in sel), key=lambda p: float(scores[(b, h)][p]))
    chosen = [p for p in sel if p not in forced]
    weakest = min(chosen, key=lambda p: float(scores[(b, h)][p]))
    new = sorted((set(sel) - {weakest}) | {worst})
    bad.sel[b, h, :cnt] = torch.tensor(new, dtype=torch.int32)
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, b, h, TOL_OUT[w.kv_dtype])


def test_output_beyond_tolerance_is_caught(case):
    w, inp, prm, bufs, _ = case
    bad = _copy(bufs)
    bad.out[1, 3, 17] += 3 * TOL_OUT[w.kv_dtype]
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, 1, 1, TOL_OUT[w.kv_dtype])


def test_score_off_by_more_than_the_bar_is_caught(case):
    w, inp, prm, bufs, _ = case
    bad = _copy(bufs)
    bad.scores[0, 0, 5] *= 1.0 + 1e-3
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, 0, 0, TOL_OUT[w.kv_dtype])


def test_pad_entries_must_be_minus_one(case):
    w, inp, prm, bufs, _ = case
    bad = _copy(bufs)
    b, h = 1, 0
    cnt = int(bad.sel_cnt[b, h])
    assert cnt < bad.sel.shape[2], "the short sequence leaves pad entries"
    bad.sel[b, h, cnt] = 0
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, b, h, TOL_OUT[w.kv_dtype])


def test_lse_off_is_caught(case):
    w, inp, prm, bufs, _ = case
    bad = _copy(bufs)
    bad.lse[0, 2] += 3 * TOL_OUT[w.kv_dtype]
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, 0, 1, TOL_OUT[w.kv_dtype])


def test_top_p_count_outside_the_mass_band_is_caught(case):
    """With top-p on, the count kept must be one the oracle's cumulative mass
    allows: keeping the whole fixed budget where p = 0.5 trims is rejected."""
    w, inp, prm0, bufs_fixed, _ = case
    prm = _params(w, top_p=0.5)
    good, _ = _fake_buffers(inp, prm)
    _check_all(w, inp, prm, good)
    trimmed = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)
               if int(good.sel_cnt[b, h]) < int(bufs_fixed.sel_cnt[b, h])]
    assert trimmed, "p = 0.5 trims at least one unit of this case"
    b, h = trimmed[0]
    bad = _copy(good)
    bad.sel[b, h] = bufs_fixed.sel[b, h]
    bad.sel_cnt[b, h] = bufs_fixed.sel_cnt[b, h]
    with pytest.raises(AssertionError):
        check_unit(inp, prm, bad, b, h, TOL_OUT[w.kv_dtype])
