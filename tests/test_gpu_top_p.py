"""The adaptive (top-p) page budget on the GPU against the oracle.

SequenceO1 close reading §3.2 / §4.2: of the candidates, in (score desc,
page asc) order, the smallest prefix whose softmax mass reaches p is kept
(at least min_pages, at most the fixed budget).  The GPU sums fp32 weights
where the oracle sums fp64 ones, so the count may differ from the oracle's
only where the oracle's cumulative mass lies within 1e-4 of p; the chosen
pages must then be the best candidates for that count (with the score tie
band of the fixed-budget tests), and the attention output must match the
oracle's on the GPU's own selection.  Every path: the cluster kernel, the
scheduled kernel and the separate select + attend launches.
"""

import math

import numpy as np
import pytest
import torch

from oracle import decode, select as oselect
from synth import get_workload, make_inputs, scaled

from conftest import oracle_params
from gpu_helpers import (TOL_OUT, allowed_top_p_counts, assert_selection_matches, gpu_selection,
                         unit_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = {
    "quest-mha": scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=4,
                        seq_len=4096 + 9, n_sel_pages=64, needles_per_head=4),
    "quest-gqa-ragged": scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8,
                               num_kv_heads=2, seq_range=(100, 3000), n_sel_pages=48),
    "sketch": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                     seq_len=64 * 30 + 17, n_sel_pages=20),
    # Quest over an int8 pool: metadata in the query's type, tau the softmax
    # scale; needles make a few pages hold most of the mass (without them
    # the bounds are flat and p = 0.5 needs more pages than the budget)
    "quest-i8": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                       page_size=16, seq_len=16 * 150 + 5, selector="quest", n_sel_pages=24,
                       n_sink=1, n_recent=1, needles_per_head=4),
}


def _run(w, path, top_p, min_pages):
    import query_aware_sparse_page_gb300 as spg

    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    p.top_p = top_p
    p.min_pages = min_pages
    bufs = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    try:
        if path == "separate":
            spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                                   bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt, bufs.ws)
            spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                        inp.page_table, inp.seq_lens, bufs.sel, bufs.sel_cnt,
                                        bufs.out, bufs.lse, bufs.ws)
        else:
            spg.spg_set_step_kernel(spg.STEP_KERNEL_CLUSTER if path == "cluster" else spg.STEP_KERNEL_SCHED)
            spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                            inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                                            bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt,
                                            bufs.out, bufs.lse, bufs.ws)
    finally:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)
    assert spg.spg_read_device_error(bufs.ws) == 0
    torch.cuda.synchronize()
    return inp, p, bufs


@pytest.mark.parametrize("path", ["cluster", "sched", "separate"])
@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("top_p,min_pages", [(0.5, 0), (0.9, 3), (0.99, 1)])
def test_adaptive_budget_matches_oracle(name, path, top_p, min_pages):
    w = CASES[name]
    inp, p, bufs = _run(w, path, top_p, min_pages)
    prm = oracle_params(w)
    prm.top_p, prm.min_pages = top_p, min_pages
    G = w.group
    trimmed = 0
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            sub = unit_inputs(inp, b, h)
            L = int(inp.seq_lens[b])
            P = -(-L // w.page_size)
            gsel = gpu_selection(bufs, b, h)
            scores = decode.unit_scores(sub, prm, 0, 0)
            forced = oselect.forced_pages(P, w.n_sink, w.n_recent)
            cand = [q for q in range(P) if q not in set(forced)]
            k_budget = min(max(w.n_sel_pages - len(forced), 0), len(cand))
            k_gpu = len(gsel) - len(forced)
            if k_budget > 0:
                ranked = sorted(cand, key=lambda q: (-float(scores[q]), q))
                ok = allowed_top_p_counts(scores, ranked, k_budget, top_p, min_pages, prm.tau)
                assert k_gpu in ok, f"unit {(b, h)}: kept {k_gpu}, allowed {sorted(ok)}"
                trimmed += k_gpu < k_budget
                # the kept pages are the best k_gpu candidates (tie band as the fixed budget)
                assert_selection_matches(gsel, scores, P, len(forced) + k_gpu, w.n_sink, w.n_recent)
            out, lse = decode.attend_selection(sub, prm, 0, 0, gsel)
            gout = bufs.out[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
            glse = bufs.lse[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
            assert np.abs(gout - out).max() <= TOL_OUT[w.kv_dtype]
            if L > 0:
                assert np.abs(glse - lse).max() <= TOL_OUT[w.kv_dtype]
    if top_p <= 0.5:
        assert trimmed > 0, "the adaptive budget kept the whole fixed budget everywhere"


def test_top_p_one_keeps_the_fixed_budget():
    """p = 1 keeps every candidate the budget allows: the fixed-budget selection."""
    import query_aware_sparse_page_gb300 as spg

    w = CASES["quest-mha"]
    inp, p, bufs = _run(w, "cluster", 1.0, 0)
    _, p0, ref = _run(w, "cluster", 0.0, 0)
    assert torch.equal(bufs.sel, ref.sel) and torch.equal(bufs.sel_cnt, ref.sel_cnt)
