"""The probe selector (Day 10·2 sparse top-k, §1-§2) on the GPU against the oracle.

A page's score is the largest q . k over its sampled tokens (and over the
group's query rows); scores within 1e-5 relative, page ids exact outside the
tie band, attention on the GPU's selection within 2e-3.  The probe selector
keeps no metadata: every entry point takes the K pool where the others take
their metadata.
"""

import numpy as np
import pytest
import torch

from synth import get_workload, make_inputs, scaled

from conftest import oracle_params
from gpu_helpers import TOL_OUT, check_unit

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = {
    "probe-mha-s32": scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=4,
                            page_size=32, seq_len=32 * 130 + 9, n_sel_pages=16, needles_per_head=4,
                            selector="probe"),
    "probe-gqa-ragged": scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=16,
                               num_kv_heads=4, seq_range=(100, 3000), n_sel_pages=24, selector="probe"),
    "probe-d64-g8": scaled(get_workload("long-scan-b4-128k"), batch=2, num_q_heads=16, num_kv_heads=2,
                           head_dim=64, page_size=32, seq_len=32 * 90 + 31, n_sel_pages=12,
                           needles_per_head=4, selector="probe"),
}


@pytest.mark.parametrize("n_probe", [0, 3, 64])
@pytest.mark.parametrize("entry", ["select_attend", "step", "separate"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_probe_selector_matches_oracle(name, entry, n_probe):
    import query_aware_sparse_page_gb300 as spg

    w = CASES[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    p.n_probe = n_probe
    bufs = spg.alloc_buffers(p, DEV)
    assert bufs.minmax is None
    pool = inp.k_pool  # the probe selector's "metadata"
    assert spg.step_kernel_name(p) == "k_probe_select+k_attn"
    assert spg.step_launch_count(p) == 2
    spg.sparse_page_meta_update(p, inp.k_pool, None, inp.page_table, inp.seq_lens, 1, pool, None,
                                None, None, bufs.ws)  # nothing to keep: a no-op
    spg.sparse_page_score(p, inp.q, inp.page_table, inp.seq_lens, pool, None, None, None,
                          bufs.scores, bufs.ws)
    if entry == "separate":
        spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, pool, None, None, None,
                               bufs.sel, bufs.sel_cnt, bufs.ws)
        spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table,
                                    inp.seq_lens, bufs.sel, bufs.sel_cnt, bufs.out, bufs.lse, bufs.ws)
    else:
        f = spg.sparse_decode_step if entry == "step" else spg.sparse_decode_select_attend
        f(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table, inp.seq_lens, pool, None,
          None, None, bufs.sel, bufs.sel_cnt, bufs.out, bufs.lse, bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0
    torch.cuda.synchronize()
    prm = oracle_params(w)
    prm.n_probe = n_probe if n_probe > 0 else 8
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])
