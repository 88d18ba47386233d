"""A bounded wait that runs out, on the GPU, without a fault.

The one-shot test hook makes the split-K attention kernel's first CTA issue
no copy for its first ring stage and never complete it, so nothing is in
flight when the consumer's wait gives up (after at most 100 ms): the launch
must finish, report SPG_DEVERR_TIMEOUT in the workspace error word, and
leave the context usable: with the workspace zeroed again the same call
gives the same result as before the hook.
"""

import time

import pytest
import torch

from synth import get_workload, make_inputs, scaled

pytestmark = pytest.mark.gpu


def test_withheld_stage_times_out_and_is_reported():
    import query_aware_sparse_page_gb300 as spg

    # one (batch, kv-head) unit and a 10-page selection: every split CTA of
    # the attention launch has a single stage, so the withheld one is the
    # only wait that runs out
    w = scaled(get_workload("tiny-quest-gqa4-1k"))
    inp = make_inputs(w, device="cuda")
    p = spg.params_for(inp)
    b = spg.alloc_buffers(p, "cuda")
    spg.sparse_page_meta_update(p, inp.k_pool, None, inp.page_table, inp.seq_lens, 1, b.minmax,
                                None, None, None, b.ws)
    spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, b.minmax, None, None, None,
                           b.sel, b.sel_cnt, b.ws)

    def attend():
        spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table,
                                    inp.seq_lens, b.sel, b.sel_cnt, b.out, b.lse, b.ws)

    attend()
    torch.cuda.synchronize()
    assert spg.spg_read_device_error(b.ws) == 0
    ref_out, ref_lse = b.out.clone(), b.lse.clone()

    spg.spg_test_withhold_first_stage(b.ws)
    t0 = time.perf_counter()
    attend()
    err = spg.spg_read_device_error(b.ws)  # synchronises
    dt = time.perf_counter() - t0
    assert err & spg.DEVERR_TIMEOUT
    assert dt < 5.0, f"the timed-out launch took {dt:.2f} s"

    # the hook is one-shot and the context still works
    b.ws.zero_()
    attend()
    torch.cuda.synchronize()
    assert spg.spg_read_device_error(b.ws) == 0
    assert torch.equal(b.out, ref_out) and torch.equal(b.lse, ref_lse)
