"""sparse_decode_attention_noalloc, the entry point for callers that cannot
allocate device memory (framework plugins given no allocator or workspace,
serving loops that forbid cudaMalloc after start-up).

It runs the same split-K attention kernel, with the same split count, as
sparse_decode_attention (the workspace entry point); only where the split
partials live differs, so the two results must be bitwise equal.  Checked on
three calls in a row: two different problems, then the first again, so that
whatever an earlier call left in the shared scratch array cannot leak into a
later one.  This file is collected last.
"""

import ctypes

import pytest
import torch

from synth import get_workload, make_inputs, scaled

pytestmark = pytest.mark.gpu


def _noalloc(spg):
    f = spg.LIB.sparse_decode_attention_noalloc
    f.argtypes = [ctypes.POINTER(spg.spg_params)] + [ctypes.c_void_p] * 12
    f.restype = ctypes.c_int32
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _problem(spg, w):
    inp = make_inputs(w, device="cuda")
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, "cuda")
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                           bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt, bufs.ws)
    spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                inp.page_table, inp.seq_lens, bufs.sel, bufs.sel_cnt, bufs.out,
                                bufs.lse, bufs.ws)
    return inp, p, bufs


def test_noalloc_matches_workspace_entry_point_call_after_call():
    import query_aware_sparse_page_gb300 as spg

    f = _noalloc(spg)
    problems = [
        scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8, num_kv_heads=2,
               seq_range=(100, 3000), n_sel_pages=24),
        scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
               seq_len=64 * 30 + 17, n_sel_pages=9),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    made = [_problem(spg, w) for w in problems]
    for inp, p, bufs in made + made[:1]:
        out = torch.full_like(bufs.out, float("nan"))
        lse = torch.full_like(bufs.lse, float("nan"))
        status = f(ctypes.byref(p), _ptr(inp.q), _ptr(inp.k_pool), _ptr(inp.v_pool),
                   _ptr(inp.k_scale), _ptr(inp.v_scale), _ptr(inp.page_table), _ptr(inp.seq_lens),
                   _ptr(bufs.sel), _ptr(bufs.sel_cnt), _ptr(out), _ptr(lse),
                   ctypes.c_void_p(stream))
        assert status == 0, spg.status_str(status)
        torch.cuda.synchronize()
        assert torch.equal(out, bufs.out), f"out differs by {(out - bufs.out).abs().max().item():.3e}"
        assert torch.equal(lse, bufs.lse), f"lse differs by {(lse - bufs.lse).abs().max().item():.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    import query_aware_sparse_page_gb300 as spg

    f = _noalloc(spg)
    # 32 x 16 = 512 (batch x q-head) rows at head_dim 128: more than the array holds
    p = spg.make_params(batch=32, num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16,
                        num_phys_pages=64, max_pages_per_seq=64, kv_dtype="f16",
                        selector="quest", token_budget=128, n_sink_pages=1, n_recent_pages=1)
    t = torch.zeros(1024, dtype=torch.float32, device="cuda")
    status = f(ctypes.byref(p), *([_ptr(t)] * 11), ctypes.c_void_p(0))
    assert status == spg.binding.SPG_EWORKSPACE
