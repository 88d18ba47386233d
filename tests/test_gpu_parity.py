"""CUDA path vs oracle, element by element, through the C ABI.

Small cases (every unit checked, several tiles and ragged tails) for each
workload recipe, edge cases, and the full-size workloads on sampled units
in the launch configuration the benchmark times.
"""

import math

import numpy as np
import pytest
import torch

from oracle import decode, quest, select as oselect, sketch as osk
from synth import get_workload, make_inputs, scaled

from conftest import oracle_inputs, oracle_params, to_numpy
from gpu_helpers import (TOL_OUT, assert_paths_agree, check_unit, gpu_selection, run_step,
                         unit_inputs, unswizzle_meta_row)

pytestmark = pytest.mark.gpu

DEV = "cuda"

# The single-launch step has two kernels: the persistent scheduled one (the
# default where it applies) and the cluster-per-unit one.  Tests marked with
# this parameter run through each.
KERNELS = ["sched", "cluster"]


def _spg():
    import query_aware_sparse_page_gb300 as spg

    return spg


@pytest.fixture
def step_kernel(request):
    """Selects the single-launch step kernel for one test, then restores the default."""
    spg = _spg()
    name = getattr(request, "param", "sched")
    spg.spg_set_step_kernel(spg.STEP_KERNEL_SCHED if name == "sched" else spg.STEP_KERNEL_CLUSTER)
    yield name
    spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)


def _expect_kernel(p, name):
    spg = _spg()
    k = spg.step_kernel_name(p)
    assert k == ("k_sched" if name == "sched" else "k_fused"), k


SMALL = {
    "tiny": scaled(get_workload("tiny-quest-gqa4-1k")),
    "tiny-ragged": scaled(get_workload("tiny-quest-gqa4-1k"), seq_len=1000 + 7),
    "mha": scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=4, seq_len=4096 + 9,
                  n_sel_pages=32, needles_per_head=4),
    "gqa-ragged": scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8, num_kv_heads=2,
                         seq_range=(100, 3000), n_sel_pages=24),
    "sals-4x": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                      seq_len=64 * 30 + 17, n_sel_pages=9),
    "sals-6x-full-tail": scaled(get_workload("sals-int8-b16-10k-6x"), batch=2, num_q_heads=8,
                                num_kv_heads=2, seq_len=64 * 24, n_sel_pages=5),
    "long-d64-g8": scaled(get_workload("long-scan-b4-128k"), batch=2, num_q_heads=16, num_kv_heads=2,
                          head_dim=64, seq_len=16 * 700 + 3, needles_per_head=8, n_sel_pages=40),
    "gqa2-f16": scaled(get_workload("tiny-quest-gqa4-1k"), num_q_heads=4, num_kv_heads=2, head_dim=128,
                       seq_len=2000, n_sel_pages=20, n_sink=2, n_recent=3),
    # every other shape spg_validate accepts: int8 pools with a bf16 query or
    # d = 64 (the CUDA-core int8 consumer), the sketch selector over 16-bit
    # pools and at 128-token blocks, Quest at 32-, 64- and 128-token pages
    "sals-bf16q": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                         seq_len=64 * 18 + 5, n_sel_pages=6, q_dtype="bf16"),
    "sals-d64": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                       head_dim=64, seq_len=64 * 18 + 33, n_sel_pages=6),
    "sals-s128-f16": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=4, num_kv_heads=2,
                            head_dim=64, page_size=128, seq_len=128 * 12 + 100, n_sel_pages=5,
                            kv_dtype="f16", q_dtype="f16"),
    "sals-s128-i8": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                           page_size=128, seq_len=128 * 10 + 128, n_sel_pages=4),
    # the sketch selector at 16- and 32-token blocks (a warp's lanes outnumber
    # a block's tokens at 16)
    "sals-s16-f16": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                           page_size=16, seq_len=16 * 90 + 5, n_sel_pages=12, kv_dtype="f16",
                           q_dtype="f16"),
    "sals-s32-i8": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                          page_size=32, seq_len=32 * 50 + 32, n_sel_pages=8),
    "quest-s32": scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=2,
                        page_size=32, seq_len=32 * 150 + 7, n_sel_pages=20, needles_per_head=4),
    "quest-s64-bf16": scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8, num_kv_heads=2,
                             page_size=64, seq_range=(300, 5000), n_sel_pages=12),
    "quest-s128-d64": scaled(get_workload("long-scan-b4-128k"), batch=2, num_q_heads=8, num_kv_heads=2,
                             head_dim=64, page_size=128, seq_len=128 * 40 + 77, n_sel_pages=8,
                             needles_per_head=4),
    # Quest over int8 pools (metadata of the dequantised keys, rounded outward)
    "quest-i8": scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
                       page_size=16, seq_len=16 * 150 + 5, selector="quest", n_sel_pages=24,
                       n_sink=1, n_recent=1),
    "quest-i8-bf16q-d64": scaled(get_workload("sals-int8-b16-10k-4x"), batch=3, num_q_heads=8,
                                 num_kv_heads=2, head_dim=64, page_size=32, seq_len=32 * 70 + 19,
                                 selector="quest", n_sel_pages=12, n_sink=1, n_recent=2,
                                 q_dtype="bf16"),
}


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workload_every_unit(name, step_kernel):
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p, bufs, err = run_step(inp)
    _expect_kernel(p, step_kernel)
    assert err == 0
    prm = oracle_params(w)
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])


@pytest.mark.parametrize("name", ["tiny", "mha", "gqa-ragged", "sals-4x", "long-d64-g8"])
def test_separate_calls_equal_fused(name):
    """The single-launch path selects exactly the same pages as the separate
    score/select and attention launches; outputs differ only by the order of
    the split merges."""
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    _, b1, _ = run_step(inp, fused=True)
    _, b2, _ = run_step(inp, fused=False)
    assert torch.equal(b1.sel, b2.sel) and torch.equal(b1.sel_cnt, b2.sel_cnt)
    assert_paths_agree(b1.out, b2.out, b1.lse, b2.lse, w.kv_dtype, inp.v_pool.float().abs().max())


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("name", ["tiny-ragged", "gqa-ragged", "sals-4x", "sals-6x-full-tail"])
def test_decode_step_appends_then_attends(name, step_kernel):
    """sparse_decode_step = append the new token's metadata, select, attend."""
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    ref = spg.alloc_buffers(p, DEV)
    got = spg.alloc_buffers(p, DEV)
    # metadata as of one token earlier, then the step appends the last token
    prev = (inp.seq_lens - 1).clamp(min=0)
    for bufs in (ref, got):
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, prev, 1, bufs.minmax,
                                    bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 0,
                                ref.minmax, ref.sketch, ref.sketch_scale, inp.proj, ref.ws)
    spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                    inp.page_table, inp.seq_lens, ref.minmax, ref.sketch,
                                    ref.sketch_scale, inp.proj, ref.sel, ref.sel_cnt, ref.out,
                                    ref.lse, ref.ws)
    spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                           inp.page_table, inp.seq_lens, got.minmax, got.sketch, got.sketch_scale,
                           inp.proj, got.sel, got.sel_cnt, got.out, got.lse, got.ws)
    assert spg.spg_read_device_error(got.ws) == 0
    assert torch.equal(ref.sel, got.sel) and torch.equal(ref.sel_cnt, got.sel_cnt)
    assert torch.equal(ref.out, got.out) and torch.equal(ref.lse, got.lse)
    if got.minmax is not None:
        assert torch.equal(ref.minmax, got.minmax)
    else:
        assert torch.equal(ref.sketch, got.sketch) and torch.equal(ref.sketch_scale, got.sketch_scale)


def test_long_page_table_takes_the_separate_path():
    """More than 8192 pages per sequence: scoring, a separate selection kernel
    and the split-K attention launch."""
    w = scaled(get_workload("long-scan-b4-128k"), batch=1, num_q_heads=2, num_kv_heads=1,
               head_dim=64, seq_len=16 * 9000 + 5, needles_per_head=4, n_sel_pages=40)
    inp = make_inputs(w, device=DEV)
    p, bufs, err = run_step(inp)
    assert err == 0
    check_unit(inp, oracle_params(w), bufs, 0, 0, TOL_OUT[w.kv_dtype])
    assert {t // 16 for t in inp.needles[(0, 0)]} <= set(gpu_selection(bufs, 0, 0))


@pytest.mark.parametrize("name", ["tiny-ragged", "mha", "gqa-ragged", "sals-4x", "long-d64-g8"])
def test_dense_baseline(name):
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, bufs.out, bufs.lse, bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0
    oi = oracle_inputs(inp)
    prm = oracle_params(w, selector="all")
    res = decode.decode_step(oi, prm)
    G = w.group
    tol = TOL_OUT[w.kv_dtype]
    for (b, h), out in res["out"].items():
        gout = bufs.out[b, h * G : (h + 1) * G].cpu().numpy()
        glse = bufs.lse[b, h * G : (h + 1) * G].cpu().numpy()
        assert np.abs(gout - out).max() <= tol
        assert np.abs(glse - res["lse"][(b, h)]).max() <= tol


@pytest.mark.parametrize("case", ["skewed-with-empty", "all-empty", "one-unit-long"])
def test_dense_length_plan_edges(case):
    """The dense baseline's split planned by length: a unit with no pages, a
    batch with no tokens at all, and one unit whose parts hit the split
    limit (every other CTA of the wave has no work)."""
    spg = _spg()
    if case == "one-unit-long":
        w = scaled(get_workload("tiny-quest-gqa4-1k"), seq_len=16 * 300 + 5, n_sel_pages=10)
        lens = None
    else:
        w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=6, num_q_heads=8, num_kv_heads=2,
                   seq_range=(1, 2), n_sel_pages=6)
        lens = [0, 1, 16, 17, 95, 1600] if case == "skewed-with-empty" else [0] * 6
    inp = make_inputs(w, device=DEV, seq_lens=lens)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    for _ in range(2):  # the arrival counters must return to zero for the next call
        spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                   inp.page_table, inp.seq_lens, bufs.out, bufs.lse, bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0
    oi = oracle_inputs(inp)
    prm = oracle_params(w, selector="all")
    res = decode.decode_step(oi, prm)
    G = w.group
    tol = TOL_OUT[w.kv_dtype]
    for (b, h), out in res["out"].items():
        gout = bufs.out[b, h * G : (h + 1) * G].cpu().numpy()
        glse = bufs.lse[b, h * G : (h + 1) * G].cpu().numpy()
        if int(inp.seq_lens[b]) == 0:
            assert (gout == 0).all() and np.isneginf(glse).all()
            continue
        assert np.abs(gout - out).max() <= tol
        assert np.abs(glse - res["lse"][(b, h)]).max() <= tol


def test_full_budget_sparse_equals_dense():
    """Selecting every page reproduces dense attention (100% retention check)."""
    spg = _spg()
    w = scaled(get_workload("tiny-quest-gqa4-1k"), seq_len=777, n_sel_pages=64)
    inp = make_inputs(w, device=DEV)
    _, bufs, _ = run_step(inp)
    p = spg.params_for(inp)
    d = spg.alloc_buffers(p, DEV)
    spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table,
                               inp.seq_lens, d.out, d.lse, d.ws)
    assert gpu_selection(bufs, 0, 0) == list(range(49))
    assert_paths_agree(bufs.out, d.out, bufs.lse, d.lse, w.kv_dtype, inp.v_pool.float().abs().max())


@pytest.mark.parametrize("name", ["tiny-ragged", "mha", "gqa-ragged", "long-d64-g8"])
def test_minmax_rebuild_bit_exact(name):
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, None, inp.page_table, inp.seq_lens, 1, bufs.minmax,
                                None, None, None, bufs.ws)
    ref = quest.page_minmax(to_numpy(inp.k_pool), to_numpy(inp.page_table), to_numpy(inp.seq_lens),
                            w.page_size)
    got = to_numpy(bufs.minmax)  # [B][Hkv][MP][2][d], logical pages, chunk-swizzled rows
    pt = to_numpy(inp.page_table)
    n = 0
    for b, L in enumerate(to_numpy(inp.seq_lens)):
        for p_ in range(-(-int(L) // w.page_size)):
            for h in range(w.num_kv_heads):
                row = unswizzle_meta_row(got[b, h, p_], p_).astype(np.float64)
                assert np.array_equal(row, ref[pt[b, p_], h])
            n += 1
    assert n > 0


def _append_sequence(spg, inp, p, bufs, lens_final):
    """Append tokens one by one (seq_lens 1..L) through the append entry point."""
    for t in range(1, int(max(lens_final)) + 1):
        lens = torch.clamp(torch.tensor(lens_final, dtype=torch.int32), max=t).to(DEV)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, lens, 0,
                                    bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)


def test_minmax_append_equals_rebuild():
    spg = _spg()
    w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8, num_kv_heads=2,
               seq_range=(20, 90), n_sel_pages=4)
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    a = spg.alloc_buffers(p, DEV)
    r = spg.alloc_buffers(p, DEV)
    a.minmax.fill_(7.0)  # stale content from a recycled page must not leak
    _append_sequence(spg, inp, p, a, inp.seq_lens.cpu().tolist())
    spg.sparse_page_meta_update(p, inp.k_pool, None, inp.page_table, inp.seq_lens, 1, r.minmax, None,
                                None, None, r.ws)
    for b, L in enumerate(inp.seq_lens.cpu().tolist()):
        P = -(-L // w.page_size)
        assert torch.equal(a.minmax[b, :, :P], r.minmax[b, :, :P])
    assert spg.spg_read_device_error(a.ws) == 0


@pytest.mark.parametrize("name", ["sals-4x", "sals-6x-full-tail"])
def test_sketch_codes_bit_exact(name):
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1, None,
                                bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    kp, ks, pt, proj = to_numpy(inp.k_pool), to_numpy(inp.k_scale), to_numpy(inp.page_table), to_numpy(inp.proj)
    sk_gpu = bufs.sketch.cpu().numpy()
    sc_gpu = bufs.sketch_scale.cpu().numpy()
    n_checked = 0
    for b, L in enumerate(to_numpy(inp.seq_lens)):
        for blk in range(int(L) // w.page_size):
            phys = int(pt[b, blk])
            for h in range(w.num_kv_heads):
                codes, scale = osk.build_sketch(osk.dequant(kp[phys, h], ks[phys, h]), proj)
                assert np.array_equal(osk.unpack_int4(sk_gpu[b, h, blk]), codes)
                assert sc_gpu[b, h, blk] == scale
                n_checked += 1
    assert n_checked > 0


def test_sketch_append_equals_rebuild():
    spg = _spg()
    w = scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
               seq_len=64 * 3 + 5, n_sel_pages=2)
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    a = spg.alloc_buffers(p, DEV)
    r = spg.alloc_buffers(p, DEV)
    _append_sequence(spg, inp, p, a, inp.seq_lens.cpu().tolist())
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1, None,
                                r.sketch, r.sketch_scale, inp.proj, r.ws)
    assert torch.equal(a.sketch, r.sketch) and torch.equal(a.sketch_scale, r.sketch_scale)


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
def test_edge_sequences(step_kernel):
    """Empty, one-token, page-aligned, and shorter-than-budget sequences."""
    w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=6, num_q_heads=8, num_kv_heads=2,
               seq_range=(1, 2), n_sel_pages=6)
    inp = make_inputs(w, device=DEV, seq_lens=[0, 1, 16, 17, 95, 1600])
    p, bufs, err = run_step(inp)
    assert err == 0
    prm = oracle_params(w)
    for b in range(6):
        for h in range(2):
            check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])
    assert bufs.sel_cnt[0].tolist() == [0, 0]
    assert (bufs.out[0] == 0).all() and torch.isneginf(bufs.lse[0]).all()


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
def test_all_equal_scores_take_lowest_pages(step_kernel):
    """Identical pages tie everywhere: the lowest candidate pages win."""
    spg = _spg()
    w = scaled(get_workload("tiny-quest-gqa4-1k"), seq_len=16 * 40, n_sel_pages=7, needles_per_head=0)
    inp = make_inputs(w, device=DEV)
    inp.k_pool[:] = inp.k_pool[0:1, :, :, :]  # every page the same
    _, bufs, _ = run_step(inp)
    assert gpu_selection(bufs, 0, 0) == [0, 1, 2, 3, 4, 5, 39]


def _integer_score_inputs(kind, n_pages=1200, n_sel=100):
    """Pages whose tokens all equal v * e_0 (v an integer, exact in fp16) and
    queries e_0: the Quest bound of a page is exactly v in fp32 and in fp64,
    so ties are exact and the selection has one right answer, also inside
    the tie band.  1200 pages spread each unit's candidates over a cluster
    of 8 CTAs."""
    w = scaled(get_workload("llama2-7b-mha-32k"), num_q_heads=4, num_kv_heads=4,
               seq_len=16 * n_pages + 5, n_sel_pages=n_sel, needles_per_head=0)
    inp = make_inputs(w, device=DEV)
    g = torch.Generator().manual_seed(11)
    shape = (inp.k_pool.shape[0], w.num_kv_heads)
    if kind == "three-values":  # ~400 pages tie at the threshold value: resolved by page index
        vals = torch.randint(0, 3, shape, generator=g)
    elif kind == "wide-integers":  # negative and positive scores, scattered small ties
        vals = torch.randint(-2048, 2049, shape, generator=g)
    else:  # "planted-ties": 40 candidates share the value just inside the top-k
        vals = torch.randint(0, 2048, shape, generator=g)
        P = -(-int(inp.seq_lens[0]) // w.page_size)
        k_top = n_sel - w.n_sink - w.n_recent
        for h in range(w.num_kv_heads):
            phys = inp.page_table[0, w.n_sink:P - w.n_recent].cpu().long()
            cand = vals[phys, h]
            v = int(torch.sort(cand, descending=True).values[k_top - 15])
            pick = torch.randperm(len(phys), generator=g)[:40]
            vals[phys[pick], h] = v
    inp.k_pool.zero_()
    inp.k_pool[..., 0] = vals[:, :, None].to(device=DEV, dtype=inp.k_pool.dtype)
    inp.q.zero_()
    inp.q[..., 0] = 1
    return w, inp


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("kind", ["three-values", "planted-ties", "wide-integers"])
def test_exact_ties_across_the_cluster(kind, step_kernel):
    """Exact ties between pages scored in different CTAs: lower page index wins."""
    w, inp = _integer_score_inputs(kind)
    p, bufs, err = run_step(inp)
    assert err == 0
    prm = oracle_params(w)
    for h in range(w.num_kv_heads):
        sub = unit_inputs(inp, 0, h)
        scores = decode.unit_scores(sub, prm, 0, 0)
        P = -(-int(inp.seq_lens[0]) // w.page_size)
        ref = oselect.select_pages(scores, P, prm.n_sel, prm.n_sink, prm.n_recent)
        assert gpu_selection(bufs, 0, h) == ref
        check_unit(inp, prm, bufs, 0, h, TOL_OUT[w.kv_dtype])


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
def test_budget_of_only_forced_pages(step_kernel):
    """A budget equal to the forced pages selects no candidate."""
    w = scaled(SMALL["mha"], n_sel_pages=2)
    inp = make_inputs(w, device=DEV)
    p, bufs, err = run_step(inp)
    assert err == 0
    P = -(-int(inp.seq_lens[0]) // w.page_size)
    prm = oracle_params(w)
    for h in range(w.num_kv_heads):
        assert gpu_selection(bufs, 0, h) == [0, P - 1]
        check_unit(inp, prm, bufs, 0, h, TOL_OUT[w.kv_dtype])


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("name", ["tiny", "long-d64-g8"])
def test_needle_pages_selected(name, step_kernel):
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    _, bufs, _ = run_step(inp)
    for (b, h), pos in inp.needles.items():
        pages = {t // w.page_size for t in pos}
        assert pages <= set(gpu_selection(bufs, b, h))


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
def test_bad_page_id_is_reported_not_read(step_kernel):
    spg = _spg()
    w = SMALL["tiny"]
    inp = make_inputs(w, device=DEV)
    inp.page_table[0, 5] = inp.num_phys_pages + 1000  # outside the pool
    p, bufs, err = run_step(inp)
    assert err & spg.DEVERR_PAGE_ID
    spg.spg_clear_device_error(bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0


def test_host_validation_errors():
    spg = _spg()
    w = SMALL["tiny"]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    with pytest.raises(spg.SpgError) as e:  # workspace too small
        spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, bufs.minmax, sel=bufs.sel,
                               sel_cnt=bufs.sel_cnt, ws=bufs.ws[:256])
    assert e.value.status == 4
    with pytest.raises(spg.SpgError) as e:  # misaligned query pointer
        spg.sparse_page_select(p, inp.q.view(-1)[1:], inp.page_table, inp.seq_lens, bufs.minmax,
                               sel=bufs.sel, sel_cnt=bufs.sel_cnt, ws=bufs.ws)
    assert e.value.status == 1


# ---- full sizes, sampled units, benchmark launch configuration ----------------
FULL = ["llama2-7b-mha-32k", "gqa-serving-b8-4k-64k", "sals-int8-b16-10k-4x",
        "sals-int8-b16-10k-6x", "long-scan-b4-128k"]


@pytest.mark.parametrize("step_kernel", KERNELS, indirect=True)
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_units(name, step_kernel):
    w = get_workload(name)
    inp = make_inputs(w, device=DEV)
    p, bufs, err = run_step(inp)
    _expect_kernel(p, step_kernel)
    assert err == 0
    prm = oracle_params(w)
    rng = np.random.default_rng(7)
    units = {(0, 0), (w.batch - 1, w.num_kv_heads - 1)}
    while len(units) < 4:
        units.add((int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))))
    for b, h in sorted(units):
        gsel = check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])
        if (b, h) in inp.needles:
            assert {t // w.page_size for t in inp.needles[(b, h)]} <= set(gsel)
    # every unit: count, order and forced pages (properties that hold at any size)
    cnt = bufs.sel_cnt.cpu().numpy()
    sel = bufs.sel.cpu().numpy()
    lens = to_numpy(inp.seq_lens)
    for b in range(w.batch):
        P = -(-int(lens[b]) // w.page_size)
        for h in range(w.num_kv_heads):
            s = sel[b, h, : cnt[b, h]]
            assert cnt[b, h] == min(w.n_sel_pages, P)
            assert np.all(np.diff(s) > 0) and s[0] >= 0 and s[-1] == P - 1
            if w.n_sink:
                assert s[0] == 0


@pytest.mark.parametrize("name", ["gqa-ragged", "sals-4x", "mha"])
def test_repeated_steps_on_one_workspace(name):
    """The scheduled kernel leaves its queue counters and per-unit flags at
    zero: steps launched back to back on one workspace, alternating with the
    cluster kernel and with the separate kernels, give identical results."""
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    ref = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                ref.minmax, ref.sketch, ref.sketch_scale, inp.proj, ref.ws)
    b = spg.alloc_buffers(p, DEV)
    if ref.minmax is not None:
        b.minmax.copy_(ref.minmax)
    else:
        b.sketch.copy_(ref.sketch)
        b.sketch_scale.copy_(ref.sketch_scale)

    def step(bufs):
        spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                        inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                                        bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt,
                                        bufs.out, bufs.lse, bufs.ws)

    try:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_SCHED)
        step(ref)
        torch.cuda.synchronize()
        for kernel in [spg.STEP_KERNEL_SCHED] * 3 + [spg.STEP_KERNEL_CLUSTER, spg.STEP_KERNEL_SCHED]:
            spg.spg_set_step_kernel(kernel)
            step(b)
            if kernel == spg.STEP_KERNEL_CLUSTER:
                spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, b.minmax, b.sketch,
                                       b.sketch_scale, inp.proj, b.sel, b.sel_cnt, b.ws)
                spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale,
                                            inp.v_scale, inp.page_table, inp.seq_lens, b.sel,
                                            b.sel_cnt, b.out, b.lse, b.ws)
                continue
            torch.cuda.synchronize()
            assert torch.equal(b.sel, ref.sel) and torch.equal(b.sel_cnt, ref.sel_cnt)
            assert torch.equal(b.out, ref.out) and torch.equal(b.lse, ref.lse)
        assert spg.spg_read_device_error(b.ws) == 0
        # the workspace's queue counters are back at zero
        hdr = b.ws[64:96].view(torch.int32).cpu()
        assert int(hdr.abs().sum()) == 0, hdr.tolist()
    finally:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)



@pytest.mark.parametrize("name", ["quest-i8", "quest-i8-bf16q-d64"])
def test_int8_quest_metadata_bit_exact_and_append_equals_rebuild(name):
    """Quest over int8 keys: the metadata rebuild equals the oracle's
    outward-rounded min/max of the dequantised keys bit for bit, and token
    by token appends give the same rows."""
    spg = _spg()
    w = SMALL[name]
    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    r = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                r.minmax, None, None, None, r.ws)
    ref = quest.page_minmax_dequant(to_numpy(inp.k_pool), to_numpy(inp.k_scale),
                                    to_numpy(inp.page_table), to_numpy(inp.seq_lens), w.page_size,
                                    w.q_dtype)
    got = to_numpy(r.minmax)
    pt = to_numpy(inp.page_table)
    for b, L in enumerate(to_numpy(inp.seq_lens)):
        for p_ in range(-(-int(L) // w.page_size)):
            for h in range(w.num_kv_heads):
                row = unswizzle_meta_row(got[b, h, p_], p_).astype(np.float64)
                assert np.array_equal(row, ref[pt[b, p_], h]), (b, h, p_)
    a = spg.alloc_buffers(p, DEV)
    a.minmax.fill_(3.0)  # stale rows from a recycled page must not leak
    lens = inp.seq_lens.cpu().tolist()
    for t in range(1, int(max(lens)) + 1):
        cur = torch.clamp(torch.tensor(lens, dtype=torch.int32), max=t).to(DEV)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, cur, 0, a.minmax,
                                    None, None, None, a.ws)
    for b, L in enumerate(lens):
        P = -(-L // w.page_size)
        assert torch.equal(a.minmax[b, :, :P], r.minmax[b, :, :P])
    assert spg.spg_read_device_error(a.ws) == 0
