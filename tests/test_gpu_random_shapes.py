"""Seeded random shapes across the space spg_validate accepts, against the oracle.

Every draw picks a pool type (fp16, bf16, int8 with an fp16 or bf16 query),
a selector (Quest, the sketch selector, or the probe selector on 16-bit
pools), a head size, a query group, a page size whose K/V page fits the
library's stage, a batch with lengths that include empty, one-token and
page-aligned sequences, forced sink / recent pages, a budget (trimmed, in
half the draws, to the smallest prefix holding a fraction p of the score
mass, with a floor), and a physical page order.  The step then runs
through the cluster kernel, the scheduled kernel and the separate score /
select / attend entry points, and through sparse_decode_step on both
single-launch kernels from metadata one token old (the appended metadata
must equal a rebuild bit for bit); every unit's scores, selection and
attention are checked against the oracle (the bars of the hand-picked
parity and top-p shapes).  The dense baseline runs on the same draws
against the oracle's attention over every page.
"""

import numpy as np
import pytest

from oracle import decode

from synth import get_workload, make_inputs, scaled

from conftest import oracle_inputs, oracle_params
from gpu_helpers import TOL_OUT, check_unit, run_step

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_CASES = 24
PATHS = ["cluster", "sched", "separate", "step-cluster", "step-sched"]
MAX_PAGE_BYTES = 34 * 1024  # K + V (+ int8 scales) of one page


def _draw(seed):
    """One valid configuration (re-drawn until spg_validate accepts it)."""
    import query_aware_sparse_page_gb300 as spg

    rng = np.random.default_rng(7_000 + seed)
    for _ in range(100):
        kv = str(rng.choice(["f16", "bf16", "i8"]))
        selector = str(rng.choice(["quest", "sketch"] + ([] if kv == "i8" else ["probe"])))
        q = kv if kv != "i8" else str(rng.choice(["f16", "bf16"]))
        D = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = int(rng.choice([1, 2]))
        B = int(rng.integers(2, 5))
        elem = 1 if kv == "i8" else 2
        sizes = [s for s in (16, 32, 64, 128)
                 if 2 * s * D * elem + (4 * s if kv == "i8" else 0) <= MAX_PAGE_BYTES]
        S = int(rng.choice(sizes))
        lens = [int(x) for x in rng.integers(S, 90 * S + 1, B)]
        # one sequence is empty, one token long, page-aligned, or as long as the first
        lens[int(rng.integers(0, B))] = [0, 1, S * int(rng.integers(1, 8)), lens[0]][int(rng.integers(0, 4))]
        n_sink = int(rng.integers(0, 3))
        n_recent = int(rng.integers(1 if selector == "sketch" else 0, 3))
        n_sel = max(n_sink + n_recent + int(rng.integers(0, 40)), 1)
        # half the draws trim the budget to a fraction of the score mass
        top_p = float(rng.choice([0.5, 0.8, 0.95])) if rng.integers(0, 2) else 0.0
        min_pages = int(rng.integers(0, 4))
        w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=B, num_q_heads=Hkv * G, num_kv_heads=Hkv,
                   head_dim=D, page_size=S, seq_len=max(max(lens), 1), seq_range=None, kv_dtype=kv,
                   q_dtype=q, selector=selector, n_sel_pages=n_sel, n_sink=n_sink, n_recent=n_recent,
                   channel_scales=bool(rng.integers(0, 2)), needles_per_head=int(rng.integers(0, 3)),
                   random_page_table=bool(rng.integers(0, 2)), seed=100 + seed)
        p = spg.make_params(batch=B, num_q_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D, page_size=S,
                            num_phys_pages=max(sum(-(-L // S) for L in lens), 1),
                            max_pages_per_seq=w.max_pages_per_seq, kv_dtype=kv, q_dtype=q,
                            selector=selector, token_budget=n_sel * S, n_sink_pages=n_sink,
                            n_recent_pages=n_recent)
        p.top_p, p.min_pages = top_p, min_pages
        if spg.spg_validate(p) == 0:
            return w, lens, top_p, min_pages
    raise AssertionError("no valid draw")


def _run_probe(spg, inp, path, top_p, min_pages):
    """The probe selector reads the key pool in place of page metadata."""
    import torch

    p = spg.params_for(inp)
    p.top_p, p.min_pages = top_p, min_pages
    bufs = spg.alloc_buffers(p, DEV)
    pool = inp.k_pool
    spg.sparse_page_score(p, inp.q, inp.page_table, inp.seq_lens, pool, None, None, None,
                          bufs.scores, bufs.ws)
    if path == "separate":
        spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, pool, None, None, None,
                               bufs.sel, bufs.sel_cnt, bufs.ws)
        spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table,
                                    inp.seq_lens, bufs.sel, bufs.sel_cnt, bufs.out, bufs.lse, bufs.ws)
    else:
        spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, None, None, inp.page_table,
                                        inp.seq_lens, pool, None, None, None, bufs.sel, bufs.sel_cnt,
                                        bufs.out, bufs.lse, bufs.ws)
    err = spg.spg_read_device_error(bufs.ws)
    torch.cuda.synchronize()
    return p, bufs, err


def _run_decode_step(spg, inp, top_p, min_pages):
    """sparse_decode_step: metadata as of one token earlier, then the step
    appends the last token's metadata, selects and attends.  The appended
    metadata must equal a full rebuild bit for bit; the scores are then taken
    from it for the oracle comparison."""
    import torch

    p = spg.params_for(inp)
    p.top_p, p.min_pages = top_p, min_pages
    got = spg.alloc_buffers(p, DEV)
    probe = inp.workload.selector == "probe"
    proj = None if probe else inp.proj
    if probe:
        got.minmax = inp.k_pool  # the probe selector reads the pool itself
    else:
        ref = spg.alloc_buffers(p, DEV)
        prev = (inp.seq_lens - 1).clamp(min=0)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, prev, 1, got.minmax,
                                    got.sketch, got.sketch_scale, proj, got.ws)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                    ref.minmax, ref.sketch, ref.sketch_scale, proj, ref.ws)
    spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                           inp.page_table, inp.seq_lens, got.minmax, got.sketch, got.sketch_scale,
                           proj, got.sel, got.sel_cnt, got.out, got.lse, got.ws)
    err = spg.spg_read_device_error(got.ws)
    torch.cuda.synchronize()
    if not probe and err == 0:
        if got.sketch is None:
            assert torch.equal(got.minmax, ref.minmax), "appended min/max differ from a rebuild"
        else:
            assert torch.equal(got.sketch, ref.sketch), "appended sketch codes differ from a rebuild"
            assert torch.equal(got.sketch_scale, ref.sketch_scale), "appended sketch scales differ"
    spg.sparse_page_score(p, inp.q, inp.page_table, inp.seq_lens, got.minmax, got.sketch,
                          got.sketch_scale, proj, got.scores, got.ws)
    torch.cuda.synchronize()
    return p, got, err


@pytest.fixture
def path(request):
    import query_aware_sparse_page_gb300 as spg

    name = request.param
    spg.spg_set_step_kernel(spg.STEP_KERNEL_SCHED if name.endswith("sched") else spg.STEP_KERNEL_CLUSTER)
    yield name
    spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)


@pytest.mark.parametrize("path", PATHS, indirect=True)
@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape_matches_oracle(seed, path):
    import query_aware_sparse_page_gb300 as spg

    w, lens, top_p, min_pages = _draw(seed)
    inp = make_inputs(w, device=DEV, seq_lens=lens)
    prm = oracle_params(w)
    prm.top_p, prm.min_pages = top_p, min_pages
    if path.startswith("step"):
        if w.selector != "probe" and w.n_recent >= 1:
            want = "k_sched" if path.endswith("sched") else "k_fused"
            assert spg.step_kernel_name(spg.params_for(inp)) == want
        p, bufs, err = _run_decode_step(spg, inp, top_p, min_pages)
        if w.selector == "probe":
            prm.n_probe = 8
    elif w.selector == "probe":
        p, bufs, err = _run_probe(spg, inp, path, top_p, min_pages)
        prm.n_probe = 8  # the library's default sample count
    else:
        p = spg.params_for(inp)
        if path != "separate" and w.n_recent >= 1:
            # the query names sparse_decode_step's kernel; without a forced
            # recent page that step appends in a separate launch, while
            # select + attend still takes the chosen single-launch kernel
            want = "k_sched" if path == "sched" else "k_fused"
            assert spg.step_kernel_name(p) == want, spg.step_kernel_name(p)
        p, bufs, err = run_step(inp, fused=path != "separate", top_p=top_p, min_pages=min_pages)
    assert err == 0, f"device error {err:#x} ({w}, lengths {lens})"
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            check_unit(inp, prm, bufs, b, h, TOL_OUT[w.kv_dtype])


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape_dense_matches_oracle(seed):
    """The dense flash-decoding baseline (split planned by sequence length)
    on the same draws: every unit's attention over its whole sequence."""
    import query_aware_sparse_page_gb300 as spg

    w, lens, _, _ = _draw(seed)
    inp = make_inputs(w, device=DEV, seq_lens=lens)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, bufs.out, bufs.lse, bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0
    res = decode.decode_step(oracle_inputs(inp), oracle_params(w, selector="all"))
    G, tol = w.group, TOL_OUT[w.kv_dtype]
    for (b, h), out in res["out"].items():
        gout = bufs.out[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
        glse = bufs.lse[b, h * G:(h + 1) * G].cpu().numpy().astype(np.float64)
        assert np.abs(gout - out).max() <= tol, f"unit {(b, h)} out"
        if lens[b] == 0:
            assert np.isneginf(glse).all()
        else:
            assert np.abs(glse - res["lse"][(b, h)]).max() <= tol, f"unit {(b, h)} lse"
