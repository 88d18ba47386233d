"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
and compare against the oracle with the stated tolerances."""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import decode, select
from conftest import to_numpy

TOL_OUT = {"f16": 2e-3, "bf16": 2e-3, "i8": 5e-3}  # max-abs on out and lse
MASS_BAND = 1e-4  # |oracle cumulative mass - p| under which several top-p counts are correct
REL_GAP = 1e-5  # k-th / (k+1)-th oracle score gap under which several selections are correct

# Two GPU paths over the same selection differ only by arithmetic order, and
# by the tensor-core path rounding the probabilities P to the pool's 16-bit
# type as a hi + lo pair: |p - hi - lo| <= 2^-(2 s) p with s = 9 (bf16) or 11
# (fp16) significand bits, so an output row moves by at most that times
# max |v|.  Bound used: 4x that, plus 1e-5 for the order of fp32 sums; the
# log-sum-exp agrees to fp32 rounding relative to its size.
_P_SPLIT = {"f16": 2.0 ** -22, "bf16": 2.0 ** -18, "i8": 0.0}


def assert_paths_agree(out_a, out_b, lse_a, lse_b, kv_dtype, vmax):
    tol_out = 1e-5 + 4 * _P_SPLIT[kv_dtype] * float(vmax)
    d_out = (out_a - out_b).abs().max().item()
    assert d_out <= tol_out, f"out differs by {d_out:.3e} > {tol_out:.3e}"
    if lse_a is not None:
        fin = torch.isfinite(lse_a) & torch.isfinite(lse_b)
        assert torch.equal(torch.isfinite(lse_a), torch.isfinite(lse_b))
        if fin.any():
            d = (lse_a[fin] - lse_b[fin]).abs()
            tol = 2e-6 * lse_a[fin].abs().clamp(min=1.0)
            assert bool((d <= tol).all()), f"lse differs by {d.max().item():.3e}"


def run_step(inp, selector=None, n_sel_pages=None, fused=True, rebuild=True, bufs=None,
             top_p=0.0, min_pages=0):
    """Metadata rebuild, then select + attend on the GPU; returns host copies."""
    import query_aware_sparse_page_gb300 as spg

    p = spg.params_for(inp, selector=selector, n_sel_pages=n_sel_pages)
    p.top_p, p.min_pages = top_p, min_pages
    if bufs is None:
        bufs = spg.alloc_buffers(p, inp.q.device)
    if rebuild:
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                    bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    spg.sparse_page_score(p, inp.q, inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                          bufs.sketch_scale, inp.proj, bufs.scores, bufs.ws)
    if fused:
        spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                        inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                                        bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt,
                                        bufs.out, bufs.lse, bufs.ws)
    else:
        spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, bufs.minmax, bufs.sketch,
                               bufs.sketch_scale, inp.proj, bufs.sel, bufs.sel_cnt, bufs.ws)
        spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                    inp.page_table, inp.seq_lens, bufs.sel, bufs.sel_cnt,
                                    bufs.out, bufs.lse, bufs.ws)
    err = spg.spg_read_device_error(bufs.ws)
    torch.cuda.synchronize()
    return p, bufs, err


def unswizzle_meta_row(row, p, elem_bytes=2):
    """A Quest metadata row as stored (16-byte chunks XOR-swizzled by page p)
    back in channel order: [2][d] (m, then M).  elem_bytes: size of one
    stored element (2 for fp16/bf16, whatever dtype `row` was widened to)."""
    row = np.asarray(row)
    flat = row.reshape(-1)
    epc = 16 // elem_bytes
    chunks = flat.reshape(-1, epc)
    perm = [c ^ (p & 7) for c in range(chunks.shape[0])]
    return chunks[perm].reshape(row.shape)


def gpu_selection(bufs, b, h):
    cnt = int(bufs.sel_cnt[b, h])
    row = bufs.sel[b, h].cpu().tolist()
    assert all(x == -1 for x in row[cnt:]), "unused sel entries must be -1"
    return row[:cnt]


def assert_selection_matches(gpu_sel, scores, P, n_sel, n_sink, n_recent, rel_gap=REL_GAP):
    """Exact equality, except inside a tie band of the oracle's k-th / (k+1)-th scores."""
    ref = select.select_pages(scores, P, n_sel, n_sink, n_recent)
    if gpu_sel == ref:
        return
    forced = select.forced_pages(P, n_sink, n_recent)
    fset = set(forced)
    cand = [p for p in range(P) if p not in fset]
    k_top = min(max(n_sel - len(forced), 0), len(cand))
    ranked = sorted(cand, key=lambda p: (-float(scores[p]), p))
    assert 0 < k_top < len(cand), f"selection differs with no tie possible: {gpu_sel} vs {ref}"
    sk, sk1 = float(scores[ranked[k_top - 1]]), float(scores[ranked[k_top]])
    band = rel_gap * max(abs(sk), 1e-30)
    assert abs(sk - sk1) <= band, (
        f"selection differs outside the tie band (gap {abs(sk - sk1):.3e}, band {band:.3e})")
    g = set(gpu_sel)
    assert len(gpu_sel) == len(ref) and fset <= g and gpu_sel == sorted(g)
    for p in cand:
        if float(scores[p]) > sk + band:
            assert p in g, f"page {p} scores above the tie band but was not selected"
    # every selected candidate lies in or above the tie band: a tied page may
    # stand in for another tied page, never for a lower-scoring one
    for p in g - fset:
        assert float(scores[p]) >= sk1 - band, (
            f"selected page {p} scores {float(scores[p]):.6e}, below the tie band at {sk1 - band:.6e}")


def allowed_top_p_counts(scores, ranked, k_budget, top_p, min_pages, tau):
    """Candidate counts the adaptive budget may keep: the oracle's, and any
    whose cumulative mass brackets p within MASS_BAND (then floored and
    capped).  The GPU sums fp32 weights where the oracle sums fp64 ones, so
    its count may differ only where the oracle's cumulative mass lies that
    close to p."""
    s = [float(scores[p]) for p in ranked]
    mx = max(s)
    w = [math.exp(tau * (x - mx)) for x in s]
    z = math.fsum(w)
    cum = np.cumsum(w) / z
    ks = set()
    for j in range(1, len(s) + 1):
        lo = cum[j - 2] if j >= 2 else 0.0
        if lo < top_p + MASS_BAND and cum[j - 1] >= top_p - MASS_BAND:
            ks.add(j)
    if not ks:
        ks.add(len(s))
    return {min(k_budget, max(k, min(min_pages, k_budget))) for k in ks}


def top_p_count(gsel, scores, P, prm):
    """Pages the adaptive budget kept (forced ones included), checked to be a
    count the oracle's cumulative mass allows."""
    forced = select.forced_pages(P, prm.n_sink, prm.n_recent)
    fset = set(forced)
    cand = [q for q in range(P) if q not in fset]
    k_budget = min(max(prm.n_sel - len(forced), 0), len(cand))
    k_gpu = len(gsel) - len(forced)
    if k_budget > 0:
        ranked = sorted(cand, key=lambda q: (-float(scores[q]), q))
        ok = allowed_top_p_counts(scores, ranked, k_budget, prm.top_p, prm.min_pages, prm.tau)
    else:
        ok = {0}
    assert k_gpu in ok, f"kept {k_gpu} candidates, allowed {sorted(ok)}"
    return len(forced) + k_gpu


def unit_inputs(inp, b, h):
    """Oracle inputs reduced to one (batch, kv-head) unit, pages renumbered 0..P-1."""
    w = inp.workload
    S, G = w.page_size, w.group
    L = int(inp.seq_lens[b])
    P = -(-L // S)
    phys = inp.page_table[b, :P].long()
    sub = lambda t: None if t is None else to_numpy(t[phys][:, h : h + 1])
    return decode.StepInputs(
        q=to_numpy(inp.q[b : b + 1, h * G : (h + 1) * G]),
        k_pool=sub(inp.k_pool), v_pool=sub(inp.v_pool),
        k_scale=sub(inp.k_scale), v_scale=sub(inp.v_scale),
        page_table=np.arange(max(P, 1))[None, :], seq_lens=np.array([L]),
        proj=to_numpy(inp.proj),
    )


def check_unit(inp, prm, bufs, b, h, tol):
    """Scores, selection and attention of one unit against the oracle."""
    sub = unit_inputs(inp, b, h)
    L = int(inp.seq_lens[b])
    P = -(-L // prm.page_size)
    G = inp.workload.group
    gsel = gpu_selection(bufs, b, h)
    if prm.selector != "all":
        scores = decode.unit_scores(sub, prm, 0, 0)
        lo = min(prm.n_sink, P)
        hi = max(P - prm.n_recent, lo)
        gsc = bufs.scores[b, h, :P].cpu().numpy().astype(np.float64)
        cand = np.arange(lo, hi)
        if len(cand):
            ref = scores[cand]
            assert np.all(np.abs(gsc[cand] - ref) <= 1e-5 * (np.abs(ref) + 1.0)), \
                f"score mismatch max {np.abs(gsc[cand] - ref).max():.3e}"
        assert np.all(np.isneginf(np.delete(gsc, cand)))
        n_sel = top_p_count(gsel, scores, P, prm) if prm.top_p > 0.0 else prm.n_sel
        assert_selection_matches(gsel, scores, P, n_sel, prm.n_sink, prm.n_recent)
    out, lse = decode.attend_selection(sub, prm, 0, 0, gsel)
    gout = bufs.out[b, h * G : (h + 1) * G].cpu().numpy().astype(np.float64)
    glse = bufs.lse[b, h * G : (h + 1) * G].cpu().numpy().astype(np.float64)
    assert np.abs(gout - out).max() <= tol, f"out max-abs {np.abs(gout - out).max():.3e}"
    if L == 0:
        assert np.isneginf(glse).all()
    else:
        assert np.abs(glse - lse).max() <= tol, f"lse max-abs {np.abs(glse - lse).max():.3e}"
    return gsel
