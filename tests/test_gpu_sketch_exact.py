"""The sketch selector's integer arithmetic, bit for bit against the oracle.

SALS长序列推理优化, Quant Sals Indexer steps 1-2: the int8 index query and
the int4 index key meet in an integer product before any dequantisation, so
the GPU's query codes, their scale and every per-token dot must equal the
oracle's exactly (the oracle builds the codes from the K pool with the same
fp32 rule, independently of the GPU's metadata).  Full-size SALS workloads
(4x and 6x), every unit's index query and sampled units' dots.
"""

import numpy as np
import pytest
import torch

from oracle import sketch as osk
from synth import get_workload, make_inputs, scaled

from conftest import to_numpy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(w):
    import query_aware_sparse_page_gb300 as spg

    inp = make_inputs(w, device=DEV)
    p = spg.params_for(inp)
    bufs = spg.alloc_buffers(p, DEV)
    spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1, None,
                                bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
    B, Hkv, MP, S = w.batch, w.num_kv_heads, p.max_pages_per_seq, w.page_size
    qc = torch.full((B, Hkv, 16), 999, dtype=torch.int32, device=DEV)
    sq = torch.full((B, Hkv), float("nan"), dtype=torch.float32, device=DEV)
    dots = torch.full((B, Hkv, MP, S), -(1 << 30), dtype=torch.int32, device=DEV)
    spg.sparse_page_sketch_dots(p, inp.q, inp.seq_lens, bufs.sketch, inp.proj, qc, sq, dots, bufs.ws)
    assert spg.spg_read_device_error(bufs.ws) == 0
    torch.cuda.synchronize()
    return inp, p, bufs, qc.cpu().numpy(), sq.cpu().numpy(), dots.cpu().numpy()


def _check(w, units_to_dot):
    inp, p, bufs, qc, sq, dots = _run(w)
    S, G = w.page_size, w.group
    q = to_numpy(inp.q).astype(np.float32)
    proj = to_numpy(inp.proj)
    kp, ks, pt = to_numpy(inp.k_pool), to_numpy(inp.k_scale), to_numpy(inp.page_table)
    lens = to_numpy(inp.seq_lens)
    # every unit's index query: codes and scale exactly
    ref_q = {}
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            qc_o, sq_o = osk.index_query(q[b, h * G:(h + 1) * G], proj)
            ref_q[(b, h)] = qc_o
            assert np.array_equal(qc[b, h], qc_o.astype(np.int32)), (b, h)
            assert np.float32(sq[b, h]) == sq_o, (b, h, float(sq[b, h]), float(sq_o))
    # every token of every candidate block of the sampled units: exact dots
    n = 0
    for b, h in units_to_dot:
        L = int(lens[b])
        P = -(-L // S)
        lo, hi = min(w.n_sink, P), max(P - w.n_recent, min(w.n_sink, P))
        for blk in range(p.max_pages_per_seq):
            got = dots[b, h, blk]
            if not (lo <= blk < hi):
                assert not got.any(), f"non-candidate block {blk} has dots"
                continue
            phys = int(pt[b, blk])
            kd = osk.dequant(kp[phys, h], ks[phys, h]) if ks is not None else kp[phys, h].astype(np.float32)
            codes, _ = osk.build_sketch(kd, proj)
            ref = osk.int_dots(ref_q[(b, h)], codes)
            assert np.array_equal(got.astype(np.int64), ref), f"unit {(b, h)} block {blk}"
            n += 1
    assert n > 0


@pytest.mark.parametrize("name", ["sals-int8-b16-10k-4x", "sals-int8-b16-10k-6x"])
def test_index_query_and_dots_bit_exact_full_size(name):
    w = get_workload(name)
    rng = np.random.default_rng(3)
    units = {(0, 0), (w.batch - 1, w.num_kv_heads - 1)}
    while len(units) < 4:
        units.add((int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))))
    _check(w, sorted(units))


@pytest.mark.parametrize("q_dtype,kv_dtype", [("bf16", "i8"), ("bf16", "bf16"), ("f16", "f16")])
def test_index_query_and_dots_other_dtypes(q_dtype, kv_dtype):
    """The query rows in bf16 (int8 pools accept either 16-bit query type),
    and the sketch selector over 16-bit pools; ragged tail, G = 4."""
    w = scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, num_q_heads=8, num_kv_heads=2,
               seq_len=64 * 21 + 9, n_sel_pages=7, q_dtype=q_dtype, kv_dtype=kv_dtype)
    _check(w, [(b, h) for b in range(2) for h in range(2)])
