"""Host-side pieces of bench.py that decide what a benchmark line may claim."""

import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "query_aware_sparse_page_gb300", "csrc")


@pytest.fixture(scope="module")
def bench():
    import bench as b

    return b


def _copy_csrc(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d, ignore=shutil.ignore_patterns("*.o", "*.so", "__pycache__"))
    return d


def test_code_hash_ignores_comments_and_whitespace(bench, tmp_path):
    """ncu traffic figures stay attached to the kernel code: editing a comment
    or the layout of a source does not detach them."""
    d = _copy_csrc(tmp_path)
    h0 = bench.csrc_sha256(str(d))
    assert h0 == bench.csrc_sha256(CSRC)
    f = d / "spg_fused.cu"
    text = f.read_text(encoding="utf-8")
    f.write_text("// a new comment line\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3),
                 encoding="utf-8")
    assert bench.csrc_sha256(str(d)) == h0


def test_code_hash_follows_code_changes(bench, tmp_path):
    d = _copy_csrc(tmp_path)
    h0 = bench.csrc_sha256(str(d))
    f = d / "spg_common.cuh"
    text = f.read_text(encoding="utf-8")
    assert "kMaxSplits = 128" in text
    f.write_text(text.replace("kMaxSplits = 128", "kMaxSplits = 64", 1), encoding="utf-8")
    assert bench.csrc_sha256(str(d)) != h0


def test_traffic_is_reported_only_for_the_captured_code(bench, monkeypatch):
    wl = "llama2-7b-mha-32k"
    traffic, src = bench.ncu_traffic(wl)
    if bench.NCU_TRAFFIC[wl][1] == bench.csrc_sha256():
        assert traffic == bench.NCU_TRAFFIC[wl][0] and src.startswith("profiles/")
    monkeypatch.setattr(bench, "csrc_sha256", lambda d=None: "0" * 64)
    assert bench.ncu_traffic(wl) == (None, "kernel sources changed since the ncu capture")
    assert bench.ncu_traffic("no-such-workload")[0] is None


def test_layer_bytes_average_the_replicas(bench):
    """Replicas of a ragged batch draw different lengths: a timed step, which
    cycles through them, is divided by the mean of their bytes, each replica
    counted with its own selection."""
    from types import SimpleNamespace

    import torch

    from synth import get_workload, make_inputs, scaled

    w = scaled(get_workload("gqa-serving-b8-4k-64k"), batch=3, num_q_heads=8, num_kv_heads=2,
               seq_range=(100, 3000), n_sel_pages=24)
    layers = []
    for l in range(2):
        inp = make_inputs(w, device="cpu", seed_offset=l)
        sel = torch.full((w.batch, w.num_kv_heads, w.n_sel_pages), -1, dtype=torch.int32)
        cnt = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32)
        for b, L in enumerate(inp.seq_lens.tolist()):
            n = min(-(-L // w.page_size), w.n_sel_pages)
            sel[b, :, :n] = torch.arange(n, dtype=torch.int32)
            cnt[b, :] = n
        layers.append((inp, None, SimpleNamespace(sel=sel, sel_cnt=cnt)))
    one = [bench.layer_bytes(w, [layer]) for layer in layers]
    both = bench.layer_bytes(w, layers)
    assert one[0] != one[1], "the two replicas should differ in length"
    for i in range(4):
        assert both[i] == (one[0][i] + one[1][i]) // 2


def test_pool_rows_match_advanced_indexing():
    """The end-to-end step writes the new tokens' K/V rows (and int8 scales)
    through flat row indices: they must address exactly pool[phys, :, slot]."""
    import torch

    import bench

    g = torch.Generator().manual_seed(3)
    NP, Hkv, S, d = 41, 3, 16, 8
    pool = torch.randn(NP, Hkv, S, d, generator=g)
    scale = torch.randn(NP, Hkv, S, generator=g)
    phys = torch.tensor([5, 40, 0, 17])
    slot = torch.tensor([0, 15, 7, 3])
    rows = bench.pool_rows(phys, slot, Hkv, S)
    assert torch.equal(pool.view(-1, d)[rows], pool[phys, :, slot].reshape(-1, d))
    assert torch.equal(scale.view(-1)[rows], scale[phys, :, slot].reshape(-1))
    src = torch.randn(len(phys), Hkv, d, generator=g)
    a, b = pool.clone(), pool.clone()
    a.view(-1, d).index_copy_(0, rows, src.reshape(-1, d))
    b[phys, :, slot] = src
    assert torch.equal(a, b)
