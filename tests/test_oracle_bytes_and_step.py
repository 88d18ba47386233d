"""Pins for the byte model (worked numbers printed on the pages) and for the
oracle decode step on the seeded workloads (planted needles are found; with
every page selected the sparse step equals the dense one)."""

import json
import os

import numpy as np
import pytest

from oracle import bytes as obytes
from oracle import decode, quest
from synth import get_workload, make_inputs, scaled

from conftest import oracle_inputs, oracle_params

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_read_ratio_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "quest_read_ratio.json")))
    r = obytes.read_ratio(g["page_size"], g["seq_len"], g["k_pages"])
    assert r == g["read_ratio"]
    assert round(1 / r) == g["reduction"]
    assert g["seq_len"] // g["page_size"] == g["page_num"]


def test_kv_cache_sizes_printed_on_pages():
    for c in json.load(open(os.path.join(GOLDEN, "kv_cache_sizes.json")))["cases"]:
        got = obytes.kv_cache_bytes(c["n_layers"], c["seq_len"], c["n_kv_heads"], c["head_dim"], c["elem_bytes"])
        assert got == c["bytes"]


def test_step_bytes_reduces_to_read_ratio():
    # one head, fp16: meta of every page + K/V of the selected pages, against the whole K/V
    S, L, K, d = 16, 65536, 256, 128
    meta_and_kv = obytes.step_bytes([L], 1, 1, d, S, 2, "quest", K * S, L // S) - (d * 2 + (d + 1) * 4)
    dense = 2 * L * d * 2
    assert meta_and_kv / dense == pytest.approx(obytes.read_ratio(S, L, K) , rel=1e-12)


@pytest.mark.parametrize("name", ["tiny-quest-gqa4-1k", "long-scan-b4-128k"])
def test_planted_needles_are_selected(name):
    w = get_workload(name)
    if name != "tiny-quest-gqa4-1k":
        w = scaled(w, batch=1, seq_len=8192, num_q_heads=8, num_kv_heads=2, needles_per_head=8)
    inp = make_inputs(w)
    oi, prm = oracle_inputs(inp), oracle_params(w)
    res = decode.decode_step(oi, prm)
    for (b, h), pos in inp.needles.items():
        pages = {t // w.page_size for t in pos}
        assert pages <= set(res["sel"][(b, h)])


def test_full_budget_equals_dense():
    w = scaled(get_workload("tiny-quest-gqa4-1k"), seq_len=301)
    inp = make_inputs(w)
    oi = oracle_inputs(inp)
    sparse = decode.decode_step(oi, decode.StepParams(16, 64, 1, 1, "quest", w.head_dim))
    dense = decode.decode_step(oi, decode.StepParams(16, 0, 0, 0, "all", w.head_dim))
    for key in dense["out"]:
        assert sparse["sel"][key] == list(range(quest.num_pages(301, 16)))
        assert np.array_equal(sparse["out"][key], dense["out"][key])


def test_sketch_step_runs_and_forces_tail():
    w = scaled(get_workload("sals-int8-b16-10k-4x"), batch=2, seq_len=64 * 20 + 5, n_sel_pages=6)
    inp = make_inputs(w)
    res = decode.decode_step(oracle_inputs(inp), oracle_params(w))
    P = 21
    for key, sel in res["sel"].items():
        assert len(sel) == 6 and sel[-1] == P - 1
        sc = res["scores"][key]
        assert np.isnan(sc[P - 1]) and np.isfinite(sc[: P - 1]).all()


@pytest.mark.parametrize("S", [16, 64, 128])
def test_sketch_metadata_bytes_are_the_stored_arrays(S):
    """The sketch term counts, per scored block, exactly the bytes the index
    key occupies: the packed int4 codes of its S tokens x d_s channels and
    one fp32 scale (measured on arrays built by the oracle's own packer)."""
    from oracle import sketch

    ds = 16
    packed = sketch.pack_int4(np.zeros((S, ds), np.int8))
    per_block = packed.nbytes + np.float32(1.0).nbytes
    small = obytes.step_bytes([S * 10], 1, 1, 128, S, 1, "sketch", 0, 0, sketch_dim=ds)
    for n in (1, 7, 159):
        got = obytes.step_bytes([S * 10], 1, 1, 128, S, 1, "sketch", 0, n, sketch_dim=ds) - small
        assert got == n * per_block
    if S == 64:
        # the 10K-token SALS workload: 16 sequences x 8 kv-heads x 159 scored
        # blocks of 512 + 4 bytes
        meta = obytes.step_bytes([10240] * 16, 8, 32, 128, 64, 1, "sketch", 0, 16 * 8 * 159,
                                 sketch_dim=16) - obytes.step_bytes([10240] * 16, 8, 32, 128, 64, 1,
                                                                    "sketch", 0, 0, sketch_dim=16)
        assert meta == 10_501_632


@pytest.mark.parametrize("name", ["tiny-quest-gqa4-1k", "llama2-7b-mha-32k", "gqa-serving-b8-4k-64k",
                                  "sals-int8-b16-10k-4x", "sals-int8-b16-10k-6x", "long-scan-b4-128k"])
def test_bench_byte_model_equals_the_oracle_byte_model(name):
    """bench.py keeps its own copy of the byte model (it may not import the
    oracle on its timed path); both must count the same bytes."""
    import bench

    w = get_workload(name)
    kvb = 1 if w.kv_dtype == "i8" else 2
    for sel_tok, cand, sel_pages in [(0, 0, 0), (2048 * w.num_kv_heads, 2046 * w.num_kv_heads, 128),
                                     (12345, 6789, 321)]:
        meta, kv, small = bench.step_bytes(w, None, sel_tok, cand, sel_pages)
        lens = [w.seq_len or w.seq_range[1]] * w.batch
        ref = obytes.step_bytes(lens, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size, kvb,
                                w.selector, sel_tok, cand, sketch_dim=w.sketch_dim,
                                scale_bytes=2 if w.kv_dtype == "i8" else 0, q_bytes=2,
                                sel_pages=sel_pages)
        assert meta + kv + small == ref
