"""The C-ABI library builds, loads and exports every symbol include/spg.h
declares; host-side validation answers without touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spg.h")


@pytest.fixture(scope="module")
def spg():
    import __graft_entry__

    __graft_entry__.build()
    import query_aware_sparse_page_gb300 as m

    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:spg_status|int32_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["sparse_page_meta_update", "sparse_page_select", "sparse_decode_attention",
              "sparse_decode_select_attend", "dense_decode_attention", "sparse_page_score",
              "spg_workspace_size", "spg_validate"]:
        assert n in names


def test_library_exports_every_declared_symbol(spg):
    lib = ctypes.CDLL(spg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(spg):
    assert spg.spg_abi_version() == 2
    assert spg.status_str(0) == "ok"
    assert spg.status_str(4) == "workspace too small"
    assert spg.status_str(99) == "unknown status"


def _valid(spg, **kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                num_phys_pages=100, max_pages_per_seq=64, kv_dtype="f16", selector="quest",
                token_budget=16 * 8, n_sink_pages=1, n_recent_pages=1)
    base.update(kw)
    return spg.make_params(**base)


def test_every_workload_validates(spg):
    from synth import WORKLOADS, make_inputs, scaled

    for w in WORKLOADS.values():
        small = scaled(w, batch=1, seq_len=w.page_size * 4, seq_range=None)
        inp = make_inputs(small)
        p = spg.params_for(inp)
        assert spg.spg_validate(p) == 0, w.name
        assert spg.spg_workspace_size(p) > 0


@pytest.mark.parametrize("change, status", [
    (dict(num_q_heads=7), 1),                 # Hq % Hkv
    (dict(head_dim=48), 1),                   # not a multiple of 32
    (dict(head_dim=96), 2),                   # valid, not built
    (dict(num_q_heads=6), 2),                 # group of 3
    (dict(page_size=12), 1),
    (dict(page_size=256), 1),
    (dict(page_size=8), 2),                   # valid, not built: tensor-core tiles are 16 tokens
    (dict(page_size=128, token_budget=512), 2),  # fp16 K + V of a 128-token d128 page: 64 KB
    (dict(page_size=128, token_budget=512, head_dim=64), 0),
    (dict(page_size=64, token_budget=256), 0),
    (dict(page_size=128, token_budget=512, selector="sketch", kv_dtype="i8"), 0),
    (dict(token_budget=100), 1),              # not a multiple of the page size
    (dict(token_budget=16), 1),               # budget below the forced pages
    (dict(n_sink_pages=-1), 1),
    (dict(kv_dtype="i8"), 0),                 # Quest over int8: dequantised metadata
    (dict(kv_dtype="i8", selector="probe"), 2),  # the probe selector samples 16-bit keys only
    (dict(kv_dtype="bf16", q_dtype="f16"), 1),
    (dict(selector="sketch", sketch_dim=8), 1),
    (dict(selector="sketch", n_recent_pages=0), 1),
    (dict(softmax_scale=-1.0), 1),
    (dict(max_pages_per_seq=100000), 2),      # beyond the shared-memory top-k
    (dict(batch=0), 1),
    (dict(top_p=1.5), 1),
    (dict(top_p=-0.1), 1),
    (dict(min_pages=-1), 1),
    (dict(top_p=0.9, min_pages=2), 0),
    (dict(top_p=0.9, token_budget=16 * 1025, max_pages_per_seq=2048, num_phys_pages=4096), 2),
])
def test_validation(spg, change, status):
    assert spg.spg_validate(_valid(spg, **change)) == status


def test_sketch_int8_and_dense_params_are_valid(spg):
    assert spg.spg_validate(_valid(spg, selector="sketch", kv_dtype="i8", page_size=64)) == 0
    assert spg.spg_validate(_valid(spg, selector="all", token_budget=0, n_sink_pages=0,
                                   n_recent_pages=0)) == 0


def test_null_arguments_rejected_on_host(spg):
    p = _valid(spg)
    L = spg.LIB
    null = None
    assert L.sparse_page_select(ctypes.byref(p), null, null, null, null, null, null, null, null,
                                null, null, 0, null) == 1
    assert L.sparse_decode_attention(ctypes.byref(p), *([null] * 12), 0, null) == 1
    assert L.dense_decode_attention(ctypes.byref(p), *([null] * 10), 0, null) == 1
    assert L.sparse_page_meta_update(ctypes.byref(p), null, null, null, null, 0, null, null, null,
                                     null, null, 0, null) == 1
    assert L.spg_validate(None) == 1
    n = ctypes.c_size_t(0)
    assert L.spg_workspace_size(ctypes.byref(_valid(spg, head_dim=48)), ctypes.byref(n)) == 1


def test_workspace_grows_with_the_problem(spg):
    a = spg.spg_workspace_size(_valid(spg))
    b = spg.spg_workspace_size(_valid(spg, batch=4))
    c = spg.spg_workspace_size(_valid(spg, max_pages_per_seq=4096))
    assert a < b and a < c


def test_binding_refuses_host_tensors(spg):
    import torch

    p = _valid(spg)
    t = torch.zeros(16)
    with pytest.raises(ValueError):
        spg.sparse_page_score(p, t, t, t, t, scores=t, ws=torch.zeros(16, dtype=torch.uint8))


def test_step_kernel_queries(spg):
    """Host-only: which kernel the decode step launches, and how many times.
    The cluster kernel takes every benchmark workload in one launch (the
    scheduled kernel when it is preferred); a page table past 8192 pages
    takes the separate kernels."""
    from synth import WORKLOADS

    for w in WORKLOADS.values():
        p = spg.make_params(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                            head_dim=w.head_dim, page_size=w.page_size, num_phys_pages=1 << 16,
                            max_pages_per_seq=w.max_pages_per_seq, kv_dtype=w.kv_dtype,
                            q_dtype=w.q_dtype, selector=w.selector, token_budget=w.token_budget,
                            n_sink_pages=w.n_sink, n_recent_pages=w.n_recent)
        assert spg.step_kernel_name(p) == "k_fused", w.name
        assert spg.step_launch_count(p) == 1
    try:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_SCHED)
        assert spg.step_kernel_name(p) == "k_sched"
        assert spg.step_launch_count(p) == 1
    finally:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)
    with pytest.raises(spg.SpgError):
        spg.spg_set_step_kernel(7)
    long = _valid(spg, max_pages_per_seq=9000, num_phys_pages=20000)
    assert spg.step_kernel_name(long) == "k_quest_select+k_attn"
    assert spg.step_launch_count(long) == 4
    assert spg.step_kernel_name(_valid(spg, head_dim=48)) is None
    assert spg.step_launch_count(_valid(spg, head_dim=48)) == 0


@pytest.mark.parametrize("selector", ["quest", "sketch", "probe"])
@pytest.mark.parametrize("n_recent", [0, 1, 2])
@pytest.mark.parametrize("pref", ["auto", "cluster", "sched"])
def test_step_routing_grid(spg, selector, n_recent, pref):
    """Host-only: the kernel sparse_decode_step takes and its launch count,
    over selector x forced recent pages x step-kernel preference.  The probe
    selector always takes its selection launch and the attention launch; the
    others take the chosen single-launch kernel when the appended token's
    page is forced (its append then runs inside the launch), else a separate
    append, the scoring/selection launch and the attention launch; the
    sketch selector requires a forced recent (tail) block."""
    code = {"auto": spg.STEP_KERNEL_AUTO, "cluster": spg.STEP_KERNEL_CLUSTER,
            "sched": spg.STEP_KERNEL_SCHED}[pref]
    p = _valid(spg, selector=selector, n_recent_pages=n_recent, n_sink_pages=0,
               page_size=64 if selector == "sketch" else 16)
    if selector == "sketch" and n_recent == 0:
        # the sketch selector always forces the open tail block
        assert spg.spg_validate(p) != 0
        assert spg.step_kernel_name(p) is None and spg.step_launch_count(p) == 0
        return
    assert spg.spg_validate(p) == 0
    try:
        spg.spg_set_step_kernel(code)
        name, launches = spg.step_kernel_name(p), spg.step_launch_count(p)
    finally:
        spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)
    if selector == "probe":
        assert (name, launches) == ("k_probe_select+k_attn", 2)
    elif n_recent >= 1:
        assert (name, launches) == ("k_sched" if pref == "sched" else "k_fused", 1)
    else:
        assert (name, launches) == (f"k_{selector}_select+k_attn", 3)


def test_dense_bypass_policy(spg):
    """Quest's short-sequence rule: sparse pays only when the sequence has a
    few times more pages than the budget selects (crossover measured at
    about 2.5x on GB300)."""
    p = _valid(spg, max_pages_per_seq=4096, num_phys_pages=8192, token_budget=16 * 128)
    assert spg.spg_prefer_dense(p, 16 * 128)             # everything is selected anyway
    assert spg.spg_prefer_dense(p, 16 * 320)             # 320 pages <= 2.5 x 128
    assert not spg.spg_prefer_dense(p, 16 * 321)
    assert not spg.spg_prefer_dense(p, 32768)
    assert spg.spg_prefer_dense(p, 32768, ratio=20.0)    # a caller's own crossover
    assert not spg.spg_prefer_dense(_valid(spg, selector="all", token_budget=0, n_sink_pages=0,
                                           n_recent_pages=0), 16)
    assert not spg.spg_prefer_dense(_valid(spg, head_dim=48), 16)
