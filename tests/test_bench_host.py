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
