"""The five decode workloads, by name, with their shapes and input recipes.

Sizes follow the problem statement of the pages (Llama-2-7B-shaped MHA at
32K, a GQA 32/8 serving batch with ragged lengths, the SALS int8 path at
10K with 64-token blocks, a 128K long-context scan, and a tiny GQA-4 check).
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    # seq_len: fixed length for every sequence, or None when seq_range is used
    seq_len: int | None
    seq_range: tuple[int, int] | None  # inclusive uniform range per sequence
    kv_dtype: str  # "f16" | "bf16" | "i8"
    q_dtype: str  # "f16" | "bf16"
    selector: str  # "quest" | "sketch"
    n_sel_pages: int  # pages attended per (batch, kv-head), forced pages included
    n_sink: int
    n_recent: int
    channel_scales: bool  # K and V multiplied by LogNormal(0, 0.5) per (kv-head, channel)
    needles_per_head: int  # planted needle keys per (batch, kv-head)
    random_page_table: bool  # seeded permutation of the physical pool
    sketch_dim: int = 16
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def token_budget(self) -> int:
        return self.n_sel_pages * self.page_size

    @property
    def max_seq_len(self) -> int:
        return self.seq_len if self.seq_len is not None else self.seq_range[1]

    @property
    def max_pages_per_seq(self) -> int:
        return math.ceil(self.max_seq_len / self.page_size)


def _sals_n_sel(n_blocks: int, sparsity: int) -> int:
    # top-k = ceil(candidate blocks / sparsity) over the 160 blocks of a 10K
    # sequence, plus the fixed tail block.
    return math.ceil(n_blocks / sparsity) + 1


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload(
            name="tiny-quest-gqa4-1k",
            batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
            seq_len=1024, seq_range=None, kv_dtype="f16", q_dtype="f16", selector="quest",
            n_sel_pages=10, n_sink=1, n_recent=1, channel_scales=False,
            needles_per_head=3, random_page_table=False, seed=0,
        ),
        Workload(
            name="llama2-7b-mha-32k",
            batch=1, num_q_heads=32, num_kv_heads=32, head_dim=128, page_size=16,
            seq_len=32768, seq_range=None, kv_dtype="f16", q_dtype="f16", selector="quest",
            n_sel_pages=128, n_sink=1, n_recent=1, channel_scales=True,
            needles_per_head=16, random_page_table=False, seed=1,
        ),
        Workload(
            name="gqa-serving-b8-4k-64k",
            batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
            seq_len=None, seq_range=(4096, 65536), kv_dtype="bf16", q_dtype="bf16",
            selector="quest", n_sel_pages=256, n_sink=1, n_recent=2, channel_scales=True,
            needles_per_head=0, random_page_table=True, seed=2,
        ),
        Workload(
            name="sals-int8-b16-10k-4x",
            batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64,
            seq_len=10240, seq_range=None, kv_dtype="i8", q_dtype="f16", selector="sketch",
            n_sel_pages=_sals_n_sel(159, 4), n_sink=0, n_recent=1, channel_scales=False,
            needles_per_head=0, random_page_table=False, seed=3,
        ),
        Workload(
            name="sals-int8-b16-10k-6x",
            batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64,
            seq_len=10240, seq_range=None, kv_dtype="i8", q_dtype="f16", selector="sketch",
            n_sel_pages=_sals_n_sel(159, 6), n_sink=0, n_recent=1, channel_scales=False,
            needles_per_head=0, random_page_table=False, seed=3,
        ),
        Workload(
            name="long-scan-b4-128k",
            batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
            seq_len=131072, seq_range=None, kv_dtype="bf16", q_dtype="bf16", selector="quest",
            n_sel_pages=256, n_sink=1, n_recent=1, channel_scales=False,
            needles_per_head=64, random_page_table=False, seed=4,
        ),
    ]
}


def get_workload(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def scaled(w: Workload, **changes) -> Workload:
    """A reduced copy of a workload (same recipe, smaller sizes) for tests."""
    return dataclasses.replace(w, **changes)
