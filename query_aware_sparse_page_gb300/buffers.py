"""Device buffers of the layouts include/spg.h documents, allocated with torch.

Allocation only: nothing here computes any part of the decode step.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from .binding import I8, SEL_QUEST, SEL_SKETCH_INT4, make_params, spg_workspace_size

_TORCH_KV = {0: torch.float16, 1: torch.bfloat16, 2: torch.int8}


@dataclass
class DecodeBuffers:
    minmax: torch.Tensor | None  # [B][Hkv][MP][2][d]      (Quest, logical pages)
    sketch: torch.Tensor | None  # [B][Hkv][MP][S][ds/2]   (sketch, logical blocks)
    sketch_scale: torch.Tensor | None  # [B][Hkv][MP]
    scores: torch.Tensor  # [B][Hkv][MP]
    sel: torch.Tensor  # [B][Hkv][n_sel]
    sel_cnt: torch.Tensor  # [B][Hkv]
    out: torch.Tensor  # [B][Hq][d]
    lse: torch.Tensor  # [B][Hq]
    ws: torch.Tensor  # workspace bytes, zero-filled


def alloc_buffers(p, device="cuda") -> DecodeBuffers:
    dev = torch.device(device)
    B, Hq, Hkv, d = p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim
    NP, S, MP = p.num_phys_pages, p.page_size, p.max_pages_per_seq
    n_sel = max(p.token_budget // S, 1)
    minmax = sketch = sketch_scale = None
    if p.selector == SEL_QUEST:
        # int8 pools keep their Quest metadata in the query's 16-bit type
        mdt = _TORCH_KV[p.q_dtype] if p.kv_dtype == I8 else _TORCH_KV[p.kv_dtype]
        minmax = torch.zeros((B, Hkv, MP, 2, d), dtype=mdt, device=dev)
    elif p.selector == SEL_SKETCH_INT4:
        sketch = torch.zeros((B, Hkv, MP, S, p.sketch_dim // 2), dtype=torch.uint8, device=dev)
        sketch_scale = torch.zeros((B, Hkv, MP), dtype=torch.float32, device=dev)
    ws = torch.zeros(spg_workspace_size(p), dtype=torch.uint8, device=dev)
    return DecodeBuffers(
        minmax=minmax, sketch=sketch, sketch_scale=sketch_scale,
        scores=torch.empty((B, Hkv, MP), dtype=torch.float32, device=dev),
        sel=torch.empty((B, Hkv, n_sel), dtype=torch.int32, device=dev),
        sel_cnt=torch.empty((B, Hkv), dtype=torch.int32, device=dev),
        out=torch.empty((B, Hq, d), dtype=torch.float32, device=dev),
        lse=torch.empty((B, Hq), dtype=torch.float32, device=dev),
        ws=ws,
    )


def params_for(inputs, selector=None, n_sel_pages=None):
    """spg_params for a set of inputs (any object with the attributes of a
    seeded decode-step input: workload, num_phys_pages, page_table)."""
    w = inputs.workload
    sel = selector or w.selector
    n_sel = w.n_sel_pages if n_sel_pages is None else n_sel_pages
    return make_params(
        batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim=w.head_dim, page_size=w.page_size, num_phys_pages=inputs.num_phys_pages,
        max_pages_per_seq=int(inputs.page_table.shape[1]), kv_dtype=w.kv_dtype,
        q_dtype=w.q_dtype, selector=sel, token_budget=n_sel * w.page_size,
        n_sink_pages=w.n_sink, n_recent_pages=w.n_recent, sketch_dim=w.sketch_dim,
    )
