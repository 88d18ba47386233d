"""Seeded tensor generation for one decode step of a workload.

Recipe (every draw comes from one ``torch.Generator`` seeded with the
workload seed, on the device the tensors are made on):

* sequence lengths: fixed, or uniform integers in the workload's range;
* page table: sequence ``b`` owns ``P_b = ceil(L_b / S)`` physical pages,
  contiguous in batch order, or a seeded random permutation of the whole
  pool when the workload asks for a non-contiguous table; entries past
  ``P_b`` are -1;
* q ~ N(0, 1) in the query dtype;
* K, V ~ N(0, 1), times a per-(kv-head, channel) LogNormal(0, 0.5) factor
  (drawn separately for K and V) when the workload asks for channel scales;
* int8 K/V: drawn in fp32 as above, then per (token, kv-head) an fp16
  scale = absmax / 127 and codes = rint(x / scale) clipped to [-127, 127];
* needles: per (batch, kv-head), positions drawn without replacement among
  the tokens of pages [n_sink, P_b - n_recent); the key there is replaced
  by 4 * sqrt(d) * u / |u| with u the mean of the group's query rows;
  V is left as drawn;
* token slots past L_b in a sequence's last page hold a large poison value
  (K = V = 60, or int8 codes 127 with scale 8) so that any read of them
  shows up in the results;
* sketch projection P (d x d_s, fp32) ~ N(0, 1/d_s), drawn last.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from .workloads import Workload

_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}

POISON = 60.0


@dataclass
class DecodeInputs:
    workload: Workload
    seq_lens: torch.Tensor  # [B] int32
    page_table: torch.Tensor  # [B][max_pages] int32
    num_phys_pages: int
    q: torch.Tensor  # [B][Hq][d]
    k_pool: torch.Tensor  # [P_phys][Hkv][S][d]
    v_pool: torch.Tensor
    k_scale: torch.Tensor | None  # [P_phys][Hkv][S] fp16, int8 pools only
    v_scale: torch.Tensor | None
    proj: torch.Tensor | None  # [d][d_s] fp32, sketch selector only
    needles: dict = field(default_factory=dict)  # (b, h) -> sorted token positions

    def to(self, device) -> "DecodeInputs":
        def mv(t):
            return None if t is None else t.to(device)

        return DecodeInputs(
            self.workload, mv(self.seq_lens), mv(self.page_table), self.num_phys_pages,
            mv(self.q), mv(self.k_pool), mv(self.v_pool), mv(self.k_scale), mv(self.v_scale),
            mv(self.proj), dict(self.needles),
        )


def _seq_lens(w: Workload, g: torch.Generator, device) -> torch.Tensor:
    if w.seq_len is not None:
        return torch.full((w.batch,), w.seq_len, dtype=torch.int32, device=device)
    lo, hi = w.seq_range
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def make_inputs(w: Workload, device="cpu", seed_offset: int = 0, seq_lens=None) -> DecodeInputs:
    """Draw one decode step's inputs for workload ``w`` on ``device``.

    ``seq_lens`` (a list of ints) overrides the workload's lengths, for edge
    cases such as empty or one-token sequences.
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * (w.seed + 1) + seed_offset)

    B, Hq, Hkv, d, S = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    G = Hq // Hkv
    if seq_lens is None:
        lens = _seq_lens(w, g, device)
    else:
        lens = torch.tensor(list(seq_lens), dtype=torch.int32, device=device)
    lens_h = [int(x) for x in lens.cpu()]
    max_pages = max(w.max_pages_per_seq, max([math.ceil(L / S) for L in lens_h] + [1]))
    pages = [math.ceil(L / S) for L in lens_h]
    n_phys = max(sum(pages), 1)

    if w.random_page_table:
        perm = torch.randperm(n_phys, generator=g, device=device).to(torch.int32)
    else:
        perm = torch.arange(n_phys, dtype=torch.int32, device=device)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32, device=device)
    off = 0
    for b in range(B):
        if pages[b]:
            pt[b, : pages[b]] = perm[off : off + pages[b]]
        off += pages[b]

    qf = torch.randn((B, Hq, d), generator=g, device=device, dtype=torch.float32)
    q = qf.to(_DT[w.q_dtype])

    def pool(chan: bool):
        x = torch.randn((n_phys, Hkv, S, d), generator=g, device=device, dtype=torch.float32)
        if chan:
            c = torch.exp(0.5 * torch.randn((Hkv, d), generator=g, device=device, dtype=torch.float32))
            x.mul_(c.view(1, Hkv, 1, d))
        return x

    kf = pool(w.channel_scales)
    vf = pool(w.channel_scales)

    # needles: keys aligned with the group-mean query
    needles = {}
    if w.needles_per_head > 0:
        qd = q.to(torch.float64)
        for b in range(B):
            P = pages[b]
            lo_tok = w.n_sink * S
            hi_tok = min((P - w.n_recent) * S, lens_h[b])
            n_avail = hi_tok - lo_tok
            if n_avail <= 0:
                continue
            for h in range(Hkv):
                u = qd[b, h * G : (h + 1) * G].mean(dim=0)
                kn = (4.0 * math.sqrt(d) * u / torch.linalg.vector_norm(u)).to(torch.float32)
                n = min(w.needles_per_head, n_avail)
                pos = torch.randperm(n_avail, generator=g, device=device)[:n] + lo_tok
                pos_sorted = sorted(int(t) for t in pos.cpu())
                needles[(b, h)] = pos_sorted
                pos_t = torch.tensor(pos_sorted, dtype=torch.int64, device=device)
                phys = pt[b].to(torch.int64)[pos_t // S]
                kf[phys, h, pos_t % S] = kn

    # poison the unused slots of each last page
    for b in range(B):
        L = lens_h[b]
        if L % S:
            phys = int(pt[b, L // S])
            kf[phys, :, L % S :] = POISON
            vf[phys, :, L % S :] = POISON

    k_scale = v_scale = None
    if w.kv_dtype == "i8":
        def quant(x):
            amax = x.abs().amax(dim=-1)
            s16 = (amax / 127.0).to(torch.float16)
            s16 = torch.where(s16 > 0, s16, torch.ones_like(s16))
            codes = torch.clamp(torch.round(x / s16.to(torch.float32).unsqueeze(-1)), -127, 127)
            return codes.to(torch.int8), s16

        k_pool, k_scale = quant(kf)
        v_pool, v_scale = quant(vf)
        # poison for int8: full-scale codes with a large scale
        for b in range(B):
            L = lens_h[b]
            if L % S:
                phys = int(pt[b, L // S])
                for t8, s8 in ((k_pool, k_scale), (v_pool, v_scale)):
                    t8[phys, :, L % S :] = 127
                    s8[phys, :, L % S :] = 8.0
    else:
        k_pool = kf.to(_DT[w.kv_dtype])
        v_pool = vf.to(_DT[w.kv_dtype])
    del kf, vf

    proj = None
    if w.selector == "sketch":
        proj = torch.randn((d, w.sketch_dim), generator=g, device=device, dtype=torch.float32)
        proj.mul_(1.0 / math.sqrt(w.sketch_dim))

    return DecodeInputs(w, lens, pt, n_phys, q, k_pool, v_pool, k_scale, v_scale, proj, needles)
