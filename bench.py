"""Decode-step benchmark of query-aware sparse-page attention on GB300.

One step = the whole hot path over one batch: page-metadata update for the
token just appended, page scoring, exact top-k, split-K sparse flash-decoding
and the log-sum-exp combine, on one "layer" of KV cache.  Layers rotate over
R independent cache replicas so that no step is served from L2 (the bytes a
step touches times R exceed four times the L2 size).

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the host cores instead, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synth import get_workload, make_inputs  # noqa: E402

METRIC = "decode attn steps/s and effective HBM GB/s (% of 8 TB/s) vs dense at 32K–128K"
DEFAULT_WORKLOAD = "llama2-7b-mha-32k"
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------- utils
# DRAM bytes (read + write) of one k_fused launch, from one ncu capture of
# that workload, and the sha256 of the kernel code it was taken on (see
# csrc_sha256; profiles/k_fused_<workload>.md).  Reported only while the code
# matches.
NCU_TRAFFIC = {
    "llama2-7b-mha-32k": (67_790_848, "acfacd6946311deefe4311f12a5b916eebf88add8f86c077f441e2e3b70e174a"),
    "long-scan-b4-128k": (205_888_768, "acfacd6946311deefe4311f12a5b916eebf88add8f86c077f441e2e3b70e174a"),
    "sals-int8-b16-10k-4x": (100_546_816, "acfacd6946311deefe4311f12a5b916eebf88add8f86c077f441e2e3b70e174a"),
}


def csrc_sha256(d: str | None = None) -> str:
    """sha256 over the kernel sources in d (the package's csrc/ by default;
    sorted by name; name, then the text with // and /* */ comments removed and
    whitespace runs collapsed): the code an ncu capture was taken on."""
    import hashlib
    import re

    if d is None:
        d = os.path.join(os.path.dirname(os.path.abspath(__file__)), "query_aware_sparse_page_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                code = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
            code = re.sub(r"//[^\n]*", "", code)
            code = " ".join(code.split())  # whitespace runs as one space
            h.update(f.encode())
            h.update(code.encode())
    return h.hexdigest()


def ncu_traffic(workload: str):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None:
        return None, "no ncu capture of this workload"
    if rec[1] != csrc_sha256():
        return None, "kernel sources changed since the ncu capture"
    return rec[0], f"profiles/k_fused_{workload}.md"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
        }


# ------------------------------------------------------------------- byte model
def step_bytes(w, lens, sel_tokens, cand_pages, sel_pages):
    """Algorithmic HBM bytes of one select + attend step (metadata of every
    scored page, K/V (+ scales) of every attended token, q, out + lse, page ids)."""
    kvb = 1 if w.kv_dtype == "i8" else 2
    scale = 2 if w.kv_dtype == "i8" else 0
    if w.selector == "quest":
        meta = cand_pages * 2 * w.head_dim * kvb
    else:
        meta = cand_pages * (w.page_size * w.sketch_dim // 2 + 4)
    kv = sel_tokens * 2 * (w.head_dim * kvb + scale)
    q = w.batch * w.num_q_heads * w.head_dim * 2
    out = w.batch * w.num_q_heads * (w.head_dim + 1) * 4
    return meta, kv, q + out + sel_pages * 8


def selection_stats(w, inp, sel, sel_cnt):
    """Attended tokens, scored candidate pages and selected pages, summed over units."""
    S = w.page_size
    lens = inp.seq_lens.cpu().tolist()
    cnt = sel_cnt.cpu().numpy()
    sel_h = sel.cpu().numpy()
    sel_tok = cand = sel_pages = 0
    for b, L in enumerate(lens):
        P = -(-L // S)
        lo = min(w.n_sink, P)
        hi = max(P - w.n_recent, lo)
        cand += (hi - lo) * w.num_kv_heads
        for h in range(w.num_kv_heads):
            n = int(cnt[b, h])
            sel_pages += n
            # every page is full except the sequence's last one
            last_in = n > 0 and int(sel_h[b, h, n - 1]) == P - 1
            sel_tok += n * S - (P * S - L if last_in else 0)
    return sel_tok, cand, sel_pages


# ----------------------------------------------------------------- our GPU arm
def max_over_ranks(value: float, world: int, device) -> float:
    """The slowest rank's value (the job finishes when its last rank does)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, world, rank, local):
    import torch.distributed as dist

    import query_aware_sparse_page_gb300 as spg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = get_workload(args.workload)
    R = args.layers
    layers = []
    for layer in range(R):
        inp = make_inputs(w, device=dev, seed_offset=1000 * rank + layer)
        p = spg.params_for(inp)
        bufs = spg.alloc_buffers(p, dev)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                    bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
        layers.append((inp, p, bufs))
    torch.cuda.synchronize()

    # the entry points of one step, per layer
    def op_meta(l):
        inp, p, b = layers[l]
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 0,
                                    b.minmax, b.sketch, b.sketch_scale, inp.proj, b.ws)

    def op_select_attend(l):
        inp, p, b = layers[l]
        spg.sparse_decode_select_attend(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                        inp.page_table, inp.seq_lens, b.minmax, b.sketch,
                                        b.sketch_scale, inp.proj, b.sel, b.sel_cnt, b.out, b.lse,
                                        b.ws)

    def op_step(l):  # the whole hot path, one call
        inp, p, b = layers[l]
        spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, b.minmax, b.sketch, b.sketch_scale,
                               inp.proj, b.sel, b.sel_cnt, b.out, b.lse, b.ws)

    def op_separate(l):  # the same step through the separate entry points
        op_meta(l)
        op_select(l)
        op_attn(l)

    def op_score(l):
        inp, p, b = layers[l]
        spg.sparse_page_score(p, inp.q, inp.page_table, inp.seq_lens, b.minmax, b.sketch,
                              b.sketch_scale, inp.proj, b.scores, b.ws)

    def op_select(l):
        inp, p, b = layers[l]
        spg.sparse_page_select(p, inp.q, inp.page_table, inp.seq_lens, b.minmax, b.sketch,
                               b.sketch_scale, inp.proj, b.sel, b.sel_cnt, b.ws)

    def op_attn(l):
        inp, p, b = layers[l]
        spg.sparse_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                    inp.page_table, inp.seq_lens, b.sel, b.sel_cnt, b.out, b.lse,
                                    b.ws)

    def op_dense(l):
        inp, p, b = layers[l]
        spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                   inp.page_table, inp.seq_lens, b.out, b.lse, b.ws)

    ops = {"step": op_step, "separate": op_separate, "meta": op_meta, "score": op_score,
           "select": op_select, "attn": op_attn, "dense": op_dense}
    for l in range(R):  # eager warm-up of every entry point (kernel attributes, caches)
        for f in ops.values():
            f(l)
    op_step(0)  # leave layer 0 with the step's own selection
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup

    # Each entry point is captured as one CUDA graph over the R layer
    # replicas in order (a decode pass over R layers, as an engine replays
    # it), plus a graph of the first K % R layers so that exactly K steps are
    # timed.  The step is also captured as one graph per layer, to report the
    # per-launch overhead of replaying single steps.
    def capture(f, layer_ids):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in layer_ids:
                f(l)
        return g

    graphs = {name: (capture(f, range(R)), capture(f, range(K % R)) if K % R else None)
              for name, f in ops.items()}
    single = [capture(op_step, [l]) for l in range(R)]
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def timed(fn, K):
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / K

    def timed_graph(name, K):
        # K steps: K // R replays of the R-layer graph, then the K % R graph
        full, part = graphs[name]
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K // R):
            full.replay()
        if part is not None:
            part.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, dev) / K

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(-(-W // R)):  # at least W warm-up steps
        graphs["step"][0].replay()
    t_end = time.perf_counter() + args.soak
    while time.perf_counter() < t_end:  # keep the GPU loaded while clocks are sampled
        graphs["step"][0].replay()
    ms_step = timed_graph("step", K)
    clock_info = clocks.stop()
    clock_info["window"] = "warm-up, soak and timed steps"

    # per-entry-point durations (K steps each, layers rotating)
    ms = {name: timed_graph(name, K)
          for name in ("separate", "meta", "score", "select", "attn", "dense")}
    ms_single = timed(lambda i: single[i % R].replay(), K)
    ms_topk = max(ms["select"] - ms["score"], 0.0)
    # the same step issued eagerly through the Python binding (host-issue bound)
    ms_eager = timed(lambda i: op_step(i % R), max(K // 4, 10))

    # bytes
    inp0, p0, b0 = layers[0]
    sel_tok, cand, sel_pages = selection_stats(w, inp0, b0.sel, b0.sel_cnt)
    meta_b, kv_b, small_b = step_bytes(w, None, sel_tok, cand, sel_pages)
    total_b = meta_b + kv_b + small_b
    lens = inp0.seq_lens.cpu().tolist()
    dense_tok = sum(lens) * w.num_kv_heads
    kvb = 1 if w.kv_dtype == "i8" else 2
    dense_b = dense_tok * 2 * (w.head_dim * kvb + (2 if w.kv_dtype == "i8" else 0)) + small_b
    peak, peak_kind = measured_peaks()

    # roofline of the dominant kernel: the step is one launch of the fused
    # kernel (k_fused), timed on its own as the whole step
    score_name = "k_quest_select" if w.selector == "quest" else "k_sketch_select"
    kname, dom_ms, dom_bytes = "k_fused", ms_step, total_b
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9 if dom_ms > 0 else 0.0

    traffic, traffic_src = ncu_traffic(w.name)
    e2e = run_e2e(args, spg, layers, stream, world, dev)
    launches_per_step = 1 if (w.selector == "quest" and w.max_pages_per_seq <= 8192) else 2

    steps_s = world * 1000.0 / ms_step
    gbs = world * total_b / (ms_step * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(steps_s, 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "kv_dtype": w.kv_dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload recipe)",
        "config": {
            "workload": w.name,
            "batch": w.batch, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "page_size": w.page_size, "seq_len": w.seq_len or list(w.seq_range),
            "token_budget": w.token_budget, "selector": w.selector,
            "layers_rotated": R,
            "l2": f"inputs larger than L2: {R} rotating cache replicas, each step reads "
                  f"{total_b / 1e6:.1f} MB of a distinct replica",
            "launch": f"CUDA graph of sparse_decode_step over the {R} layer replicas in order",
            "parallelism": "replicas" if world > 1 else "single",
        },
        "hbm_gbs_effective": round(gbs, 1),
        "hbm_frac_nominal": round(gbs / world / NOMINAL_HBM_GBS, 4),
        "hbm_frac_measured": round(gbs / world / peak, 4),
        "bytes_per_step": {"metadata": meta_b, "selected_kv": kv_b, "q_out_idx": small_b,
                           "total": total_b},
        "dense": {
            "steps_per_s": round(world * 1000.0 / ms["dense"], 2),
            "ms_per_step": round(ms["dense"], 5),
            "bytes_per_step": dense_b,
            "hbm_gbs": round(dense_b / (ms["dense"] * 1e-3) / 1e9, 1),
            "speedup_sparse_vs_dense": round(ms["dense"] / ms_step, 3),
        },
        "separate_entry_points": {
            "steps_per_s": round(world * 1000.0 / ms["separate"], 2),
            "ms_meta_append": round(ms["meta"], 5), "ms_" + score_name: round(ms["score"], 5),
            "ms_select_minus_score": round(ms_topk, 5), "ms_k_attn": round(ms["attn"], 5),
        },
        "eager_steps_per_s": round(world * 1000.0 / ms_eager, 2),
        "graph_per_step_steps_per_s": round(world * 1000.0 / ms_single, 2),
        "roofline": {
            "kernel": kname,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": peak_kind,
            "traffic": traffic,
            "traffic_source": traffic_src,
            "algorithmic_bytes": dom_bytes,
            "ms_per_launch": round(float(dom_ms), 5),
        },
        "clocks": clock_info,
        "e2e": e2e,
        "gpu_launches": K * launches_per_step,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, layers[0][0], budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)


def run_e2e(args, spg, layers, stream, world, dev):
    """Same step through the public API with host buffers: q and the appended
    token's K/V go host -> device each step, out and lse come back."""
    K = max(5, args.steps // 2)
    R = len(layers)
    hosts = []
    for inp, p, b in layers:
        w = inp.workload
        q_h = inp.q.cpu().pin_memory()
        lens = inp.seq_lens.cpu().tolist()
        kv_rows = []
        for bb, L in enumerate(lens):
            if L <= 0:
                continue
            t = L - 1
            phys = int(inp.page_table[bb, t // w.page_size])
            k_h = inp.k_pool[phys, :, t % w.page_size].cpu().pin_memory()
            v_h = inp.v_pool[phys, :, t % w.page_size].cpu().pin_memory()
            kv_rows.append((phys, t % w.page_size, k_h, v_h))
        out_h = torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory()
        lse_h = torch.empty(b.lse.shape, dtype=b.lse.dtype).pin_memory()
        hosts.append((q_h, kv_rows, out_h, lse_h))
    h2d = d2h = 0

    def e2e_step(i):
        nonlocal h2d, d2h
        inp, p, b = layers[i % R]
        q_h, kv_rows, out_h, lse_h = hosts[i % R]
        inp.q.copy_(q_h, non_blocking=True)
        h2d_i = q_h.numel() * q_h.element_size()
        for phys, slot, k_h, v_h in kv_rows:
            inp.k_pool[phys, :, slot].copy_(k_h, non_blocking=True)
            inp.v_pool[phys, :, slot].copy_(v_h, non_blocking=True)
            h2d_i += 2 * k_h.numel() * k_h.element_size()
        spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, b.minmax, b.sketch, b.sketch_scale,
                               inp.proj, b.sel, b.sel_cnt, b.out, b.lse, b.ws)
        out_h.copy_(b.out, non_blocking=True)
        lse_h.copy_(b.lse, non_blocking=True)
        stream.synchronize()  # the host reads the result every step
        h2d, d2h = h2d_i, out_h.numel() * 4 + lse_h.numel() * 4

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        e2e_step(i)
    dt = (time.perf_counter() - t0) / K
    return {"value": round(world / dt, 2), "unit": "steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K}


# ------------------------------------------------------------------ CPU oracle
def _oracle_unit_inputs(inp, b, h):
    from oracle import decode

    w = inp.workload
    S, G = w.page_size, w.group
    L = int(inp.seq_lens[b])
    P = -(-L // S)
    phys = inp.page_table[b, :P].long()

    def npy(t):
        if t is None:
            return None
        t = t[phys][:, h : h + 1].cpu()
        return (t.float() if t.dtype == torch.bfloat16 else t).numpy()

    q = inp.q[b : b + 1, h * G : (h + 1) * G].cpu()
    q = (q.float() if q.dtype == torch.bfloat16 else q).numpy()
    proj = None if inp.proj is None else inp.proj.cpu().numpy()
    return decode.StepInputs(q, npy(inp.k_pool), npy(inp.v_pool), npy(inp.k_scale), npy(inp.v_scale),
                             np.arange(max(P, 1))[None, :], np.array([L]), proj)


def cpu_baseline(w, inp, budget_s=12.0, max_units=None):
    """Time the oracle, as it stands, on whole steps (every (batch, kv-head)
    unit) of this workload, repeated until about `budget_s` seconds of CPU
    work are spent; `cores` is the process CPU time over the wall time."""
    from oracle import decode

    prm = decode.StepParams(w.page_size, w.n_sel_pages, w.n_sink, w.n_recent, w.selector, w.head_dim)
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    if max_units:
        units = units[:max_units]
    subs = [_oracle_unit_inputs(inp, b, h) for b, h in units]  # host copies, not timed
    done, wall, cpu = 0, 0.0, 0.0
    while wall < budget_s and done < 1000 * len(units):
        for sub in subs:
            t0, c0 = time.perf_counter(), time.process_time()
            decode.decode_step(sub, prm, units=[(0, 0)])
            wall += time.perf_counter() - t0
            cpu += time.process_time() - c0
            done += 1
            if wall >= budget_s:
                break
    steps = done / len(units)
    cores = max(1, round(cpu / wall)) if wall > 0 else 1
    return {"value": round(steps / wall, 6), "unit": "steps/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} (batch, kv-head) units = {steps:.2f} steps of {w.name} "
                      f"({len(units)} units per step), {wall:.1f} s wall / {cpu:.1f} s CPU of "
                      f"fp64 numpy on the host"}


def run_reference(args, world, rank, local):
    """The oracle as the reference arm: rank 0 only, host cores."""
    if rank != 0:
        return
    w = get_workload(args.workload)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(w, device=dev)
    K, W = args.steps, args.warmup
    per_step = max(0.2, min(1.0, 120.0 / max(K + W, 1)))
    n_units = w.batch * w.num_kv_heads
    from oracle import decode

    prm = decode.StepParams(w.page_size, w.n_sel_pages, w.n_sink, w.n_recent, w.selector, w.head_dim)
    subs = {}

    def one_step(i):
        # a bounded sample of the step: as many units as fit in the per-step budget
        t0, c0 = time.perf_counter(), time.process_time()
        done = 0
        while done < n_units:
            u = (i * 7 + done) % n_units
            b, h = divmod(u, w.num_kv_heads)
            if (b, h) not in subs:
                subs[(b, h)] = _oracle_unit_inputs(inp, b, h)
            decode.decode_step(subs[(b, h)], prm, units=[(0, 0)])
            done += 1
            if time.perf_counter() - t0 >= per_step:
                break
        wall = time.perf_counter() - t0
        return wall * n_units / done, done, wall, time.process_time() - c0

    for i in range(W):
        one_step(i)
    times, units, wall_s, cpu_s = [], 0, 0.0, 0.0
    for i in range(K):
        t, d, wl, cp = one_step(i)
        times.append(t)
        units += d
        wall_s += wl
        cpu_s += cp
    cores = max(1, round(cpu_s / wall_s)) if wall_s > 0 else 1
    step_s = float(np.mean(times))
    val = 1.0 / step_s
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 6),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(step_s * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the workload recipe)",
        "config": {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "page_size": w.page_size, "seq_len": w.seq_len or list(w.seq_range),
                   "token_budget": w.token_budget, "selector": w.selector},
        "cpu_baseline": {"value": round(val, 6), "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": f"{units} (batch, kv-head) units over {K} timed steps of "
                                   f"{n_units}; each step scaled from its sampled units"},
        "e2e": {"value": round(val, 6), "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--soak", type=float, default=0.5, help="seconds of untimed steps before timing")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, local)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
