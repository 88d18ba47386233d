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
    # workload: (DRAM bytes of one launch, code hash, kernel)
    "llama2-7b-mha-32k": (67_890_432, "ebd83aa240f926a217a97b62897c56d90e8d4000d7273d0df5caa2a35bec27ee", "k_fused"),
    "long-scan-b4-128k": (205_280_000, "ebd83aa240f926a217a97b62897c56d90e8d4000d7273d0df5caa2a35bec27ee", "k_fused"),
    "sals-int8-b16-10k-4x": (100_827_136, "ebd83aa240f926a217a97b62897c56d90e8d4000d7273d0df5caa2a35bec27ee", "k_fused"),
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


def ncu_traffic(workload: str, kernel: str = "k_fused"):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None or rec[2] != kernel:
        return None, f"no ncu capture of {kernel} on this workload"
    if rec[1] != csrc_sha256():
        return None, "kernel sources changed since the ncu capture"
    return rec[0], f"profiles/{kernel}_{workload}.md"


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


PER_WORKLOADS = ["long-scan-b4-128k", "gqa-serving-b8-4k-64k", "sals-int8-b16-10k-4x",
                 "sals-int8-b16-10k-6x", "llama2-7b-mha-32k"]


def build_layers(spg, w, R, dev, rank):
    """R independent cache replicas ("layers") of workload w, metadata built."""
    layers = []
    for layer in range(R):
        inp = make_inputs(w, device=dev, seed_offset=1000 * rank + layer)
        p = spg.params_for(inp)
        bufs = spg.alloc_buffers(p, dev)
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 1,
                                    bufs.minmax, bufs.sketch, bufs.sketch_scale, inp.proj, bufs.ws)
        layers.append((inp, p, bufs))
    torch.cuda.synchronize()
    return layers


def entry_points(spg, layers):
    """The entry points of one step, each as a function of the layer index."""

    def op_meta(l):
        inp, p, b = layers[l]
        spg.sparse_page_meta_update(p, inp.k_pool, inp.k_scale, inp.page_table, inp.seq_lens, 0,
                                    b.minmax, b.sketch, b.sketch_scale, inp.proj, b.ws)

    def op_step(l):  # the whole hot path, one call
        inp, p, b = layers[l]
        spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, b.minmax, b.sketch, b.sketch_scale,
                               inp.proj, b.sel, b.sel_cnt, b.out, b.lse, b.ws)

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

    def op_separate(l):  # the same step through the separate entry points
        op_meta(l)
        op_select(l)
        op_attn(l)

    def op_dense(l):
        inp, p, b = layers[l]
        spg.dense_decode_attention(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                                   inp.page_table, inp.seq_lens, b.out, b.lse, b.ws)

    return {"step": op_step, "separate": op_separate, "meta": op_meta, "score": op_score,
            "select": op_select, "attn": op_attn, "dense": op_dense}


class Timer:
    """CUDA-event timing of K steps on the launching stream, bracketed by a
    barrier and a device synchronise; max over ranks."""

    def __init__(self, stream, world, dev):
        self.stream, self.world, self.dev = stream, world, dev

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.barrier()

    def region(self, fn, K):
        self.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        fn(K)
        e1.record(self.stream)
        torch.cuda.synchronize()
        self.barrier()
        return max_over_ranks(e0.elapsed_time(e1), self.world, self.dev) / K


def graph_runner(ops, names, R, K):
    """Each entry point captured as one CUDA graph over the R layer replicas
    in order (a decode pass over R layers, as an engine replays it), plus a
    graph of the first K % R layers, so that exactly K steps run."""

    def capture(f, layer_ids):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in layer_ids:
                f(l)
        return g

    graphs = {name: (capture(ops[name], range(R)), capture(ops[name], range(K % R)) if K % R else None)
              for name in names}

    def run(name):
        full, part = graphs[name]

        def go(K_):
            for _ in range(K_ // R):
                full.replay()
            if part is not None:
                part.replay()

        return go

    return graphs, run


def layer_bytes(w, layers):
    """Algorithmic bytes of one step, and of the dense read, as the mean over
    the layer replicas the timed regions cycle through (replicas of a ragged
    batch draw different lengths; each replica's own selection is counted)."""
    kvb = 1 if w.kv_dtype == "i8" else 2
    tot = [0, 0, 0, 0]
    for inp, _, bufs in layers:
        sel_tok, cand, sel_pages = selection_stats(w, inp, bufs.sel, bufs.sel_cnt)
        meta_b, kv_b, small_b = step_bytes(w, None, sel_tok, cand, sel_pages)
        lens = inp.seq_lens.cpu().tolist()
        dense_b = sum(lens) * w.num_kv_heads * 2 * (w.head_dim * kvb + (2 if w.kv_dtype == "i8" else 0)) + small_b
        for i, x in enumerate((meta_b, kv_b, small_b, dense_b)):
            tot[i] += x
    n = len(layers)
    return tuple(x // n for x in tot)


def median_spread(xs):
    return statistics.median(xs), min(xs), max(xs)


def measure_workload(spg, name, args, timer, rank, dev):
    """Step (repeated timed regions), single-step replays and the dense
    baseline on one workload; a smaller record than the headline's."""
    w = get_workload(name)
    R, K = args.layers, args.steps
    layers = build_layers(spg, w, R, dev, rank)
    ops = entry_points(spg, layers)
    for l in range(R):
        ops["step"](l)
        ops["dense"](l)
    ops["step"](0)
    torch.cuda.synchronize()
    graphs, run = graph_runner(ops, ["step", "dense"], R, K)
    single = [torch.cuda.CUDAGraph() for _ in range(R)]
    for l, g in enumerate(single):
        with torch.cuda.graph(g):
            ops["step"](l)
    for _ in range(max(3, -(-args.warmup // R))):
        run("step")(R)
    reps = [timer.region(run("step"), K) for _ in range(args.repeats)]
    ms_dense = timer.region(run("dense"), K)
    ms_single = timer.region(lambda K_: [single[i % R].replay() for i in range(K_)], K)
    ms, lo, hi = median_spread(reps)
    meta_b, kv_b, small_b, dense_b = layer_bytes(w, layers)
    total = meta_b + kv_b + small_b
    peak, _ = measured_peaks()
    res = {
        "ms_per_step": round(ms, 5), "ms_min": round(lo, 5), "ms_max": round(hi, 5),
        "repeats": args.repeats, "steps_per_repeat": K,
        "steps_per_s": round(1000.0 / ms, 2),
        "bytes_per_step": total,
        "hbm_gbs": round(total / (ms * 1e-3) / 1e9, 1),
        "frac_measured": round(total / (ms * 1e-3) / 1e9 / peak, 4),
        "single_step_ms": round(ms_single, 5),
        "single_step_frac_measured": round(total / (ms_single * 1e-3) / 1e9 / peak, 4),
        "dense_ms": round(ms_dense, 5),
        "dense_hbm_gbs": round(dense_b / (ms_dense * 1e-3) / 1e9, 1),
        "speedup_vs_dense": round(ms_dense / ms, 3),
        "kernel": spg.step_kernel_name(layers[0][1]),
    }
    del graphs, single, ops, layers
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    import query_aware_sparse_page_gb300 as spg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = get_workload(args.workload)
    R, K, W = args.layers, args.steps, args.warmup
    layers = build_layers(spg, w, R, dev, rank)
    ops = entry_points(spg, layers)
    for l in range(R):  # eager warm-up of every entry point (kernel attributes, caches)
        for f in ops.values():
            f(l)
    ops["step"](0)  # leave layer 0 with the step's own selection
    torch.cuda.synchronize()

    graphs, run = graph_runner(ops, list(ops), R, K)
    # the step also as one graph per layer: a step replayed alone, the rate a
    # model sees when each layer's query depends on the previous layer's output
    single = []
    for l in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ops["step"](l)
        single.append(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    timer = Timer(stream, world, dev)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(max(3, -(-W // R))):  # at least W warm-up steps
        run("step")(R)
    t_end = time.perf_counter() + args.soak
    while time.perf_counter() < t_end:  # keep the GPU loaded while clocks are sampled
        run("step")(R)
    reps = [timer.region(run("step"), K) for _ in range(args.repeats)]
    clock_info = clocks.stop()
    clock_info["window"] = "warm-up, soak and timed steps"
    ms_step, ms_lo, ms_hi = median_spread(reps)

    # per-entry-point durations (K steps each, layers rotating)
    ms = {name: timer.region(run(name), K)
          for name in ("separate", "meta", "score", "select", "attn", "dense")}
    ms_single = timer.region(lambda K_: [single[i % R].replay() for i in range(K_)], K)
    ms_topk = max(ms["select"] - ms["score"], 0.0)
    # the same step issued eagerly through the Python binding (host-issue bound)
    ms_eager = timer.region(lambda K_: [ops["step"](i % R) for i in range(K_)], max(K // 4, 10))

    meta_b, kv_b, small_b, dense_b = layer_bytes(w, layers)
    total_b = meta_b + kv_b + small_b
    peak, peak_kind = measured_peaks()
    # the other single-launch step kernel on the same replicas (the library
    # picks the faster one by default; both compute the same step)
    alt = {}
    p0 = layers[0][1]
    default_kernel = spg.step_kernel_name(p0)
    for code in (spg.STEP_KERNEL_CLUSTER, spg.STEP_KERNEL_SCHED):
        spg.spg_set_step_kernel(code)
        name = spg.step_kernel_name(p0)
        if name == default_kernel or name is None:
            continue
        g_alt, run_alt = graph_runner(ops, ["step"], R, K)
        run_alt("step")(R)
        ms_alt = statistics.median(timer.region(run_alt("step"), K) for _ in range(3))
        alt[name] = {"ms_per_step": round(ms_alt, 5), "steps_per_s": round(1000.0 / ms_alt, 2),
                     "frac_measured": round(total_b / (ms_alt * 1e-3) / 1e9 / peak, 4)}
        del g_alt
    spg.spg_set_step_kernel(spg.STEP_KERNEL_AUTO)
    score_name = "k_quest_select" if w.selector == "quest" else "k_sketch_select"
    # the step is one launch of the persistent kernel, timed as the whole step
    kname = spg.step_kernel_name(layers[0][1])
    achieved = total_b / (ms_step * 1e-3) / 1e9 if ms_step > 0 else 0.0
    traffic, traffic_src = ncu_traffic(w.name, kname)
    e2e = run_e2e(args, spg, layers, stream, world, dev)
    launches_per_step = spg.step_launch_count(layers[0][1])

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
            "timing": f"median of {args.repeats} timed regions of exactly {K} steps each",
            "parallelism": "replicas" if world > 1 else "single",
        },
        "repeats_ms_per_step": [round(x, 5) for x in reps],
        "ms_per_step_min": round(ms_lo, 5),
        "ms_per_step_max": round(ms_hi, 5),
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
        "graph_per_step_frac_measured": round(total_b / (ms_single * 1e-3) / 1e9 / peak, 4),
        "other_step_kernels": alt,
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
            "algorithmic_bytes": total_b,
            "ms_per_launch": round(float(ms_step), 5),
        },
        "clocks": clock_info,
        "e2e": e2e,
        "gpu_launches": K * launches_per_step,
    }
    del graphs, single, ops
    if not args.no_per_workload:
        layers = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        res["per_workload"] = {n: measure_workload(spg, n, args, timer, rank, dev)
                               for n in PER_WORKLOADS if n != w.name}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp0 = make_inputs(w, device=dev, seed_offset=1000 * rank)
        res["cpu_baseline"] = cpu_baseline(w, inp0, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)


def pool_rows(phys, slot, n_kv_heads, page_size):
    """Rows of (page phys[i], every kv-head, slot slot[i]) in a pool
    [pages][Hkv][S][...] seen as [pages * Hkv * S][...], sequence-major then
    head: the order of pool[phys, :, slot] flattened over its first two dims."""
    heads = torch.arange(n_kv_heads, dtype=torch.long, device=phys.device)
    return ((phys[:, None] * n_kv_heads + heads[None, :]) * page_size + slot[:, None]).reshape(-1)


def run_e2e(args, spg, layers, stream, world, dev):
    """Same step through the public API with host buffers.  Every step one
    host -> device copy brings q and the appended token's K and V rows of
    every sequence (with their int8 scales), packed in one pinned buffer; the
    rows are written into the pools on the device, q is read where it landed;
    one device -> host copy brings out and lse back (one device buffer holds
    both).  The host synchronises on the stream every step."""
    K = max(5, args.steps // 2)
    R = len(layers)

    def seg(n):  # 16-byte aligned segments of the staging buffers
        return (n + 15) & ~15

    plans = []
    for inp, p, b in layers:
        S = inp.workload.page_size
        lens = inp.seq_lens.cpu().tolist()
        rows = [(int(inp.page_table[bb, (L - 1) // S]), (L - 1) % S) for bb, L in enumerate(lens) if L > 0]
        phys = torch.tensor([r[0] for r in rows], dtype=torch.long, device=dev)
        slot = torch.tensor([r[1] for r in rows], dtype=torch.long, device=dev)
        rows_idx = pool_rows(phys, slot, inp.workload.num_kv_heads, S)
        # what the host sends: q, then K, V (and their scales) of the new tokens
        parts = [inp.q]
        dsts = []
        for pool in (inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale):
            if pool is not None:
                parts.append(pool[phys, :, slot].contiguous())
                dsts.append(pool.view(-1, pool.shape[-1]) if pool.dim() == 4 else pool.view(-1))
        offs, n = [], 0
        for t in parts:
            offs.append(n)
            n += seg(t.numel() * t.element_size())
        stage_h = torch.zeros(n, dtype=torch.uint8).pin_memory()
        for t, o in zip(parts, offs):
            nb = t.numel() * t.element_size()
            stage_h[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
        stage_d = torch.empty(n, dtype=torch.uint8, device=dev)
        views = [stage_d[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for t, o in zip(parts, offs)]
        srcs = [v.reshape(-1, v.shape[-1]) if v.dim() == 3 else v.reshape(-1) for v in views[1:]]
        n_out = b.out.numel()
        res_d = torch.empty(n_out + seg(b.lse.numel() * 4) // 4, dtype=torch.float32, device=dev)
        out_d = res_d[:n_out].view(b.out.shape)
        lse_d = res_d[n_out:n_out + b.lse.numel()].view(b.lse.shape)
        res_h = torch.empty(res_d.numel(), dtype=torch.float32).pin_memory()
        plans.append((rows_idx, srcs, dsts, views, stage_h, stage_d, out_d, lse_d, res_d, res_h))

    def e2e_step(i):
        inp, p, b = layers[i % R]
        rows_idx, srcs, dsts, views, stage_h, stage_d, out_d, lse_d, res_d, res_h = plans[i % R]
        stage_d.copy_(stage_h, non_blocking=True)
        for dst, src in zip(dsts, srcs):
            dst.index_copy_(0, rows_idx, src)
        spg.sparse_decode_step(p, views[0], inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, b.minmax, b.sketch, b.sketch_scale,
                               inp.proj, b.sel, b.sel_cnt, out_d, lse_d, b.ws)
        res_h.copy_(res_d, non_blocking=True)
        stream.synchronize()  # the host reads the result every step

    # the staged step is the plain step: same inputs, same results (reported)
    same = True
    for i in range(R):
        inp, p, b = layers[i]
        spg.sparse_decode_step(p, inp.q, inp.k_pool, inp.v_pool, inp.k_scale, inp.v_scale,
                               inp.page_table, inp.seq_lens, b.minmax, b.sketch, b.sketch_scale,
                               inp.proj, b.sel, b.sel_cnt, b.out, b.lse, b.ws)
        e2e_step(i)
        out_d, lse_d = plans[i][6], plans[i][7]
        same = same and torch.equal(out_d, b.out) and torch.equal(lse_d, b.lse)
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        e2e_step(i)
    dt = (time.perf_counter() - t0) / K
    return {"value": round(world / dt, 2), "unit": "steps/s",
            "h2d_bytes_per_step": int(plans[0][4].numel()), "d2h_bytes_per_step": int(plans[0][9].numel() * 4),
            "steps": K, "equals_plain_step": bool(same)}


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


def cpu_baseline_single(w, inp, budget_s=12.0, max_units=None):
    """Time the oracle, as it stands, on whole steps (every (batch, kv-head)
    unit) of this workload in this process, repeated until about `budget_s`
    seconds of CPU work are spent; `cores` is the process CPU time over the
    wall time."""
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
                      f"fp64 numpy in one process"}


def cpu_baseline_parallel(w, inp, budget_s=12.0):
    """The oracle on every host core at once: one process per core (started
    with python -m oracle.run_units, no torch in them, one BLAS thread each),
    each running its share of the step's (batch, kv-head) units round-robin
    for `budget_s` seconds; steps/s = the sum of the processes' unit rates
    over the units of a step."""
    import tempfile

    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    n_cores = os.cpu_count() or 1
    n_proc = max(1, min(n_cores, len(units)))
    sel_id = {"quest": 0, "sketch": 1, "all": 2}[w.selector]
    arrays = {"params": np.array([w.page_size, w.n_sel_pages, w.n_sink, w.n_recent, w.head_dim,
                                  sel_id, len(units)], dtype=np.int64)}
    for i, (b, h) in enumerate(units):
        sub = _oracle_unit_inputs(inp, b, h)
        for k, v in (("q", sub.q), ("k", sub.k_pool), ("v", sub.v_pool), ("ks", sub.k_scale),
                     ("vs", sub.v_scale), ("pt", sub.page_table), ("lens", sub.seq_lens),
                     ("proj", sub.proj)):
            if v is not None:
                arrays[f"u{i}_{k}"] = v
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "units.npz")
        np.savez(path, **arrays)
        procs = [subprocess.Popen([sys.executable, "-m", "oracle.run_units", path, str(i), str(n_proc),
                                   str(budget_s)], cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                  stderr=subprocess.PIPE, text=True)
                 for i in range(n_proc)]
        outs = [p.communicate(timeout=budget_s + 300) for p in procs]
    recs = []
    for (o, e), p in zip(outs, procs):
        if p.returncode != 0:
            return {"error": f"oracle worker failed: {e.strip()[-300:]}"}
        recs.append(json.loads(o.strip().splitlines()[-1]))
    unit_rate = sum(r["units"] / r["wall"] for r in recs if r["wall"] > 0)
    done = sum(r["units"] for r in recs)
    cpu = sum(r["cpu"] for r in recs)
    return {"value": round(unit_rate / len(units), 6), "unit": "steps/s", "cores": n_proc,
            "kind": "oracle", "host_cores": n_cores,
            "sample": f"{done} (batch, kv-head) units of {w.name} ({len(units)} per step) on "
                      f"{n_proc} processes x {budget_s:.0f} s, {cpu:.0f} s CPU in all, fp64 numpy"}


def cpu_baseline(w, inp, budget_s=12.0):
    """Both oracle timings; the headline is the one on every host core."""
    single = cpu_baseline_single(w, inp, budget_s=budget_s / 2)
    par = cpu_baseline_parallel(w, inp, budget_s=budget_s / 2)
    if "error" in par:
        single["parallel"] = par
        single["host_cores"] = os.cpu_count() or 1
        return single
    par["single_process"] = single
    return par


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
    ap.add_argument("--repeats", type=int, default=5, help="timed regions of K steps (median reported)")
    ap.add_argument("--no-per-workload", action="store_true", help="only the headline workload")
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
