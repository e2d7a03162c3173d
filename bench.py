#!/usr/bin/env python
"""Benchmark of the CacheBlend blend step on one GB300.

One step = one cb_blend call: re-RoPE placement of the chunk caches, layer 0 over every row, the
check layer (deviation + top-k), selective recompute of the chosen rows in every later layer and
the last-token logits.  Workload (default): the Llama-3-8B shape (32 layers, d 4096, 32/8 heads,
head_dim 128, SwiGLU 14336, vocab 128256), random-init N(0, 0.02) weights, 6 chunks of 512 uniform
random tokens, each prefilled alone on the GPU, placed back to back, plus a 64-token query, r = 0.15.

Metric: blended context tokens per second (n_ctx / blend time); blend latency is reported beside
it.  Inputs are resident in HBM when the timed region starts; the weights (16 GB) and chunk caches
(384 MiB) exceed L2, and an L2-sized buffer is rewritten between steps (outside the timed events).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload  # noqa: E402

METRIC = "blended context tokens/sec & blend latency ms at r=0.15 (1×GB300), % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------
def blend_flops(shape: workload.ModelShape, n_layers: int, n_ctx: int, n_query: int, k: int) -> float:
    """Algorithmic FLOPs of a blend with `n_layers` layers (projections, attention, logits)."""
    d, hd, Hq, Hkv, F = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads, shape.ffn_hidden
    N, M = n_ctx + n_query, k + n_query
    per_row = 2 * d * (Hq * hd + 2 * Hkv * hd + Hq * hd + 3 * F)
    keys0 = N * (N + 1) / 2
    keysA = n_query * (n_ctx + 1) + n_query * (n_query - 1) / 2 + k * (n_ctx + 1) / 2
    attn = lambda keys: 4 * hd * Hq * keys
    f = N * per_row + attn(keys0)                                  # layer 0 (context K/V projections skipped
    f -= n_ctx * 2 * d * 2 * Hkv * hd                              # for reused rows)
    f += N * 2 * d * 2 * Hkv * hd + M * (per_row - 2 * d * 2 * Hkv * hd) + attn(keysA)   # check layer
    f += (n_layers - 2) * (M * per_row + attn(keysA))
    return f + 2 * d * shape.vocab


def blend_floor_ms(prof, steps: int, tensor_tflops, hbm_gbs: float) -> float:
    """Roofline time of one blend: the sum over kernel classes of max(FLOPs / tensor peak, bytes / HBM
    peak), from the per-class algorithmic work the library records (totals over `steps` blends).  A
    class with FLOPs but no tensor peak (fp32 configurations) counts its bytes only."""
    floor = 0.0
    for p in prof:
        t_f = p["flops"] / steps / (tensor_tflops * 1e12) if (tensor_tflops and p["flops"] > 0) else 0.0
        t_b = p["bytes"] / steps / (hbm_gbs * 1e9) if p["bytes"] > 0 else 0.0
        floor += max(t_f, t_b)
    return floor * 1e3


_SAMPLE = {}


def oracle_sample(spec: workload.WorkloadSpec, seed: int, ratio: float, sample_layers: int = 3):
    """Time the CPU oracle on the workload truncated to its first `sample_layers` layers (same
    request, same rows); return (seconds, full/sample FLOP ratio, description).  Inputs are made
    once and kept; only the oracle's blend is timed."""
    import oracle
    shape = spec.shape
    sample_layers = min(sample_layers, shape.n_layers)
    trunc = workload.ModelShape(**dict(shape.as_dict(), n_layers=sample_layers))
    key = (spec.name, seed, ratio, sample_layers)
    if key not in _SAMPLE:
        _SAMPLE.clear()
        _SAMPLE[key] = (workload.make_weights(trunc, seed), workload.make_request(spec, seed, ratio),
                        workload.synthetic_cache(trunc, seed, spec.n_ctx, workload.kv_std(shape)))
    w, req, caches = _SAMPLE[key]
    k = oracle.selected_count(spec.n_ctx, ratio)
    t0 = time.perf_counter()
    oracle.blend(trunc.as_dict(), w, req.tokens, caches, req.chunks, ratio, shape.dtype)
    dt = time.perf_counter() - t0
    scale = blend_flops(shape, shape.n_layers, spec.n_ctx, spec.n_query, k) / \
        blend_flops(shape, sample_layers, spec.n_ctx, spec.n_query, k)
    if sample_layers == shape.n_layers:
        desc = f"fp64 numpy oracle, {spec.name} request (r={ratio}), the whole blend ({shape.n_layers} layers)"
    else:
        desc = (f"fp64 numpy oracle, {spec.name} request (r={ratio}) on the first {sample_layers} of "
                f"{shape.n_layers} layers; time scaled to the full blend by the FLOP ratio {scale:.2f}")
    return dt, scale, desc


def oracle_k(spec: workload.WorkloadSpec, ratio: float) -> int:
    import oracle
    return oracle.selected_count(spec.n_ctx, ratio)


def cpu_cores():
    n = os.cpu_count() or 1
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            n = min(n, int(os.environ[v]))
    return n


# ------------------------------------------------------------------------------------------------
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(ws: int, units_per_rank: float, steps: int, local_ms: float):
    """Whole-job throughput of `ws` independent replicas: every rank processed `units_per_rank`
    units per step; the job took as long as its slowest rank.  Returns (units/s, ms per step)."""
    total_ms = max_over_ranks(ws, float(local_ms))
    return ws * units_per_rank * steps / (total_ms / 1e3), total_ms / steps


def run_reference(args, spec, ws, rank):
    """The reference arm: the CPU oracle, as it stands, on host cores (rank 0 only)."""
    if rank != 0:
        return
    ratio = args.ratio if args.ratio is not None else spec.ratios[0]
    seed = spec.seeds[0]
    for _ in range(args.warmup):
        oracle_sample(spec, seed, ratio)
    times, scale, desc = [], 1.0, ""
    for _ in range(args.steps):
        dt, scale, desc = oracle_sample(spec, seed, ratio)
        times.append(dt)
    # One step is one timed sample (the blend's first layers); ms_per_step is its measured time.  The
    # sample does 1/scale of a whole blend's FLOPs, so it blends n_ctx/scale context tokens' worth of work.
    t = float(np.sum(times))
    value = spec.n_ctx / scale * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "latency_ms": 1e3 * t * scale / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random-init weights, uniform random "
                                                          "tokens, generator chunk caches)",
            "config": {"workload": spec.name, "n_layers": spec.shape.n_layers, "d_model": spec.shape.d_model,
                       "n_ctx": spec.n_ctx, "n_query": spec.n_query, "n_chunks": spec.n_chunks,
                       "chunk_len": spec.chunk_len, "ratio": ratio, "k": oracle_k(spec, ratio),
                       "recomputed_rows": oracle_k(spec, ratio) + spec.n_query, "seed": seed, "parallelism": "cpu",
                       "step": f"one timed oracle sample ({desc}); ms_per_step is the sample's measured time, "
                               f"latency_ms the whole blend's (sample time x {scale:.2f})",
                       "blend_fraction_per_step": 1.0 / scale},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b-3k", choices=sorted(workload.WORKLOADS))
    ap.add_argument("--ratio", type=float, default=None)
    ap.add_argument("--gradual", action="store_true",
                    help="gradual filtering: 2r at the check layer, shrinking to r over the next 4 layers")
    ap.add_argument("--paged", type=int, default=0, metavar="P",
                    help="keep the chunk caches and the blended K/V in a paged pool of P-row pages (shuffled block table)")
    ap.add_argument("--matcher", action="store_true",
                    help="time the GPU fragment matcher instead (32K-token request, 4096 indexed 256-token chunks)")
    ap.add_argument("--low-entropy", action="store_true",
                    help="with --matcher: a request of one repeated token, so every window verifies")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-profile", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct cb_blend calls instead of a graph replay")
    # profiling-capture helpers: a smaller case with the same per-layer kernel shapes
    ap.add_argument("--layers", type=int, default=None, help="truncate the model to its first N layers")
    ap.add_argument("--vocab", type=int, default=None, help="override the vocabulary size")
    ap.add_argument("--synthetic-cache", action="store_true",
                    help="draw the chunk caches from the generator instead of prefilling them on the GPU")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    spec = workload.WORKLOADS[args.workload]
    if args.layers or args.vocab:
        import dataclasses
        shape = dataclasses.replace(spec.shape, n_layers=args.layers or spec.shape.n_layers,
                                    vocab=args.vocab or spec.shape.vocab)
        spec = dataclasses.replace(spec, shape=shape, name=f"{spec.name}-L{shape.n_layers}-V{shape.vocab}")
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, spec, ws, rank)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    import cacheblend_selective_kv_gb300 as cb
    if args.matcher:
        run_matcher(args, cb, ws, rank, local)
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape = spec.shape
    seed = spec.seeds[0]
    ratio = args.ratio if args.ratio is not None else spec.ratios[0]
    req = workload.make_request(spec, seed, ratio)

    t_setup = time.perf_counter()
    weights = workload.make_weights(shape, seed)
    model = cb.BlendModel(shape.as_dict(), weights, max_tokens=spec.n_tokens, max_chunks=spec.n_chunks, device=dev)
    del weights
    if args.synthetic_cache:
        raw = workload.synthetic_cache(shape, seed, spec.n_ctx, workload.kv_std(shape))
        cached = cb.to_device(raw, dev)
        del raw
    else:
        # chunk caches: each chunk prefilled alone at positions 0..len-1 by the library itself
        parts = [model.prefill_chunk(torch.from_numpy(t).to(dev)).clone() for t in req.chunk_tokens]
        cached = torch.cat(parts, dim=2).contiguous()
        del parts
    tokens = torch.from_numpy(req.tokens).to(dev)
    n = spec.n_tokens
    out_kv = model.kv_buffer(n)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
    k = cb.cb_selected_count(spec.n_ctx, ratio)
    schedule = workload.funnel_ratios(shape.n_layers, ratio) if args.gradual else None
    n_sel = k
    if schedule:
        counts = [cb.cb_selected_count(spec.n_ctx, r) for r in schedule]
        n_sel = counts[0] + sum(b for a, b in zip(counts, counts[1:]) if b < a)
    sel = torch.empty(max(n_sel, 1), dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > L2 (129 MB)
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    stream = torch.cuda.Stream(dev)

    paged = None
    if args.paged:
        P = args.paged
        nb = (n + P - 1) // P
        n_pages = nb + 16
        table = torch.from_numpy(np.random.default_rng(seed).permutation(n_pages)[:nb].astype(np.int32)).to(dev)
        pool = torch.empty((shape.n_layers, 2, n_pages * P, shape.n_kv_heads, shape.head_dim), dtype=cached.dtype,
                           device=dev)
        cb.cb_kv_scatter_pages(model.handle, cached, spec.n_ctx, pool, n_pages, P, table)
        torch.cuda.synchronize()
        paged = (pool, n_pages, P, table)

    def blend_call(tok, cache, st=False):
        if paged is not None:
            pool, n_pages, P, table = paged
            return cb.cb_blend_paged(model.handle, tok, n, pool, n_pages, P, table, table, req.chunks,
                                     schedule or (ratio,) * (shape.n_layers - 1), out_kv, logits, sel, None, stream,
                                     stats=st)
        if schedule:
            return cb.cb_blend_gradual(model.handle, tok, n, cache, req.chunks, schedule, out_kv, logits, sel, None,
                                       stream, stats=st)
        return cb.cb_blend(model.handle, tok, n, cache, req.chunks, ratio, out_kv, logits, sel, None, stream, stats=st)

    def step():
        return blend_call(tokens, cached, True)

    st = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st = step()
    torch.cuda.synchronize()

    def timed(fn, label):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier(ws)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            torch.cuda.nvtx.range_push(label)
            for i in range(args.steps):
                flush.zero_()
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        barrier(ws)
        return float(np.sum([a.elapsed_time(b) for a, b in evs]))

    # the blend is captured once in a CUDA graph (launch-latency free replays of the same kernels)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region --------------------------------------------------------------------------
    with ClockSampler(local) as clk:
        time.sleep(0.25)
        w0 = time.perf_counter()
        local_ms = timed(graph.replay if graph is not None else step, "timed_steps")
        wall = time.perf_counter() - w0
    value, ms_per_step = replica_throughput(ws, spec.n_ctx, args.steps, local_ms)
    direct_ms = None
    if graph is not None:
        direct_ms = replica_throughput(ws, spec.n_ctx, args.steps, timed(step, "direct_steps"))[1]

    # ---- per-kernel-class device time (CUDA events around each launch, a separate pass) -------
    kernels, roofline, blend_roofline = {}, None, None
    peaks, peak_src = load_peaks()
    if not args.no_profile:
        cb.cb_profile_enable(model.handle, True, 8192)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                flush.zero_()
                step()
        prof = cb.cb_profile_read(model.handle)
        cb.cb_profile_enable(model.handle, False)
        tensor_peak = peaks["bf16_tflops_sustained"] if shape.dtype == "bf16" else None
        for p in prof:
            ms = p["ms"]
            is_mma = p["name"].startswith("gemm") or p["name"] == "attention"
            ent = {"launches": p["launches"], "ms_total": ms, "ms_per_step": ms / args.steps,
                   "share": None}
            if ms > 0 and is_mma and p["flops"] > 0:
                ent["tflops"] = p["flops"] / (ms / 1e3) / 1e12
                if tensor_peak:
                    ent["frac_tensor"] = ent["tflops"] / tensor_peak
            if ms > 0 and p["bytes"] > 0:
                ent["gbs"] = p["bytes"] / (ms / 1e3) / 1e9
                ent["frac_hbm"] = ent["gbs"] / peaks["hbm_gbs"]
            kernels[p["name"]] = ent
        tot = sum(e["ms_total"] for e in kernels.values()) or 1.0
        for e in kernels.values():
            e["share"] = e["ms_total"] / tot
        floor_ms = blend_floor_ms(prof, args.steps, tensor_peak, peaks["hbm_gbs"])
        blend_roofline = {"floor_ms": floor_ms, "frac": floor_ms / ms_per_step,
                          "definition": "sum over kernel classes of max(algorithmic FLOPs / sustained tensor peak, "
                                        "algorithmic bytes / HBM peak), over the measured blend time"}
        top = max(kernels, key=lambda n_: kernels[n_]["ms_total"])
        e = kernels[top]
        pinfo = next(p for p in prof if p["name"] == top)
        traffic = load_traffic(top, spec.name)
        if (top.startswith("gemm") or top == "attention") and shape.dtype == "bf16":
            ach = pinfo["flops"] / pinfo["launches"] / (e["ms_total"] / e["launches"] / 1e3) / 1e12
            roofline = {"kernel": top, "bound": "tensor", "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                        "frac": ach / tensor_peak, "traffic": traffic,
                        "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside a long step)"}
        else:
            ach = pinfo["bytes"] / pinfo["launches"] / (e["ms_total"] / e["launches"] / 1e3) / 1e9
            roofline = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"], "traffic": traffic, "peak_source": f"{peak_src} hbm_gbs"}

    # ---- end to end through the public API with host buffers ----------------------------------
    # The caller's tokens and chunk caches sit in pinned host memory and the blended K/V and logits
    # must end up there.  Pipelined: cb_blend_streamed loads the caches layer by layer on a copy stream
    # (overlapping the recompute of earlier layers) and copies every finished layer back on another.
    # Serial (for comparison): copy everything in, blend, copy everything out.
    e2e = None
    if not args.no_e2e and not args.paged:
        h_tokens = torch.from_numpy(req.tokens).pin_memory()
        h_cached = cached.cpu().pin_memory()
        h_out = torch.empty(out_kv.shape, dtype=out_kv.dtype).pin_memory()
        h_logits = torch.empty(shape.vocab, dtype=torch.float32).pin_memory()
        d_tokens = torch.empty_like(tokens)
        d_cached = torch.empty_like(cached)
        cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ratios_l = schedule if schedule else (ratio,) * (shape.n_layers - 1)

        def e2e_streamed():
            d_tokens.copy_(h_tokens, non_blocking=True)
            cb.cb_blend_streamed(model.handle, d_tokens, n, h_cached, req.chunks, ratios_l, out_kv, logits,
                                 out_kv_host=h_out, out_selected=sel, stream=stream, copy_stream=cs_in,
                                 copy_back_stream=cs_out)
            h_logits.copy_(logits, non_blocking=True)

        def e2e_serial():
            d_tokens.copy_(h_tokens, non_blocking=True)
            d_cached.copy_(h_cached, non_blocking=True)
            blend_call(d_tokens, d_cached)
            h_out.copy_(out_kv, non_blocking=True)
            h_logits.copy_(logits, non_blocking=True)

        def time_e2e(fn):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            with torch.cuda.stream(stream):
                for _ in range(2):
                    fn()
                torch.cuda.synchronize()
                for i in range(args.steps):
                    flush.zero_()
                    ev[i][0].record(stream)
                    fn()
                    ev[i][1].record(stream)
            torch.cuda.synchronize()
            return replica_throughput(ws, spec.n_ctx, args.steps, float(np.sum([a.elapsed_time(b) for a, b in ev])))

        e_val, e_ms = time_e2e(e2e_streamed)
        s_val, s_ms = time_e2e(e2e_serial)
        bi = h_tokens.numel() * 4 + h_cached.numel() * h_cached.element_size()
        bo = h_out.numel() * h_out.element_size() + h_logits.numel() * 4
        e2e = {"value": e_val, "unit": "tokens/s", "latency_ms": e_ms, "h2d_bytes_per_step": int(bi),
               "d2h_bytes_per_step": int(bo),
               "path": "cb_blend_streamed: caches loaded layer by layer from pinned host memory on a copy "
                       "stream, each finished layer copied back on another, overlapping the recompute",
               "serial": {"value": s_val, "latency_ms": s_ms,
                          "path": "copy all in, cb_blend, copy all out, one stream"}}

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----------------------------------------------
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not schedule:
        dt, scale, desc = oracle_sample(spec, seed, ratio)
        cpu = {"value": spec.n_ctx / (dt * scale), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc, "sample_seconds": dt}

    clocks = clk.summary()
    model.close()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "latency_ms": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": shape.dtype, "data": "synthetic (seeded random-init weights and uniform random tokens)",
                "config": {"workload": spec.name, "n_layers": shape.n_layers, "d_model": shape.d_model,
                           "n_ctx": spec.n_ctx, "n_query": spec.n_query, "n_chunks": spec.n_chunks,
                           "chunk_len": spec.chunk_len, "ratio": ratio, "k": k, "recomputed_rows": k + spec.n_query,
                           "seed": seed, "parallelism": "replicas" if ws > 1 else "single",
                           "schedule": ("gradual filtering, per-layer ratios " + ",".join(f"{r:.4g}" for r in schedule))
                           if schedule else "one selection at the check layer",
                           "kv_layout": (f"paged pool, {args.paged}-row pages, shuffled block table (read and "
                                         "written in place)") if args.paged else "contiguous",
                           "l2": "inputs exceed L2 (16 GB weights, 384 MiB caches) and a 256 MiB buffer is "
                                 "rewritten between steps outside the timed events",
                           "timing": ("CUDA events around each step on the launching stream, summed over the steps; "
                                      + ("each step replays one cb_blend captured in a CUDA graph"
                                         if graph is not None else "each step is a direct cb_blend call")),
                           "direct_call_ms_per_step": direct_ms,
                           "setup_s": round(setup_s, 1), "wall_s_timed": round(wall, 4)},
                "gpu_launches": int(st["kernel_launches"]) * args.steps if st else None,
                "clocks": clocks, "roofline": roofline, "blend_roofline": blend_roofline, "kernels": kernels, "e2e": e2e, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)


def run_matcher(args, cb, ws, rank, local):
    """Fragment lookup of a 32K-token request against 4096 indexed 256-token chunks (half of them planted
    in the request, the rest absent), timed with CUDA events around each cb_index_match."""
    import torch
    torch.cuda.set_device(local)
    C, V, n_tok, n_idx, seed = 256, 128256, 32768, 4096, 9
    chunks = np.stack([workload.tokens(seed, 1000 + i, C, V) for i in range(n_idx)]).astype(np.uint32)
    req = workload.tokens(seed, 1, n_tok, V)
    rng = np.random.default_rng(seed)
    if args.low_entropy:
        # one repeated token: every one of the 32513 windows verifies against chunk 0 (made of that token)
        chunks[0] = 77
        req[:] = 77
    else:
        for slot, i in enumerate(rng.permutation(n_idx)[: n_tok // C]):
            req[slot * C:(slot + 1) * C] = chunks[i]
    index = cb.FragmentIndex(C, chunks, np.arange(n_idx), np.zeros(n_idx, np.int32), np.ones(n_idx, np.int32), n_tok)
    dev = torch.device("cuda", local)
    t = torch.from_numpy(req).to(dev)
    out = torch.empty((4096, 3), dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            index.match_async(t, 1, out, cnt, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            index.match_async(t, 1, out, cnt, stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
    n_match = int(cnt.item())
    # ALU roofline of the window kernel: one 64-bit multiply-add per token of every window
    windows = n_tok - C + 1
    line = {"metric": "fragment match: request tokens/s (GPU matcher)", "value": n_tok / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "u64", "data": "synthetic (seeded tokens)",
            "config": {"workload": f"{n_tok}-token request{' of one repeated token' if args.low_entropy else ''}, "
                                   f"{n_idx} indexed {C}-token chunks, stride 1, leftmost-greedy", "matches": n_match,
                       "window_hash_macs": windows * C}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    index.close()


def load_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was captured on this
    workload's per-layer shapes and still matches the source it was taken from (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        ent = d.get(f"{kernel}@{workload_name}") or d.get(kernel)
        if not ent or ent.get("workload") != workload_name:
            return None
        import hashlib
        src = os.path.join(ROOT, ent["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != ent["source_sha"]:
            return None
        return ent["dram_bytes_per_launch_full"]
    except Exception:
        return None


if __name__ == "__main__":
    main()
