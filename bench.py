#!/usr/bin/env python
"""Benchmark of the BFP MoE decode layer on GB300.

Metric: MoE decode layer us and effective weight GB/s (BFP weight bytes the
step actually streams / device time; % of ~8 TB/s HBM). The headline
workload is the full-size layer at M=16 rows (hidden 2048, 256 experts of
width 512, top-8, shared expert of width 512, BFP4 experts, bf16 router):
each step streams the union of the experts the 16 rows select (~100) plus the
shared expert, ~180 MB, more than the 129 MB L2, and steps rotate over
several independently drawn layer instances. Secondary lines (same run): the
same layer at M=1, the hot-expert routing variant at M=16, the dense BFP8
projection [8192 x 2048] at M=1/8/16 and the greedy token over [16 x 151936]
logits (steps smaller than L2, each timed alone after a 256 MB L2-flushing
write); the BFP8 LM head [151936 x 2048] alone, the 8-row decode stack (40
layers, LM head, greedy token) and decode attention over two BFP KV caches of
131,072 tokens, all larger than L2, timed back to back.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
layer does not need a second GPU); value = all ranks' bytes / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode layer µs & effective weight GB/s (% of ~8 TB/s HBM) at M=1/16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the M=16 layer kernel, from one ncu
# capture of the same workload, valid while the kernel sources hash to src_sha (null otherwise).
NCU_TRAFFIC = {"moe_layer_m16": {"bytes_per_launch": 187_170_000, "src_sha": "08922c1bc8d4cb11"}}


def kernel_src_sha() -> str:
    """Hash of the layer kernel's sources with comments and blank space removed, so
    that editing a comment keeps a traffic figure taken from the same code. Of
    moe_layer.cu only the part before its public entry points counts (the kernel,
    its plan and its launch); the entry points after it validate and forward."""
    h = hashlib.sha256()
    for f in ("moe_layer.cu", "bfp_tiles.cuh", "bfp_device.cuh", "bfp_launch.h"):
        with open(os.path.join(ROOT, "block_floating_point_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        if f == "moe_layer.cu":
            src = src.split('\nextern "C" {\n', 1)[0]
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


CASES = ("m1", "m16_hot", "dense_m1", "dense_m16", "dense_m32", "dense_m32_tc", "lm_greedy_m8", "attn_32k")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--instances", type=int, default=3)
    ap.add_argument("--stack-layers", type=int, default=40)
    ap.add_argument("--seed", type=int, default=20261202)
    ap.add_argument("--quick", action="store_true", help="headline line only (no secondary workloads, no oracle)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="run one kernel's small workload a few times and exit (a short capture for a profiler)")
    return ap.parse_args()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = self.samples
        if self.window:
            inside = [s for s in rows if self.window[0] - 0.15 <= s[0] <= self.window[1] + 0.15]
            rows = inside or rows
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, v in rows:
            try:
                sm.append(float(v[1]))
                mx.append(float(v[2]))
            except Exception:
                continue
            for n, val in zip(names, v[5:9]):
                if val.lower() not in ("not active", "0x0000000000000000", "[n/a]", "n/a"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- ranks
def reduce_over_ranks(value: float, op: str, device=None) -> float:
    """max or sum of a per-rank scalar over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(bytes_per_step: float, steps: int, ms: float, device=None):
    """Whole-job GB/s: every rank's streamed bytes over the slowest rank's time. Returns (GB/s, max ms)."""
    ms_max = reduce_over_ranks(ms, "max", device)
    total = reduce_over_ranks(bytes_per_step * steps, "sum", device)
    return total / (ms_max * 1e-3) / 1e9, ms_max


# --------------------------------------------------------------------------- workload
def build_layers(n, seed, device):
    """n full-size layers with independent seeded weights (layer l: synth.LayerWeights(FULL, seed, layer=l)),
    each packed on the host and uploaded before the next is drawn."""
    import block_floating_point_gb300 as bfp
    import synth
    spec = synth.FULL
    layers = []
    for i in range(n):
        lw = synth.LayerWeights(spec, seed, layer=i)

        def src(e, lw=lw):
            key = synth.SHARED_EXPERT if e == "shared" else e
            return lw.gate(key), lw.up(key), lw.down(key)
        layers.append(bfp.MoELayer.from_source(spec.hidden, spec.n_experts, spec.ffn, spec.top_k, spec.shared_ffn,
                                               bfp.BFP4, lw.router_bf16(), lw.shared_gate_bf16(), src,
                                               lambda src=src: src("shared"), device=device))
    return spec, layers


def make_x(spec, seed, m, instance, device):
    import torch
    import synth
    x = np.stack([synth.activation_row(seed, 1000 * instance + r, spec.hidden, True, instance=instance)
                  for r in range(m)])
    return x, torch.from_numpy(x.view(np.int16)).to(device)


def union_bytes(layer, idx):
    return layer.weight_bytes(len(np.unique(idx)))


def other_bytes(layer, m):
    """bf16 router + shared gate read, bf16 x in, fp32 y out (the kernel's non-BFP traffic)."""
    return layer.n_experts * layer.hidden * 2 + layer.hidden * 2 + m * layer.hidden * (2 + 4)


def timed_graph(step, k, warmup, use_graph, group=99):
    """Run warmup then exactly k steps; returns device ms for the k steps (CUDA events on the launch stream)."""
    import torch
    stream = torch.cuda.current_stream()
    graphs = []
    if use_graph:
        try:
            for size in sorted({min(group, k), k % group} - {0}, reverse=True):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(size):
                        step(i)
                graphs.append((size, g))
        except Exception as exc:  # capture unsupported: eager launches
            print(f"# graph capture failed ({exc}); timing eager launches", file=sys.stderr)
            graphs = []
            torch.cuda.synchronize()

    def run(n):
        if graphs:
            full = dict(graphs)
            big = graphs[0][0]
            for _ in range(n // big):
                full[big].replay()
            rem = n % big
            if rem:
                if rem in full:
                    full[rem].replay()
                else:
                    for i in range(rem):
                        step(i)
        else:
            for i in range(n):
                step(i)

    run(warmup)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(k)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def timed_flushed(step, k, warmup, flush_buf, batch=32):
    """Each step timed alone (events around its launch) after a write of flush_buf (> L2); launches are queued
    behind a device sleep so the host never starves the device between the events. Returns (sum ms, per-step ms)."""
    import torch
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        flush_buf.zero_()
        step(i)
    torch.cuda.synchronize()
    times = []
    done = 0
    while done < k:
        n = min(batch, k - done)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda._sleep(int(4e6))
        for j in range(n):
            flush_buf.zero_()
            evs[j][0].record(stream)
            step(done + j)
            evs[j][1].record(stream)
        torch.cuda.synchronize()
        times += [a.elapsed_time(b) for a, b in evs]
        done += n
    return float(np.sum(times)), times


# --------------------------------------------------------------------------- reference arm (the oracle)
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    import synth
    spec = synth.FULL
    lw = synth.LayerWeights(spec, args.seed, 0, 0)

    def src(e):
        key = synth.SHARED_EXPERT if e == "shared" else e
        return lw.gate(key), lw.up(key), lw.down(key)
    router, sgate = lw.router_bf16(), lw.shared_gate_bf16()
    cache = oracle.ExpertCache(4, src)
    rows = [synth.activation_row(args.seed, r, spec.hidden, True) for r in range(16)]
    per_expert = 1769472
    # setup (not timed): the oracle's own encoding of every expert the sample rows select
    for x in rows:
        idx, _ = oracle.route_row(oracle.router_logits(router, x[None])[0], spec.top_k)
        for e in idx:
            cache(int(e))
    cache("shared")
    times = []
    for s in range(args.warmup + args.steps):
        x = rows[s % 16][None]
        t = time.perf_counter()
        oracle.moe_layer(x, router, sgate, cache, spec.top_k)
        if s >= args.warmup:
            times.append(time.perf_counter() - t)
    sec = float(np.mean(times))
    bytes_row = (spec.top_k + 1) * per_expert
    val = bytes_row / sec / 1e9
    out = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "MoE decode layer, full size (H=2048, 256 experts F=512, top-8, shared F=512, BFP4); "
                               "oracle step = one row of the M=16 workload", "rows_per_step": 1},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "one row of the M=16 decode step per step (its 8 experts + shared), single thread"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def cpu_baseline_sample(args, spec, x_np):
    """The oracle as it stands, single-threaded, on one full M=16 step of instance 0 (encoding excluded)."""
    import oracle
    import synth
    lw = synth.LayerWeights(spec, args.seed, 0, 0)

    def src(e):
        key = synth.SHARED_EXPERT if e == "shared" else e
        return lw.gate(key), lw.up(key), lw.down(key)
    router, sgate = lw.router_bf16(), lw.shared_gate_bf16()
    cache = oracle.ExpertCache(4, src)
    logits = oracle.router_logits(router, x_np)
    sel = set()
    for r in range(x_np.shape[0]):
        idx, _ = oracle.route_row(logits[r], spec.top_k)
        sel.update(int(e) for e in idx)
    for e in sel:
        cache(e)
    cache("shared")
    t = time.perf_counter()
    oracle.moe_layer(x_np, router, sgate, cache, spec.top_k)
    sec = time.perf_counter() - t
    return (len(sel) + 1) * 1769472 / sec / 1e9, sec


# --------------------------------------------------------------------------- our arm
def run_case(args):
    """One kernel's workload, launched `--steps` times after `--warmup` (for profiler captures: a few
    launches, a few GB on the device at most). Prints one line and exits 0."""
    import torch
    import block_floating_point_gb300 as bfp
    import synth
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    bfp.load()
    case = args.case
    if case in ("m1", "m16_hot"):
        spec, layers = build_layers(1, args.seed, device)
        L = layers[0]
        m = 1 if case == "m1" else 16
        if case == "m16_hot":
            bias = torch.from_numpy(synth.hot_bias(spec.n_experts, args.seed)).to(device)
            L = bfp.MoELayer(L.hidden, L.n_experts, L.ffn, L.top_k, L.shared_ffn, L.expert_fmt, L.router, L.shared_gate,
                             L.experts_gate_up, L.experts_down, L.shared_gate_up, L.shared_down, router_bias=bias)
        x = make_x(spec, args.seed, m, 0, device)[1]
        ws = bfp.moe_workspace(L, m)
        y = torch.empty((m, spec.hidden), dtype=torch.float32, device=device)
        step = lambda: bfp.moe_decode_layer(L, x, ws, y=y)
    elif case.startswith("dense_m"):
        m = int(case[len("dense_m"):].split("_")[0])
        if case.endswith("_tc"):
            bfp.set_linear_path(2)  # the tcgen05 kernel
        w = synth.normal(args.seed, synth.stream_id(synth.KIND_DENSE), (8192, 2048), std=0.02)
        mat = bfp.DeviceMatrix.from_host(8, 8192, 2048, bfp.encode(8, w), device=device)
        x = torch.from_numpy(np.stack([synth.activation_row(args.seed, 50000 + r, 2048, False)
                                       for r in range(m)]).view(np.int16)).to(device)
        ws = bfp.linear_workspace(mat, m)
        yl = torch.empty((m, 8192), dtype=torch.int16, device=device)
        step = lambda: bfp.linear(mat, x, ws, y_bf16=yl)
    elif case == "lm_greedy_m8":
        w = synth.normal(args.seed, synth.stream_id(synth.KIND_LMHEAD), (151936, 2048), std=synth.W_STD)
        mat = bfp.DeviceMatrix.from_host(8, 151936, 2048, bfp.encode(8, w), device=device)
        del w
        x = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, synth.stream_id(synth.KIND_STACK_H),
                                                             (8, 2048))).view(np.int16)).to(device)
        ws = bfp.linear_workspace(mat, 8)
        tk = torch.empty(8, dtype=torch.int32, device=device)
        step = lambda: bfp.linear_greedy(mat, x, ws, tokens=tk)
    else:  # attn_32k: 2 KV heads x 256, BFP8 K and V, 16 query heads, 32768 cached tokens
        n_ctx, d, kvh, g = 32768, 256, 2, 8
        kvc = bfp.KvCache(kvh, d, n_ctx, 8, 8, False, device=device)
        kk = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 42, (n_ctx, kvh, d))).view(np.int16)).to(device)
        vv = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 52, (n_ctx, kvh, d))).view(np.int16)).to(device)
        bfp.kv_append(kvc, kk, vv, 0)
        qa = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 60, (kvh * g, d))).view(np.int16)).to(device)
        ws = bfp.attn_workspace(kvc, kvh * g, n_ctx)
        oa = torch.empty((kvh * g, d), dtype=torch.float32, device=device)
        step = lambda: bfp.attn_decode(kvc, qa, n_ctx, d ** -0.5, ws, out=oa)
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    print(json.dumps({"case": case, "launches": args.warmup + args.steps}))


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist
    import block_floating_point_gb300 as bfp

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    bfp.load()
    peak, peak_kind = measured_peak()

    # every layer of the run has its own seeded weights: the headline rotates over the first `instances`, the
    # one-row line and the decode stacks run over all `stack_layers` of them (about 18 GB resident)
    n_all = args.instances if args.quick else max(args.instances, args.stack_layers)
    t_build = time.perf_counter()
    spec, all_layers = build_layers(n_all, args.seed + 7919 * rank, device)
    build_s = time.perf_counter() - t_build
    layers = all_layers[:args.instances]
    R = len(layers)
    M = 16
    xs, xts, ys, idxs = [], [], [], []
    ws = bfp.moe_workspace(layers[0], M)
    for i, L in enumerate(layers):
        x, xt = make_x(spec, args.seed + rank, M, i, device)
        xs.append(x)
        xts.append(xt)
        ys.append(torch.empty((M, spec.hidden), dtype=torch.float32, device=device))
        idx = torch.empty((M, spec.top_k), dtype=torch.int32, device=device)
        bfp.moe_decode_layer(L, xt, ws, y=ys[i], topk_idx=idx)
        idxs.append(idx)
    torch.cuda.synchronize()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    step_bytes = [union_bytes(L, idxs[i].cpu().numpy()) for i, L in enumerate(layers)]
    n_union = [len(np.unique(idxs[i].cpu().numpy())) for i in range(R)]
    avg_bytes = float(np.mean([step_bytes[i % R] for i in range(args.steps)]))
    avg_other = float(other_bytes(layers[0], M))

    def step16(i):
        j = i % R
        bfp.moe_decode_layer(layers[j], xts[j], ws, y=ys[j])

    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ms = timed_graph(step16, args.steps, args.warmup, not args.no_graph)
    t1 = time.time()
    sampler.mark(t0, t1)
    gbs, ms = aggregate_throughput(avg_bytes, args.steps, ms, device)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    assert bfp.workspace_status(ws) == bfp.BFP_OK
    us_layer = ms * 1e3 / args.steps
    kernel_gbs = (avg_bytes + avg_other) / (us_layer * 1e-6) / 1e9
    sha = kernel_src_sha()
    tr = NCU_TRAFFIC["moe_layer_m16"]
    traffic = tr["bytes_per_launch"] if tr["src_sha"] == sha else None

    # ---- e2e through the public API with host buffers (pinned x in, y out, synchronised every step)
    xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs]
    yh = torch.empty((M, spec.hidden), dtype=torch.float32).pin_memory()
    xd = torch.empty((M, spec.hidden), dtype=torch.int16, device=device)
    yd = torch.empty((M, spec.hidden), dtype=torch.float32, device=device)
    ke = max(1, min(args.steps, 300))
    for i in range(3):
        xd.copy_(xh[i % R], non_blocking=True)
        bfp.moe_decode_layer(layers[i % R], xd, ws, y=yd)
        yh.copy_(yd, non_blocking=True)
        torch.cuda.synchronize()
    t = time.perf_counter()
    for i in range(ke):
        xd.copy_(xh[i % R], non_blocking=True)
        bfp.moe_decode_layer(layers[i % R], xd, ws, y=yd)
        yh.copy_(yd, non_blocking=True)
        torch.cuda.synchronize()
    e2e_sec = (time.perf_counter() - t) / ke
    e2e_bytes = float(np.mean([step_bytes[i % R] for i in range(ke)]))

    out = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us_layer / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bfp4 weights x bf16 activations, fp16 tensor-core products, fp32 accumulate",
        "data": "synthetic (seeded N(0,0.02) weights encoded to BFP4, RMS-normalised N(0,1) bf16 rows)",
        "config": {"workload": "MoE decode layer M=16 (H=2048, 256 experts F=512, top-8, shared F=512, BFP4 "
                               "experts, bf16 router)", "rows": M, "instances": R,
                   "union_experts_per_step": n_union, "us_per_layer": us_layer,
                   "bfp_bytes_per_step": avg_bytes, "pct_of_8tbs": 100 * gbs / world / NOMINAL_HBM_GBS,
                   "pct_of_measured_copy": 100 * gbs / world / peak,
                   "gbs_incl_bf16_router_gate": (avg_bytes + layers[0].n_experts * layers[0].hidden * 2
                                                 + layers[0].hidden * 2) * args.steps * world / (ms * 1e-3) / 1e9,
                   "l2": "inputs larger than L2: each step streams ~180 MB of experts (> 129 MB L2), "
                         f"rotating over {R} independently drawn layer instances",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "layers_built": n_all, "host_build_s": build_s},
        "roofline": {"bound": "hbm", "achieved": kernel_gbs, "peak": peak, "unit": "GB/s",
                     "frac": kernel_gbs / peak, "traffic": traffic,
                     "kernel": "moe_layer_kernel<4,2> (one launch per step)",
                     "algorithmic_bytes_per_launch": avg_bytes + avg_other, "peak_source": peak_kind},
        "e2e": {"value": e2e_bytes / e2e_sec / 1e9, "unit": "GB/s", "h2d_bytes_per_step": M * spec.hidden * 2,
                "d2h_bytes_per_step": M * spec.hidden * 4, "us_per_step": e2e_sec * 1e6,
                "note": "public Python API over the C-ABI; pinned host x -> device, layer, y -> host, sync each step"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }

    if not args.quick:
        sec = {}
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        ksec = max(20, min(200, args.steps))
        # M=1: one launch per layer back to back (dependent launches in CUDA graphs) over the run's distinct
        # layers, each with its own row; the 9 experts one row selects differ from layer to layer, and 40
        # layers' selections (~640 MB) exceed L2, as in single-sequence decode. Also each step alone after an
        # L2 flush (launch latency included).
        NL = len(all_layers)
        ws1 = bfp.moe_workspace(all_layers[0], 1)
        x1 = [make_x(spec, args.seed + rank, 1, i, device)[1] for i in range(NL)]
        y1 = torch.empty((1, spec.hidden), dtype=torch.float32, device=device)
        b1 = []
        for i, L in enumerate(all_layers):
            idx = torch.empty((1, spec.top_k), dtype=torch.int32, device=device)
            bfp.moe_decode_layer(L, x1[i], ws1, y=y1, topk_idx=idx)
            b1.append(union_bytes(L, idx.cpu().numpy()))
        k1 = 2 * NL * max(1, (ksec + 2 * NL - 1) // (2 * NL))
        us1 = timed_graph(lambda i: bfp.moe_decode_layer(all_layers[i % NL], x1[i % NL], ws1, y=y1), k1, 2 * NL,
                          True, group=2 * NL) * 1e3 / k1
        g1 = float(np.mean(b1)) / (us1 * 1e-6) / 1e9
        tot, _ = timed_flushed(lambda i: bfp.moe_decode_layer(all_layers[i % R], x1[i % R], ws1, y=y1), ksec, 5, flush)
        us1f = tot * 1e3 / ksec
        assert bfp.workspace_status(ws1) == bfp.BFP_OK
        sec["m1"] = {"us_per_layer": us1, "gbs": g1, "pct_of_8tbs": 100 * g1 / NOMINAL_HBM_GBS,
                     "pct_of_measured_copy": 100 * g1 / peak, "bfp_bytes_per_step": float(np.mean(b1)),
                     "layers": NL, "kernel": "moe_row_kernel<4> (one launch per layer)",
                     "timing": f"{k1} launches back to back in CUDA graphs over {NL} distinct layers, CUDA events",
                     "us_alone_after_flush": us1f,
                     "alone_timing": "each step alone after a 256 MB L2 flush, CUDA events (includes launch latency)"}
        # hot-expert routing at M=16 (logit bias +2.0 on 8 fixed experts), same weights
        import synth
        bias = torch.from_numpy(synth.hot_bias(spec.n_experts, args.seed)).to(device)
        hot = [bfp.MoELayer(L.hidden, L.n_experts, L.ffn, L.top_k, L.shared_ffn, L.expert_fmt, L.router,
                            L.shared_gate, L.experts_gate_up, L.experts_down, L.shared_gate_up, L.shared_down,
                            router_bias=bias) for L in layers]
        bh, nh = [], []
        for i, L in enumerate(hot):
            idx = torch.empty((M, spec.top_k), dtype=torch.int32, device=device)
            bfp.moe_decode_layer(L, xts[i], ws, y=ys[i], topk_idx=idx)
            bh.append(union_bytes(L, idx.cpu().numpy()))
            nh.append(len(np.unique(idx.cpu().numpy())))
        tot, _ = timed_flushed(lambda i: bfp.moe_decode_layer(hot[i % R], xts[i % R], ws, y=ys[i % R]), ksec, 5,
                               flush)
        ush = tot * 1e3 / ksec
        gh = float(np.mean([bh[i % R] for i in range(ksec)])) / (ush * 1e-6) / 1e9
        sec["m16_hot"] = {"us_per_layer": ush, "gbs": gh, "pct_of_8tbs": 100 * gh / NOMINAL_HBM_GBS,
                          "union_experts_per_step": nh, "timing": "each step alone after a 256 MB L2 flush"}
        # dense BFP8 projection [8192 x 2048], M = 1 / 8 / 16 / 32: alone after a flush (launch latency included)
        # and back to back (a CUDA graph over 12 distinct matrices, 214 MB > L2, as inside a decode step); at 16
        # and 32 rows also the tcgen05 kernel (bfp_set_linear_path(2))
        w = synth.normal(args.seed, synth.stream_id(synth.KIND_DENSE), (8192, 2048), std=0.02)
        mats = [bfp.DeviceMatrix.from_host(8, 8192, 2048, bfp.encode(8, w), device=device)]
        for i in range(1, 12):
            mats.append(bfp.DeviceMatrix.from_host(8, 8192, 2048, bfp.encode(8, synth.normal(
                args.seed, synth.stream_id(synth.KIND_DENSE, i), (8192, 2048), std=0.02)), device=device))
        mat = mats[0]
        for m, path in ((1, 0), (8, 0), (16, 0), (32, 0), (16, 2), (32, 2)):
            xd_ = torch.from_numpy(np.stack([synth.activation_row(args.seed, 50000 + r, 2048, False)
                                             for r in range(m)]).view(np.int16)).to(device)
            wsl = bfp.linear_workspace(mat, m)
            yl = torch.empty((m, 8192), dtype=torch.int16, device=device)
            bfp.set_linear_path(path)
            try:
                tot, _ = timed_flushed(lambda i: bfp.linear(mat, xd_, wsl, y_bf16=yl), ksec, 5, flush)
                usb = timed_graph(lambda i: bfp.linear(mats[i % 12], xd_, wsl, y_bf16=yl), 198, 10, True) * 1e3 / 198
            finally:
                bfp.set_linear_path(0)
            assert bfp.workspace_status(wsl) == bfp.BFP_OK
            usd = tot * 1e3 / ksec
            gd = mat.nbytes / (usd * 1e-6) / 1e9
            key = f"dense_bfp8_m{m}" + ("_tcgen05" if path == 2 else "")
            sec[key] = {"us": usd, "gbs": gd, "pct_of_8tbs": 100 * gd / NOMINAL_HBM_GBS, "bytes": mat.nbytes,
                        "us_back_to_back": usb,
                        "gbs_back_to_back": mat.nbytes / (usb * 1e-6) / 1e9,
                        "kernel": "bfp_linear_tc_kernel (tcgen05)" if path == 2 else "bfp_linear_kernel (mma.sync)",
                        "timing": "us: each call alone after a 256 MB L2 flush; us_back_to_back: CUDA graph over "
                                  "12 distinct matrices"}
        del mats
        # greedy next token over LM-head logits [16 x 151936] fp32 (read from HBM after a flush)
        lg = torch.from_numpy(synth.normal(args.seed, 7, (16, 151936), std=3.0)).to(device)
        wsg = bfp.greedy_workspace(16, 151936, device)
        tokg = torch.empty(16, dtype=torch.int32, device=device)
        tot, _ = timed_flushed(lambda i: bfp.greedy_tokens(lg, wsg, tokg), ksec, 5, flush)
        usg = tot * 1e3 / ksec
        # the same calls back to back in a CUDA graph (logits L2-resident, as right after the LM head that
        # wrote them; no host launch overhead between calls)
        usb = timed_graph(lambda i: bfp.greedy_tokens(lg, wsg, tokg), ksec, 5, True) * 1e3 / ksec
        sec["greedy_m16_v151936"] = {"us": usg, "gbs": lg.numel() * 4 / (usg * 1e-6) / 1e9, "bytes": lg.numel() * 4,
                                     "us_back_to_back": usb, "launches": 2,
                                     "timing": "us: each call alone after a 256 MB L2 flush; us_back_to_back: "
                                               "consecutive calls in a CUDA graph on L2-resident logits"}
        # decode stacks over the run's distinct layers (40 by default, ~18 GB of BFP weights resident) + the BFP8
        # LM head [151936 x 2048], then the greedy next token; h is updated in place from step to step, as in
        # decoding. 8 rows (config 5) and 1 row (single-sequence decode).
        nl, vocab = len(all_layers), 151936
        stack = all_layers
        lm = bfp.DeviceMatrix.from_host(8, vocab, spec.hidden, bfp.encode(8, synth.normal(
            args.seed, synth.stream_id(synth.KIND_LMHEAD), (vocab, spec.hidden), std=synth.W_STD)), device=device)
        for mst in (8, 1):
            hst = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, synth.stream_id(synth.KIND_STACK_H),
                                                                   (mst, spec.hidden))).view(np.int16)).to(device)
            wss = bfp.moe_stack_workspace(stack, lm, mst)
            toks = torch.empty(mst, dtype=torch.int32, device=device)
            kst = 10
            sel = torch.empty((kst, nl, mst, spec.top_k), dtype=torch.int32, device=device)
            # one step: the stack, then the greedy next token taken in the LM head's epilogue (the logits are
            # not written out)
            for i in range(3):
                bfp.moe_stack_decode_greedy(stack, lm, hst, wss, tokens=toks, topk_idx=sel[0])
            es0, es1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            es0.record()
            for i in range(kst):
                bfp.moe_stack_decode_greedy(stack, lm, hst, wss, tokens=toks, topk_idx=sel[i])
            es1.record()
            torch.cuda.synchronize()
            assert bfp.workspace_status(wss) == bfp.BFP_OK
            ust_eager = es0.elapsed_time(es1) * 1e3 / kst
            # the same step captured once in a CUDA graph and replayed (no host work between launches)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                bfp.moe_stack_decode_greedy(stack, lm, hst, wss, tokens=toks)
            for i in range(3):
                g.replay()
            torch.cuda.synchronize()
            es0.record()
            for i in range(kst):
                g.replay()
            es1.record()
            torch.cuda.synchronize()
            assert bfp.workspace_status(wss) == bfp.BFP_OK
            ust = es0.elapsed_time(es1) * 1e3 / kst
            sa = sel.cpu().numpy()
            bst = float(np.mean([sum(union_bytes(stack[l], sa[i, l]) for l in range(nl)) for i in range(kst)])) \
                + lm.nbytes
            nun = float(np.mean([len(np.unique(sa[i, l])) for i in range(kst) for l in range(nl)]))
            # one row: up to 48 layers per launch (the residual row passes between layers inside the launch)
            layer_launches = -(-nl // 48) if mst == 1 else nl
            sec[f"stack_m{mst}_{nl}layers"] = {
                "us_per_step": ust, "tokens_per_s": mst / (ust * 1e-6), "bfp_bytes_per_step": bst,
                "gbs": bst / (ust * 1e-6) / 1e9, "pct_of_measured_copy": 100 * bst / (ust * 1e-6) / 1e9 / peak,
                "union_experts_per_layer": nun, "launches_per_step": layer_launches + 1,
                "timing": f"{kst} consecutive replays of the step ({nl} layers in {layer_launches} launch(es), then "
                          "the LM head with the greedy token in its epilogue) captured in one CUDA graph, CUDA events",
                "us_per_step_eager": ust_eager,
                "weights": f"{nl} layers with independent seeded weights (no layer repeats within a step); LM head "
                           f"BFP8 [{vocab} x {spec.hidden}] seeded N(0,0.02)",
                "layer_kernel": "moe_row_kernel<4, multi-layer>" if mst == 1 else "moe_layer_kernel<4,1>"}
            del wss
        # the LM head alone (330 MB, larger than L2: consecutive calls stream it from HBM)
        m8 = 8
        x8 = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, synth.stream_id(synth.KIND_STACK_H),
                                                              (m8, spec.hidden))).view(np.int16)).to(device)
        lg8 = torch.empty((m8, vocab), dtype=torch.float32, device=device)
        wsl8 = bfp.linear_workspace(lm, m8)
        for _ in range(3):
            bfp.linear(lm, x8, wsl8, y=lg8)
        el0, el1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        el0.record()
        for _ in range(20):
            bfp.linear(lm, x8, wsl8, y=lg8)
        el1.record()
        torch.cuda.synchronize()
        usl = el0.elapsed_time(el1) * 1e3 / 20
        tk8 = torch.empty(m8, dtype=torch.int32, device=device)
        for _ in range(3):
            bfp.linear_greedy(lm, x8, wsl8, tokens=tk8)
        torch.cuda.synchronize()
        el0.record()
        for _ in range(20):
            bfp.linear_greedy(lm, x8, wsl8, tokens=tk8)
        el1.record()
        torch.cuda.synchronize()
        uslg = el0.elapsed_time(el1) * 1e3 / 20
        sec["lm_head_bfp8_m8"] = {"us": usl, "gbs": lm.nbytes / (usl * 1e-6) / 1e9,
                                  "pct_of_measured_copy": 100 * lm.nbytes / (usl * 1e-6) / 1e9 / peak,
                                  "bytes": lm.nbytes, "timing": "20 consecutive calls (330 MB each, > L2)",
                                  "us_with_greedy_token_no_logits": uslg,
                                  "gbs_with_greedy_token": lm.nbytes / (uslg * 1e-6) / 1e9}
        # decode attention over a BFP KV cache, one query token: the 35B card's cache (2 KV heads x 256,
        # BFP8 K and V, 16 query heads) and the 27B card's bfp8_v4r cache (4 KV heads x 256, BFP8 K,
        # Hadamard-rotated BFP4 V, 24 query heads); caches of 128K tokens (> L2) timed back to back
        for name, kvh, g, kf, vf, rot in (("attn_bfp8_kv2_q16", 2, 8, 8, 8, False),
                                          ("attn_v4r_kv4_q24", 4, 6, 8, 4, True)):
            n_ctx, d = 131072, 256
            kvc = bfp.KvCache(kvh, d, n_ctx, kf, vf, rot, device=device)
            for p0 in range(0, n_ctx, 16384):  # fill by appends of seeded bf16 rows
                kk = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 40 + kvh, (16384, kvh, d),
                                                                      offset=p0 * kvh * d)).view(np.int16)).to(device)
                vv = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 50 + kvh, (16384, kvh, d),
                                                                      offset=p0 * kvh * d)).view(np.int16)).to(device)
                bfp.kv_append(kvc, kk, vv, p0)
            qa = torch.from_numpy(synth.to_bf16_bits(synth.normal(args.seed, 60, (kvh * g, d))).view(np.int16)).to(device)
            wsa = bfp.attn_workspace(kvc, kvh * g, n_ctx)
            oa = torch.empty((kvh * g, d), dtype=torch.float32, device=device)
            usa = timed_graph(lambda i: bfp.attn_decode(kvc, qa, n_ctx, d ** -0.5, wsa, out=oa), 50, 5, True) * 1e3 / 50
            assert bfp.workspace_status(wsa) == bfp.BFP_OK
            nb = n_ctx * kvc.bytes_per_token()
            sec[name] = {"us": usa, "context": n_ctx, "cache_bytes": nb, "gbs": nb / (usa * 1e-6) / 1e9,
                         "pct_of_measured_copy": 100 * nb / (usa * 1e-6) / 1e9 / peak, "launches": 2,
                         "timing": "50 consecutive calls in a CUDA graph (cache larger than L2)"}
            del kvc
        out["secondary"] = sec
        if rank == 0 and world == 1:
            v, s_ = cpu_baseline_sample(args, spec, xs[0])
            out["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                   "sample": f"one full M=16 step of instance 0 (16 rows), {s_:.2f} s, single "
                                             "thread, expert encoding excluded"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
