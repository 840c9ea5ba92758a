#!/usr/bin/env python3
"""Benchmark: decode over a compressed KV cache on GB300, one JSON line on stdout.

Default workload ("streaming"): the Llama-2-7B attention shape -- 32 layers, 32 MHA heads,
d_head 128, bf16, batch 16 -- decoding over a StreamingLLM cache of 4 sinks + a 2044-token
ring filled from a 4096-token prompt, keys stored pre-rotation and rotated at in-cache
positions on every step.  One step = for every layer: append the new token's key/value into
its ring slot, then decode attention of the 32 query heads over the 2049 attended slots; then
the decode position advances.  Metric: tokens/s (batch x steps / time); the decode kernel's
HBM bandwidth is reported against the measured copy peak.

Other workloads (--workload): snapkv (select + compact + 256-step decode), h2o (prompt
selection + per-step accumulate/evict), pyramid (per-layer budgets, D=256, GQA 6), tiny.

Multi-GPU: the path shards into independent replicas (no exchange step); under torchrun every
rank runs the same workload on its own GPU and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from kv_cache_compression_kvc_gb300 import inputs as I  # noqa: E402

PEAK_FALLBACK_GBS = 6800.0


# ----------------------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and time.perf_counter() - t0 < timeout:
            time.sleep(0.02)

    def window(self, t_begin, t_end):
        self.t_begin, self.t_end = t_begin, t_end

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = getattr(self, "t_begin", -1e30), getattr(self, "t_end", 1e30)
        for ts, ln in self.lines:
            if not (lo <= ts <= hi + 0.25):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_traffic(kernel_file: str, key: str):
    """DRAM bytes per launch from a committed ncu summary, or None if the kernel source has
    changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[key]
        src = open(os.path.join(ROOT, "kv_cache_compression_kvc_gb300", "csrc", kernel_file),
                   "rb").read()
        if hashlib.sha256(src).hexdigest()[:16] != d["source_sha"]:
            return None
        return float(d["bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- workloads
class Streaming:
    """StreamingLLM decode: per layer append into the ring + RoPE decode over 4 + W + 1 slots."""

    kernel_file = "decode_attn.cuh"
    traffic_key = "decode_attn/streaming"

    def __init__(self, w: I.Workload, dev, kvc):
        self.w, self.dev, self.kvc = w, dev, kvc
        L, B, H, D, S, W = w.layers, w.batch, w.n_heads_kv, w.d_head, w.n_sink, w.window
        self.slots = S + W + 1
        self.K = torch.empty((L, B, H, self.slots, D), dtype=w.dtype, device=dev)
        self.V = torch.empty_like(self.K)
        ring_slot = [a if a < S else S + (a - S) % (W + 1) for a in
                     list(range(S)) + list(range(w.prompt - W, w.prompt))]
        idx = torch.tensor(ring_slot, device=dev)
        for l in range(L):
            k, v, _ = I.streaming_prefill(w, l, dev)
            self.K[l][:, :, idx] = k
            self.V[l][:, :, idx] = v
        self.table = kvc.kvc_rope_table(self.slots, D, w.theta).to(dev)
        self.t = torch.tensor([w.prompt], dtype=torch.int64, device=dev)
        self.q_s = torch.empty((L, B, w.n_heads_q, D), dtype=w.dtype, device=dev)
        self.k_s = torch.empty((L, B, H, D), dtype=w.dtype, device=dev)
        self.v_s = torch.empty_like(self.k_s)
        self.out = torch.empty((L, B, w.n_heads_q, D), dtype=torch.float32, device=dev)
        self.caches = [kvc.cache_view(self.K[l], self.V[l]) for l in range(L)]
        self.rope = kvc.make_rope(S, W, self.t, self.table)
        self.ws = kvc.decode_workspace(B, w.n_heads_q, H, D, self.slots, dev)
        self.launches_per_step = 2 * L + 1

    def step_inputs(self, step, seed_base):
        w = self.w
        g = I.generator(seed_base + step, self.dev)
        shp_q = (w.layers, w.batch, w.n_heads_q, w.d_head)
        shp_k = (w.layers, w.batch, w.n_heads_kv, w.d_head)
        q = torch.randn(shp_q, generator=g, device=self.dev).to(w.dtype)
        k = torch.randn(shp_k, generator=g, device=self.dev).to(w.dtype)
        v = torch.randn(shp_k, generator=g, device=self.dev).to(w.dtype)
        return q, k, v

    def load_inputs(self, q, k, v):
        self.q_s.copy_(q, non_blocking=True)
        self.k_s.copy_(k, non_blocking=True)
        self.v_s.copy_(v, non_blocking=True)

    def appends(self):
        kvc, w = self.kvc, self.w
        for l in range(w.layers):
            kvc.kvc_stream_append(None, None, kvc.KVC_APPEND_RING, self.k_s[l], self.v_s[l],
                                  t=self.t, n_sink=w.n_sink, window=w.window,
                                  cache=self.caches[l])

    def decodes(self):
        kvc, w = self.kvc, self.w
        for l in range(w.layers):
            kvc.kvc_decode_attn(self.q_s[l], None, None, scale=w.scale, rope=self.rope,
                                out=self.out[l], ws=self.ws, cache=self.caches[l])
        kvc.kvc_position_advance(self.t, 1)

    def decode_bytes_per_launch(self):
        """Algorithmic bytes of one decode launch: the attended K and V rows once, q and out."""
        w = self.w
        n = min(int(self.t.item()) + 1, self.slots)
        eb = torch.tensor([], dtype=w.dtype).element_size()
        kv = 2 * w.batch * w.n_heads_kv * n * w.d_head * eb
        return kv + w.batch * w.n_heads_q * w.d_head * (eb + 4)

    def describe(self):
        w = self.w
        return {"workload": "streaming decode, Llama-2-7B attention shape",
                "layers": w.layers, "batch": w.batch, "n_heads": w.n_heads_q,
                "d_head": w.d_head, "sinks": w.n_sink, "window": w.window,
                "prompt": w.prompt, "slots_per_step": self.slots, "kv_dtype": "bf16",
                "rope": "in-cache positions, theta 10000",
                "l2": "inputs larger than L2 (17.2 GB of KV per step)",
                "graph": "appends and decodes captured as two CUDA graphs per step"}

    def oracle_sample(self, budget_s=12.0):
        """Time the oracle's StreamingLLM decode on (b, head, layer) slices; returns
        (seconds per slice, slices per step, n timed)."""
        import oracle
        w = self.w
        rng = np.random.default_rng(0)
        D, S, W, t = w.d_head, w.n_sink, w.window, w.prompt
        hk = rng.standard_normal((t + 1, D))
        hv = rng.standard_normal((t + 1, D))
        q = rng.standard_normal(D)
        oracle.stream_decode(t, S, W, q, hk, hv, w.scale)     # build + warm
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            oracle.stream_decode(t, S, W, q, hk, hv, w.scale)
            n += 1
        per = (time.perf_counter() - t0) / n
        return per, w.batch * w.n_heads_q * w.layers, n


WORKLOAD_CLASSES = {"streaming": Streaming}


# ----------------------------------------------------------------------------- main arms
def run_gpu(args):
    rank, world, local = dist_env()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from kv_cache_compression_kvc_gb300 import build, kvc
    build.build()
    kvc.load()
    w = I.WORKLOADS[args.workload]
    if args.layers:
        w = dataclasses.replace(w, layers=args.layers)
    R = WORKLOAD_CLASSES[args.workload](w, dev, kvc)
    stream = torch.cuda.current_stream()

    # distinct per-step inputs (reused cyclically past 64 steps)
    total = min(args.warmup + args.steps, 64)
    inputs = [R.step_inputs(i, w.seed * 7 + 17) for i in range(total)]
    torch.cuda.synchronize()

    # --- capture the step as two graphs (appends; decodes + position advance) ---------------
    R.load_inputs(*inputs[0])
    t_save = R.t.clone()
    R.appends()                             # one eager pass: per-device library set-up happens
    R.decodes()                             # outside capture (it rewrites the same ring slot)
    torch.cuda.synchronize()
    R.t.copy_(t_save)
    g_app, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_app):
        R.appends()
    with torch.cuda.graph(g_dec):
        R.decodes()
    R.t.copy_(t_save)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(args.warmup):
        R.load_inputs(*inputs[i % total])
        g_app.replay()
        g_dec.replay()
    bytes_per_launch = R.decode_bytes_per_launch()
    code = kvc.kvc_device_status()
    if code != 0:
        raise RuntimeError(f"device range check fired during warm-up: {code}")

    ev_s = torch.cuda.Event(enable_timing=True)
    ev_e = torch.cuda.Event(enable_timing=True)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.wait_first()
        torch.cuda.synchronize()
        t_host0 = time.perf_counter()
        ev_s.record(stream)
        for i in range(args.steps):
            R.load_inputs(*inputs[(args.warmup + i) % len(inputs)])
            g_app.replay()
            marks[i][0].record(stream)
            g_dec.replay()
            marks[i][1].record(stream)
        ev_e.record(stream)
        torch.cuda.synchronize()
        clocks.window(t_host0, time.perf_counter())
    barrier()
    elapsed_ms = ev_s.elapsed_time(ev_e)
    decode_ms = sum(a.elapsed_time(b) for a, b in marks) / args.steps / w.layers
    code = kvc.kvc_device_status()
    if code != 0:
        raise RuntimeError(f"device range check fired in the timed region: {code}")

    # --- end to end: host inputs -> C-ABI calls -> host outputs ------------------------------
    host_in = [tuple(x.cpu().pin_memory() for x in inputs[i]) for i in range(total)]
    host_out = torch.empty(R.out.shape, dtype=R.out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host_in[0])
    d2h = host_out.numel() * host_out.element_size()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        R.load_inputs(*host_in[i % total])
        R.appends()
        R.decodes()
        host_out.copy_(R.out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = e0.elapsed_time(e1)

    times = torch.tensor([elapsed_ms, e2e_ms, decode_ms], dtype=torch.float64, device=dev)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    elapsed_ms, e2e_ms, decode_ms = times.tolist()
    if rank != 0:
        return
    tokens = w.batch * args.steps * world
    value = tokens / (elapsed_ms / 1e3)
    peak, peak_kind = measured_peak()
    achieved = bytes_per_launch / (decode_ms / 1e3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        per, slices, n = R.oracle_sample()
        cpu = {"value": w.batch / (per * slices), "unit": "tokens/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{n} oracle StreamingLLM decodes of one (batch, head, layer) slice at "
                         f"the workload's shape, extrapolated to {slices} slices per step "
                         f"(extrapolated)"}
    line = {
        "metric": "compressed-KV decode attention tokens/s (HBM GB/s and % of roofline in "
                  "'roofline')",
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) keys/values/queries, sink-boosted keys; no model)",
        "config": R.describe(),
        "roofline": {"bound": "hbm", "kernel": "decode_attn_kernel",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": round(decode_ms, 5),
                     "traffic": kernel_traffic(R.kernel_file, R.traffic_key)},
        "e2e": {"value": round(tokens / (e2e_ms / 1e3), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": R.launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The oracle as it stands, on the host cores, on bounded samples of the same workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = I.WORKLOADS[args.workload]
    import oracle
    oracle.build()
    R = WORKLOAD_CLASSES[args.workload].__new__(WORKLOAD_CLASSES[args.workload])
    R.w = w
    per_step = []
    budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        per, slices, n = R.oracle_sample(budget_s=budget)
        if i >= args.warmup:
            per_step.append(per * slices)
    step_s = statistics.mean(per_step)
    value = w.batch / step_s
    line = {
        "impl": "reference", "metric": "compressed-KV decode attention tokens/s (HBM GB/s and "
                                       "% of roofline in 'roofline')",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} (oracle on host cores, sampled slices)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "per step, oracle decodes of single (batch, head, layer) "
                                   "slices for a fixed time, extrapolated to the full step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (smaller case for profiling)")
    ap.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_CLASSES), default="streaming")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
