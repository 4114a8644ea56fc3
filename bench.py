"""Benchmark of the CSA KV compressor on one GB300 (or N, one process per GPU).

A step is one ratio-4 overlapped prefill of the Flash CSA layer (B=1 sequence of 4096 tokens,
dim 4096, two branches x 512, fp4 latent): projection, 8-candidate softmax pool, bf16,
RMSNorm, YaRN RoPE, fp4 round trip and the state update.  `value` is compressed KV entries/s
over all ranks; tokens/s and the batched-decode rate (B=128, ratio-4 overlapped + ratio-128
compressors, one token per sequence per step) are reported beside it.  Inputs are seeded
synthetic data resident in HBM before the timed region; L2 is flushed (a 2x-L2 buffer is
written) between timed iterations.  Under torchrun every rank runs its own sequences
(weak scaling, no collective on the data path; the barrier and the max-over-ranks of the
time are the only communication).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "compressed KV entries/s & input tokens/s (ratio-4 prefill), decode steps/s; % roofline"
WORKLOAD = "Flash CSA layer prefill: B=1, N=4096, dim=4096, head_dim=512, ratio 4 overlapped, YaRN RoPE 64, fp4"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="decode steps timed (0: the batched decode workload's 512)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--decode-only", action="store_true",
                    help="run and print only the decode measurement (for profiling)")
    ap.add_argument("--other-only", choices=["hca", "indexer", "pairs"], default=None,
                    help="run and print only the prefill of that other compressor instance (for profiling)")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="layer instances rotated in the decode measurement (0: enough to exceed L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the long-context prefill sweep")
    ap.add_argument("--prefill-pair", action="store_true",
                    help="prefill compressors with the option prefill_pair = 2 (two CTAs sharing one MMA of 256 "
                         "rows where the tiles pair up; off by default, measured slower): for profiling it")
    ap.add_argument("--clock-seconds", type=float, default=1.0,
                    help="seconds of untimed steps run under the clock sampler before the timed region")
    return ap.parse_args()


def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sources_hash(files):
    """First 16 hex digits of the sha256 of the library sources `files`, concatenated in order."""
    import hashlib
    csrc = os.path.join(ROOT, "deepseek_v4_compressed_wkv_gb300", "csrc")
    m = hashlib.sha256()
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            m.update(f.read())
    return m.hexdigest()[:16]


def profiled_traffic(entry, key):
    """DRAM bytes (read + write) that an ncu capture measured for a kernel, from
    profiles/traffic.json, or None when the kernel's sources no longer hash as they did at the
    capture (the counters then describe another kernel)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(entry)
    if not rec or key not in rec:
        return None
    if sources_hash(rec["sources"]) != rec.get("sources_sha256_16"):
        return None
    return int(rec[key])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is under load."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 6:
                self.samples.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if not self.samples:
            return None
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[2:6]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def clock_rejection(clk):
    """Why a timed region's clock record rejects it, or None: a hardware or thermal slowdown
    was active, or the median SM clock sat well below the maximum with no reason given (a
    leftover clock lock).  A power cap alone is kept (normal under sustained tensor load)."""
    if not clk:
        return None
    bad = [r for r in clk.get("reasons", []) if r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")]
    if bad:
        return bad
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if sm and mx and sm < 0.8 * mx and not clk.get("reasons"):
        return ["sm_clock_below_max_without_reason"]
    return None


# ---------------------------------------------------------------------------------------------

def hold_gpu(flush, n=64):
    """Enqueues about n x 40 us of device work (writes of the L2-flush buffer) so that the host,
    enqueueing the timed steps behind it, is never what the device waits for: each step is timed
    by its own events on the device, and a gap while the host issues the next call would be
    counted in it."""
    for i in range(n):
        flush.fill_(float(-i))


def make_inputs(torch, csa, synthetic, layer, seed, B, N, rank, device, args=None):
    x = np.stack([synthetic.tokens(seed, rank * B + b, 0, N, layer.dim) for b in range(B)])
    xb = torch.from_numpy(x).to(torch.bfloat16).to(device)
    wkv, wgate, gain = synthetic.weights(seed, layer)
    opts = {"prefill_pair": 2} if args is not None and getattr(args, "prefill_pair", False) else {}
    comp = csa.Compressor(layer.dim, layer.head_dim, layer.ratio, layer.overlap, max_batch=max(B, 1),
                          rope_dim=layer.rope_dim, fp4=layer.fp4, **opts)
    comp.set_weights(torch.from_numpy(wkv).to(device), torch.from_numpy(wgate).to(device),
                     torch.from_numpy(gain).to(device))
    return comp, xb


def run_ours(args, rank, world, local):
    import torch

    import deepseek_v4_compressed_wkv_gb300 as csa
    import synthetic

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(device)
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    B, N = 1, wl.tokens[0]
    G = N // layer.ratio
    comp, x = make_inputs(torch, csa, synthetic, layer, wl.seed, B, N, rank, device, args)
    H = layer.head_dim
    out = comp._alloc_out(B * G, device, prequant=False)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(int(2 * getattr(props, "L2_cache_size", 128 << 20)) // 4 + 1, dtype=torch.float32,
                        device=device)

    def step():
        comp.prefill(x, out=out, prequant=False)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b_ in kev:  # torch creates an event on its first record; the library re-records it
        a.record(stream)
        b_.record(stream)
    def timed_loop():
        clocks = ClockSampler(local)
        clocks.start()
        # keep the GPU busy long enough for the clock sampler to see it under this load
        t_end = time.time() + args.clock_seconds
        while time.time() < t_end:
            step()
            torch.cuda.synchronize()
        launches0 = comp.kernel_launches()
        barrier(world)
        torch.cuda.synchronize()
        hold_gpu(flush)
        for i in range(K):
            flush.fill_(float(i))
            comp.set_profile_events(*kev[i])
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        clk = clocks.stop()
        comp.set_profile_events(None, None)
        return clk, comp.kernel_launches() - launches0

    clk, launches = timed_loop()
    bad = clock_rejection(clk)
    if bad:  # a throttled or clock-locked run is measured once more, and the line says so
        clk, launches = timed_loop()
        clk["remeasured_after"] = bad
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    total_ms = max_over_ranks(sum(step_ms), world, device)
    ms = total_ms / K
    entries = B * G * world
    value = entries / (ms * 1e-3)
    tokens_s = B * N * world / (ms * 1e-3)

    # dominant kernel: the projection (fp32-equivalent: three bf16 products per weight on the
    # tensor-core path, f32 FMA on the CUDA-core path)
    flops = 2.0 * B * N * layer.dim * 2 * layer.width
    kms = statistics.mean(kern_ms)
    achieved = flops / (kms * 1e-3) / 1e12
    tc = comp.uses_tensor_cores()
    if tc:
        peak = peaks["bf16_tflops"] / 3.0
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": profiled_traffic("prefill_tc_flash_csa", "traffic_bytes_per_launch"),
                "kernel": "csa_prefill_tc (projection + fused pool/norm/RoPE/fp4)",
                "peak_basis": f"{peaks['source']} bf16 dense {peaks['bf16_tflops']} TFLOP/s / 3 bf16 passes"}
    else:
        sm_clock = (clk or {}).get("sm_max_mhz") or 2070.0
        peak = props.multi_processor_count * 128 * 2 * sm_clock * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None, "kernel": "gemm_ffma_kernel (f32 FMA projection)",
                "peak_basis": f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 flop x {sm_clock:.0f} MHz"}

    e2e_ms, h2d, d2h = measure_e2e(torch, comp, x, out, B * G, K, stream, world, device)

    line = {"metric": METRIC, "value": value, "unit": "entries/s", "n_gpus": world, "steps": K,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": N, "entries_per_step": entries,
                       "l2": "flushed between timed iterations (2x L2 buffer written)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tokens_per_s": tokens_s, "kernel_ms": kms, "roofline": roof,
            "e2e": {"value": entries / (e2e_ms * 1e-3), "unit": "entries/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches, "clocks": clk,
            "launch_geometry": comp.prefill_geometry(B, N) if tc else None}
    comp.close()
    line["chunked_prefill"] = bench_chunked(args, torch, csa, synthetic, device, peaks, world)
    line["other_prefill"] = [bench_prefill_workload(args, torch, csa, synthetic, device, peaks, world, wl)
                             for wl in (synthetic.HCA, synthetic.INDEXER, synthetic.PAIRS)]
    line["other_prefill"].append(bench_prefill_workload(args, torch, csa, synthetic, device, peaks, world,
                                                        synthetic.FLASH_CSA, gate_bias=True))
    if not args.no_long:
        line["long_prefill"] = bench_long(args, torch, csa, synthetic, device, peaks, world)
    if not args.no_decode:
        line["decode"] = bench_decode(args, torch, csa, synthetic, device, peaks, world, rank)
    return line


def measure_e2e(torch, comp, x, out, rows, K, stream, world, device, start_pos=0):
    """End to end through the public call with host buffers (pinned): every step copies its x in
    (H2D), runs the prefill and copies latent + codes + scales out (D2H), all inside the timed
    region.  As a serving loop would, the steps are pipelined: step i+1's input copy (split over two
    copy streams) runs while step i computes, and step i's outputs go back on a third stream; inputs
    and outputs are double-buffered.  Returns (ms per step, H2D bytes, D2H bytes per step)."""
    x_host = x.cpu().pin_memory()
    x_dev = [x, torch.empty_like(x)]
    outs2 = [out, comp._alloc_out(rows, device, prequant=False)]
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items() if v is not None}
    h2d_streams = [torch.cuda.Stream(device) for _ in range(2)]
    d2h_stream = torch.cuda.Stream(device)
    # the two halves of each input copy: along the batch when there are several sequences, else
    # along the tokens (each half one contiguous range)
    ax = 0 if x.shape[0] > 1 else 1
    half = x.shape[ax] // 2

    def e2e_steps(n):
        done = [None, None]  # compute of the step that last used buffer 0 / 1
        outs_done = [None, None]  # D2H of the step that last used output set 0 / 1
        for i in range(n):
            j = i % 2
            copied = []
            for part, cs in enumerate(h2d_streams):
                with torch.cuda.stream(cs):
                    if done[j] is not None:
                        cs.wait_event(done[j])
                    sl = slice(0, half) if part == 0 else slice(half, x.shape[ax])
                    if ax == 0:
                        x_dev[j][sl].copy_(x_host[sl], non_blocking=True)
                    else:
                        x_dev[j][:, sl].copy_(x_host[:, sl], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    copied.append(ev)
            for ev in copied:
                stream.wait_event(ev)
            if outs_done[j] is not None:
                stream.wait_event(outs_done[j])
            comp.prefill(x_dev[j], out=outs2[j], prequant=False, start_pos=start_pos)
            ev = torch.cuda.Event()
            ev.record(stream)
            done[j] = ev
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev)
                for k, h in host_out.items():
                    h.copy_(outs2[j][k], non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(d2h_stream)
                outs_done[j] = ev2
        for cs in h2d_streams + [d2h_stream]:
            stream.wait_stream(cs)

    e2e_steps(2)
    torch.cuda.synchronize()
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    e2e_ev[0].record(stream)
    for cs in h2d_streams + [d2h_stream]:
        cs.wait_stream(stream)
    e2e_steps(K)
    e2e_ev[1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2e_ev[0].elapsed_time(e2e_ev[1]), world, device) / K
    h2d = x.numel() * 2
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    return e2e_ms, h2d, d2h


def time_prefill(torch, comp, x, out, K, stream, flush, world, device, start_pos=0):
    """K prefill calls, each bracketed by CUDA events on the launching stream (ms per call, max over
    ranks) and by the library's events around its projection kernel (ms, mean); a buffer of twice the
    L2 is written between calls."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b_ in kev:  # torch creates an event on its first record; the library re-records it
        a.record(stream)
        b_.record(stream)
    launches0 = comp.kernel_launches()
    hold_gpu(flush)
    for i in range(K):
        flush.fill_(float(i))
        comp.set_profile_events(*kev[i])
        ev[i][0].record(stream)
        comp.prefill(x, out=out, prequant=False, start_pos=start_pos)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    comp.set_profile_events(None, None)
    ms = max_over_ranks(sum(a.elapsed_time(b_) for a, b_ in ev), world, device) / K
    kms = statistics.mean(a.elapsed_time(b_) for a, b_ in kev)
    return ms, kms, comp.kernel_launches() - launches0


def prefill_line(name, comp, layer, B, N, G, ms, kms, world, peaks):
    flops = 2.0 * B * N * layer.dim * 2 * layer.width
    achieved = flops / (kms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] / 3.0
    return {"workload": name, "value": B * G * world / (ms * 1e-3), "unit": "entries/s", "ms_per_step": ms,
            "tokens_per_s": B * N * world / (ms * 1e-3), "kernel_ms": kms, "tensor_cores": comp.uses_tensor_cores(),
            "launch_geometry": comp.prefill_geometry(B, N) if comp.uses_tensor_cores() else None,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak}}


def bench_prefill_workload(args, torch, csa, synthetic, device, peaks, world, wl, gate_bias=False):
    """Prefill throughput of another compressor instance of the model (same kernels): the HCA
    layer (ratio 128), the indexer's 128-wide compressor, the ratio-2 layers; or of the Flash CSA
    layer with a gate positional bias set (random, std 1).  With an end-to-end figure through host
    buffers and the oracle on the host cores beside it."""
    layer = wl.layers[0]
    B, N = wl.batch, wl.tokens[0]
    G = N // layer.ratio
    comp, x = make_inputs(torch, csa, synthetic, layer, wl.seed, B, N, 0, device, args)
    if gate_bias:
        ape = torch.randn(layer.ratio, layer.width, generator=torch.Generator().manual_seed(7)).to(device)
        comp.set_gate_bias(ape)
    out = comp._alloc_out(B * G, device, prequant=False)
    stream = torch.cuda.current_stream(device)
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(int(2 * getattr(props, "L2_cache_size", 128 << 20)) // 4 + 1, dtype=torch.float32,
                        device=device)
    for _ in range(max(args.warmup, 3)):
        comp.prefill(x, out=out, prequant=False)
    torch.cuda.synchronize()
    K = args.steps
    ms, kms, _ = time_prefill(torch, comp, x, out, K, stream, flush, world, device)
    name = wl.name + (", gate positional bias set" if gate_bias else "")
    line = prefill_line(name, comp, layer, B, N, G, ms, kms, world, peaks)
    e2e_ms, h2d, d2h = measure_e2e(torch, comp, x, out, B * G, min(K, 5), stream, world, device)
    line["e2e"] = {"value": B * G * world / (e2e_ms * 1e-3), "unit": "entries/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h}
    comp.close()
    if not args.no_cpu_baseline and not gate_bias:
        line["cpu_baseline"] = oracle_prefill_baseline(layer, wl.seed, B, N, min(N, 16 * 128 if layer.ratio == 128
                                                                                 else 2048))
    return line


def bench_long(args, torch, csa, synthetic, device, peaks, world):
    """The long-context prefill sweep: one sequence of 16384, 65536 and 131072 tokens through the
    ratio-4 overlapped (Flash CSA) and the ratio-128 (HCA) compressors, and a batch of 8 sequences of
    8192 tokens; 1% of the tokens are outliers (x20).  Each line times the prefill call (the inputs
    are larger than L2, which is also flushed between calls) with the oracle's per-token time on the
    host cores beside it (a prefix of 2048 tokens, extrapolated)."""
    wl = synthetic.LONG
    lines = []
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(int(2 * getattr(props, "L2_cache_size", 128 << 20)) // 4 + 1, dtype=torch.float32,
                        device=device)
    stream = torch.cuda.current_stream(device)
    cases = [(1, n) for n in wl.tokens] + [wl.extra["batched"]]
    cpu = {}
    comps = []
    for layer in wl.layers:
        comp = csa.Compressor(layer.dim, layer.head_dim, layer.ratio, layer.overlap, max_batch=8,
                              rope_dim=layer.rope_dim, fp4=layer.fp4)
        wkv, wgate, gain = synthetic.weights(wl.seed, layer)
        comp.set_weights(torch.from_numpy(wkv).to(device), torch.from_numpy(wgate).to(device),
                         torch.from_numpy(gain).to(device))
        comps.append(comp)
    for B, N in cases:
        # the tokens depend on the sequence and position only: one input serves both compressors
        x = torch.from_numpy(np.stack([synthetic.tokens(wl.seed, b, 0, N, wl.layers[0].dim, wl.outlier_frac,
                                                        wl.outlier_scale) for b in range(B)])) \
            .to(torch.bfloat16).to(device)
        for layer, comp in zip(wl.layers, comps):
            G = N // layer.ratio
            out = comp._alloc_out(B * G, device, prequant=False)
            for _ in range(3):
                comp.prefill(x, out=out, prequant=False)
            torch.cuda.synchronize()
            K = max(3, min(args.steps, 10 if B * N <= 65536 else 5))
            ms, kms, _ = time_prefill(torch, comp, x, out, K, stream, flush, world, device)
            name = (f"long-context prefill: B={B} N={N} dim={layer.dim} ratio={layer.ratio}"
                    f"{' overlapped' if layer.overlap else ''}, 1% outlier tokens x20")
            line = prefill_line(name, comp, layer, B, N, G, ms, kms, world, peaks)
            line["steps"] = K
            if not args.no_cpu_baseline:
                key = layer.ratio
                if key not in cpu:
                    cpu[key] = oracle_prefill_rate(layer, wl.seed, 2048, outlier_frac=wl.outlier_frac)
                dt, n = cpu[key]
                t_all = dt * (B * N) / 2048
                line["cpu_baseline"] = {"value": B * G / t_all, "unit": "entries/s", "cores": n, "kind": "oracle",
                                        "tokens_per_s": B * N / t_all, "extrapolated": True,
                                        "sample": f"prefill of a 2048-token prefix of sequence 0 "
                                                  f"({2048 // layer.ratio} entries), {dt:.2f} s on {n} threads, "
                                                  f"per-token time scaled to {B} x {N} tokens"}
            lines.append(line)
            del out
        del x
    for comp in comps:
        comp.close()
    return lines


def bench_chunked(args, torch, csa, synthetic, device, peaks, world):
    """A prefill chunk that continues a sequence: the Flash CSA layer, 4096 new tokens at position
    4098 (two tokens into a group, so the first two entries also pool candidates from the state).
    Every step is the same call on the same input; the state it reads is whatever the previous
    step left, which changes the values but not the work."""
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    B, N, p0 = 1, wl.tokens[0], wl.tokens[0] + 2
    comp, x = make_inputs(torch, csa, synthetic, layer, wl.seed, B, N, 0, device, args)
    G = (p0 + N) // layer.ratio - p0 // layer.ratio
    out = comp._alloc_out(B * G, device, prequant=False)
    stream = torch.cuda.current_stream(device)
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(int(2 * getattr(props, "L2_cache_size", 128 << 20)) // 4 + 1, dtype=torch.float32,
                        device=device)
    comp.prefill(torch.cat([x, x[:, :2]], dim=1), out=comp._alloc_out(B * (p0 // 4), device, False), prequant=False)

    def step():
        comp.prefill(x, out=out, prequant=False, start_pos=p0)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b_ in kev:
        a.record(stream)
        b_.record(stream)
    launches0 = comp.kernel_launches()
    hold_gpu(flush)
    for i in range(K):
        flush.fill_(float(i))
        comp.set_profile_events(*kev[i])
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    comp.set_profile_events(None, None)
    launches = comp.kernel_launches() - launches0
    ms = max_over_ranks(sum(a.elapsed_time(b_) for a, b_ in ev), world, device) / K
    kms = statistics.mean(a.elapsed_time(b_) for a, b_ in kev)
    flops = 2.0 * B * N * layer.dim * 2 * layer.width
    achieved = flops / (kms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] / 3.0
    geometry = comp.prefill_geometry(B, N, p0)
    comp.close()
    return {"workload": f"Flash CSA chunk: B={B}, {N} tokens at start_pos {p0} after a {p0}-token prefill",
            "value": B * G * world / (ms * 1e-3), "unit": "entries/s", "ms_per_step": ms, "steps": K,
            "tokens_per_s": B * N * world / (ms * 1e-3), "kernel_ms": kms, "gpu_launches": launches,
            "launch_geometry": geometry,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "kernel": "csa_prefill_tc (projection + fused pool, the carried candidates read from the state)"}}


def bench_decode(args, torch, csa, synthetic, device, peaks, world, rank):
    """B=128 decode steps through both compressors (ratio 4 overlapped + ratio 128), weights
    of several layer instances rotated so that each step streams its weights from HBM.  As in a
    model, every layer instance sees consecutive positions: step k runs layer k % L at position
    start + k // L, and the positions move on between graph replays."""
    wl = synthetic.DECODE
    B = wl.batch
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    w_bytes = sum(2 * L.width * L.dim * 4 for L in wl.layers)
    # at least 8 instances, and at least 2.5 x L2 of f32 weight bytes (the planes read are 1.5 x that)
    n_layers = args.decode_layers or max(8, math.ceil(2.5 * l2 / w_bytes))
    sp0 = synthetic.start_positions(wl.seed, B, wl.start_pos_hi)
    layers = []
    for li in range(n_layers):
        pair = []
        for L in wl.layers:
            Ls = synthetic.Layer(L.dim, L.head_dim, L.ratio, L.overlap, L.w_std, L.gate_scale, L.rope_dim, L.fp4,
                                 weight_stream=L.weight_stream + 2 * li)
            wkv, wgate, gain = synthetic.weights(wl.seed, Ls)
            c = csa.Compressor(L.dim, L.head_dim, L.ratio, L.overlap, max_batch=B)
            c.set_weights(torch.from_numpy(wkv).to(device), torch.from_numpy(wgate).to(device),
                          torch.from_numpy(gain).to(device))
            for b in range(B):
                s = int(sp0[b])
                t0 = csa.state_window_start(s, L.ratio, L.overlap)
                if s > t0:
                    xb = torch.from_numpy(synthetic.tokens(wl.seed, rank * B + b, t0, s, L.dim)).to(torch.bfloat16)
                    c.prefill(xb[None].to(device), slot_offset=b, prequant=False)
            outs = c._alloc_out(B, device, prequant=False)
            pair.append((c, outs))
        layers.append(pair)
    steps = n_layers * max(1, -(-(args.decode_steps or wl.decode_steps) // n_layers))
    xs = [torch.from_numpy(np.stack([synthetic.tokens(wl.seed, rank * B + b, int(sp0[b]) + k, int(sp0[b]) + k + 1,
                                                      wl.layers[0].dim)[0] for b in range(B)])).to(torch.bfloat16)
          .to(device) for k in range(8)]
    pos_all = torch.from_numpy(np.stack([(sp0 + k // n_layers).astype(np.int32) for k in range(steps)])).to(device)
    sps = [pos_all[k] for k in range(steps)]
    emitted = torch.empty(B, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(k):
        for c, outs in layers[k % n_layers]:
            c.decode(xs[k % 8], sps[k], out=outs, emitted=emitted, prequant=False)

    for k in range(n_layers):  # every layer once, at the first position
        step(k)
    pos_all += 1
    torch.cuda.synchronize()
    # The timed steps run as one captured CUDA graph (the library's decode calls allocate and
    # synchronise nothing once warmed up), so the measurement is of the GPU work rather than of
    # Python and driver launch overhead; eager launches are the fallback.
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(steps):
                step(k)
        graph.replay()
        torch.cuda.synchronize()
    except Exception:
        graph = None
        for k in range(steps):
            step(k)
        torch.cuda.synchronize()
    pos_all += steps // n_layers  # the timed steps continue where the warm-up stopped
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(steps):
            step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world, device) / steps
    # algorithmic bytes per step: both weight sets (f32), the two x_tok batches, the state slot
    # writes, the state read by emitting sequences (expected counts), the outputs
    wbytes = w_bytes
    xbytes = 2 * B * wl.layers[0].dim * 2
    slot_w = sum(B * 2 * L.width * 4 for L in wl.layers)
    emit_r = sum(B / L.ratio * (8 if L.overlap else L.ratio) * 2 * L.head_dim * 4 for L in wl.layers)
    outb = sum(B / L.ratio * (L.head_dim * 2 + L.head_dim // 2 + L.head_dim // 16) for L in wl.layers)
    alg = wbytes + xbytes + slot_w + emit_r + outb
    gbs = alg / (ms * 1e-3) / 1e9
    for pair in layers:
        for c, _ in pair:
            c.close()
    cpu = None if args.no_cpu_baseline or rank != 0 else oracle_decode_baseline(wl.seed)
    return {"steps_per_s": world / (ms * 1e-3) * 1.0, "ms_per_step": ms, "batch": B, "layers_rotated": n_layers,
            "cpu_baseline": cpu,
            "launch": "cuda graph" if graph is not None else "eager",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("decode_tc_batched", "traffic_bytes_per_step"),
                         "algorithmic_bytes_per_step": alg}}


# ---------------------------------------------------------------------------------------------
# The CPU oracle as it stands, timed on the host cores (a reported baseline, not a target).

def oracle_prefill_rate(layer, seed, ntok, nthreads=None, outlier_frac=0.0):
    """Seconds the oracle takes for a prefill of the first `ntok` tokens of sequence 0 of a workload
    (a prefix of whole groups), and the threads it used."""
    import torch

    import oracle
    import synthetic
    x = synthetic.tokens(seed, 0, 0, ntok, layer.dim, outlier_frac)
    xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[None]
    wkv, wgate, gain = synthetic.weights(seed, layer)
    o = oracle.Compressor(layer.dim, layer.head_dim, layer.ratio, layer.overlap, rope_dim=layer.rope_dim,
                          fp4=layer.fp4)
    o.set_weights(wkv, wgate, gain)
    n = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    o.prefill(xb, nthreads=n)
    return time.perf_counter() - t0, n


def oracle_prefill_baseline(layer, seed, B, N, prefix, outlier_frac=0.0):
    """cpu_baseline of a prefill workload of B sequences of N tokens from a prefix of `prefix` tokens
    (whole groups) of one sequence: the oracle's per-token time, extrapolated to the workload."""
    dt, n = oracle_prefill_rate(layer, seed, prefix, outlier_frac=outlier_frac)
    G = N // layer.ratio
    t_all = dt * (B * N) / prefix
    return {"value": B * G / t_all, "unit": "entries/s", "cores": n, "kind": "oracle",
            "tokens_per_s": B * N / t_all, "extrapolated": prefix < B * N,
            "sample": f"prefill of a {prefix}-token prefix of one sequence ({prefix // layer.ratio} entries), "
                      f"{dt:.2f} s on {n} threads, per-token time scaled to {B} x {N} tokens"}


def oracle_decode_baseline(seed, steps=2):
    """cpu_baseline of the batched decode workload: whole steps (128 sequences through both
    compressors) of the oracle at the workload's positions.  The oracle starts from a fresh state:
    the work of a step does not depend on the state's values."""
    import torch

    import oracle
    import synthetic
    wl = synthetic.DECODE
    B = wl.batch
    sp0 = synthetic.start_positions(wl.seed, B, wl.start_pos_hi)
    comps = []
    for L in wl.layers:
        wkv, wgate, gain = synthetic.weights(wl.seed, L)
        o = oracle.Compressor(L.dim, L.head_dim, L.ratio, L.overlap, max_batch=B, rope_dim=L.rope_dim, fp4=L.fp4)
        o.set_weights(wkv, wgate, gain)
        comps.append(o)
    n = oracle.default_threads()
    xs = [torch.from_numpy(np.stack([synthetic.tokens(wl.seed, b, int(sp0[b]) + k, int(sp0[b]) + k + 1,
                                                      wl.layers[0].dim)[0] for b in range(B)]))
          .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for k in range(steps)]
    t0 = time.perf_counter()
    for k in range(steps):
        for o in comps:
            o.decode(xs[k], (sp0 + k).astype(np.int32), nthreads=n)
    dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": "steps/s", "cores": n, "kind": "oracle",
            "sample": f"{steps} whole steps (B={B}, both compressors), {dt:.2f} s on {n} threads"}


class OracleArm:
    """The CPU oracle, as it stands, on the Flash CSA prefill workload: one step is the whole
    4096-token sequence (1024 entries), on all host cores."""

    def __init__(self):
        import torch

        import oracle
        import synthetic
        wl = synthetic.FLASH_CSA
        layer = wl.layers[0]
        self.N = wl.tokens[0]
        x = synthetic.tokens(wl.seed, 0, 0, self.N, layer.dim)
        self.x = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[None]
        wkv, wgate, gain = synthetic.weights(wl.seed, layer)
        self.o = oracle.Compressor(layer.dim, layer.head_dim, 4, 1, rope_dim=64, fp4=1)
        self.o.set_weights(wkv, wgate, gain)
        self.cores = oracle.default_threads()

    def step(self):
        t0 = time.perf_counter()
        r = self.o.prefill(self.x, nthreads=self.cores)
        return r["G"], time.perf_counter() - t0


def oracle_sample():
    arm = OracleArm()
    g, dt = arm.step()
    return {"value": g / dt, "unit": "entries/s", "cores": arm.cores, "kind": "oracle",
            "sample": f"the whole workload: {g} entries ({arm.N} tokens), {dt:.2f} s on {arm.cores} threads"}


def oracle_single_thread():
    """The same oracle on one host thread, on a 256-token prefix of the Flash CSA workload."""
    import synthetic
    wl = synthetic.FLASH_CSA
    layer = wl.layers[0]
    dt, n = oracle_prefill_rate(layer, wl.seed, 256, nthreads=1)
    return {"value": (256 // layer.ratio) / dt, "unit": "entries/s", "cores": 1, "kind": "oracle",
            "sample": f"prefill of a 256-token prefix (64 entries) of the Flash CSA workload, {dt:.2f} s on 1 thread"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    arm = OracleArm()
    for _ in range(args.warmup):
        arm.step()
    times = []
    g = 0
    for _ in range(args.steps):
        g, dt = arm.step()
        times.append(dt)
    ms = 1e3 * statistics.mean(times)
    val = g / (ms * 1e-3)
    cpu = {"value": val, "unit": "entries/s", "cores": arm.cores, "kind": "oracle",
           "sample": f"the whole workload per step: {g} entries ({arm.N} tokens) on {arm.cores} threads"}
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "entries/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": arm.N, "entries_per_step": g,
                       "l2": "not applicable: the oracle runs on the host cores",
                       "parallelism": f"host threads x{arm.cores}"}, "cpu_baseline": cpu,
            "e2e": {"value": val, "unit": "entries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
        # each step is a few seconds of CPU work: keep the whole run within a few minutes
        args.steps = max(1, min(args.steps, 30))
        args.warmup = min(args.warmup, 3)
        line = run_reference(args, rank, world)
        if line:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.decode_only:
        import torch

        import deepseek_v4_compressed_wkv_gb300 as csa
        import synthetic
        torch.cuda.set_device(local)
        d = bench_decode(args, torch, csa, synthetic, torch.device("cuda", local), load_peaks(), world, rank)
        if rank == 0:
            print(json.dumps({"decode": d}), flush=True)
        return
    if args.other_only:
        import torch

        import deepseek_v4_compressed_wkv_gb300 as csa
        import synthetic
        torch.cuda.set_device(local)
        wl = {"hca": synthetic.HCA, "indexer": synthetic.INDEXER, "pairs": synthetic.PAIRS}[args.other_only]
        o = bench_prefill_workload(args, torch, csa, synthetic, torch.device("cuda", local), load_peaks(), world, wl)
        if rank == 0:
            print(json.dumps({"other_prefill": [o]}), flush=True)
        return
    line = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_sample()
            line["cpu_baseline_single_thread"] = oracle_single_thread()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
