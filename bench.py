#!/usr/bin/env python3
"""Benchmark of the causal differential-attention forward on GB300.

One step = one fused DIFF V1 forward (lambda, both causal attentions, the
combine, RMSNorm and the (1 - lam_init) scale -- every step of the V1 path)
over the workload B=4, T=2048, 16 diff heads, d=64, dv=128, layer_index=12,
bf16 inputs drawn N(0,1) with a seeded generator.  The line also carries, as
auxiliary measurements, DIFF V2 prefill (B=8, T=4096, Hq=32, Hkv=8, D=128,
TFLOP/s), long-context DIFF V1 (B=1, T=32768, 12 heads, d=128, TFLOP/s),
DIFF V2 decode (B=64, L=32768, Hq=64, Hkv=8, D=128, HBM GB/s), the same decode
with per-sequence cache lengths uniform on 1..L, DIFF V1 decode (B=32,
L=16384, 12 heads, d=128, HBM GB/s), and the backward (training) pass of the
V1 headline and V2 prefill workloads (TFLOP/s), and the prologue (rotary q,
k and the projected V2 lambda, HBM GB/s).

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own batch of the same workload
(seed + rank), no collective on the data path; timing is max over ranks.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from differential_attention_causal_gb300 import inputs  # noqa: E402

HEADLINE = "v1_bf16_B4_T2048_H16_d64"
METRIC = "fused diff-attn fwd TFLOP/s (% bf16 TC peak); V2 decode HBM GB/s (% peak)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
SPINUP_S = 0.3

# DRAM traffic per launch from an ncu capture, valid only for the kernel source
# it was taken on (sha256 of the .cu file, first 16 hex digits).
TRAFFIC_RECORDS: dict = {
    # profiles/prefill_onepass_v1_B4_T2048_H16_d64.md: dram__bytes_read.sum + dram__bytes_write.sum
    "prefill_v1_d64": {"src_sha": "9d7bf7215e00e1fe", "bytes_per_launch": 127620608 + 10393600},
}


# ----------------------------------------------------------------- helpers

def v1_flops(s) -> float:
    """Algorithmic FLOPs of one DIFF V1 forward: per causal (query, key) pair
    2d (S1) + 2d (S2) + 2*2d (P1 V) + 2*2d (P2 V) = 12d; pairs = T(T+1)/2."""
    return float(s.B) * s.H * s.T * (s.T + 1) / 2 * 12 * s.d


def v2_flops(s) -> float:
    """DIFF V2 prefill: per query head and causal pair 2D (QK) + 2D (PV)."""
    return float(s.B) * s.Hq * s.T * (s.T + 1) / 2 * 4 * s.D


def paired_flops(s) -> float:
    """Paired Head Attention: one causal attention per head pair over the
    interleaved 2T positions: per causal (query, key) position pair 2D (QK)
    + 2D (PV); pairs per head pair = 2T (2T + 1) / 2."""
    return float(s.B) * (s.H // 2) * (2 * s.T) * (2 * s.T + 1) / 2 * 4 * s.D


def v1_bwd_flops(s) -> float:
    """Algorithmic FLOPs of the DIFF V1 backward: two attention backwards, each
    per causal pair 2d (S recomputed) + 2*2d (dP) + 2*2d (dV) + 2d (dK) + 2d
    (dQ) = 14d; 28d per pair."""
    return float(s.B) * s.H * s.T * (s.T + 1) / 2 * 28 * s.d


def v2_bwd_flops(s) -> float:
    """DIFF V2 backward: per query head and causal pair 2D (S) + 2D (dP) + 2D
    (dV) + 2D (dK) + 2D (dQ) = 10D."""
    return float(s.B) * s.Hq * s.T * (s.T + 1) / 2 * 10 * s.D


def decode_bytes(s) -> int:
    """Bytes one decode must move: K and V caches once, q, lam, out."""
    return (2 * s.B * s.L * s.Hkv * s.D * 2 + s.B * s.Hq * s.D * 2
            + s.B * (s.Hq // 2) * 4 + s.B * (s.Hq // 2) * s.D * 2)


def decode_varlen_bytes(s, lens) -> int:
    """Bytes a decode with per-sequence lengths must move: each sequence's
    first len_b cache rows of K and V, q, lam, out and the lengths."""
    rows = int(sum(int(n) for n in lens))
    return (2 * rows * s.Hkv * s.D * 2 + s.B * s.Hq * s.D * 2
            + s.B * (s.Hq // 2) * 4 + s.B * (s.Hq // 2) * s.D * 2 + s.B * 4)


def v1_decode_bytes(s, lens=None) -> int:
    """Bytes one DIFF V1 decode must move: k1, k2 (d) and v (2d) cache rows
    attended, q1, q2, out (2d) and the four lambda vectors."""
    rows = s.B * s.L if lens is None else int(sum(int(n) for n in lens))
    return (rows * s.H * 4 * s.d * 2 + 2 * s.B * s.H * s.d * 2 + s.B * s.H * 2 * s.d * 2
            + 4 * s.d * 4 + (0 if lens is None else s.B * 4))


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def src_sha(rel: str) -> str:
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index, self.period = index, period_ms
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
            time.sleep(0.5)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        busy = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, steps: int, world: int, max_ms: float, scale: float = 1e12) -> float:
    """Whole-job rate: every rank processes its own batch (weak scaling), so the
    work done is units_per_step * steps * world in the slowest rank's time."""
    return units_per_step * steps * world / (max_ms * 1e-3) / scale


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch of the workload."""
    return seed + rank


# NVTX: every timed step runs inside a range named after the measurement it
# belongs to (set with section()), so a timeline profiler shows which launches
# each number covers.  Without a profiler attached the ranges cost nothing.
_SECTION = "bench"


def section(name: str) -> None:
    global _SECTION
    _SECTION = name


def time_steps(step, steps: int, flush: torch.Tensor | None):
    """Per-step device time (ms) with CUDA events on the current stream; the
    L2 flush (if any) runs between steps, outside the events."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (a, b) in enumerate(evs):
        if flush is not None:
            flush.add_(1)
        torch.cuda.nvtx.range_push(f"{_SECTION}: timed step {i}")
        a.record()
        step()
        b.record()
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


# ------------------------------------------------------------- our arm

def run_ours(args, rank: int, world: int, dev: torch.device) -> dict | None:
    from differential_attention_causal_gb300 import binding
    import torch.distributed as dist

    peaks, peak_kind = load_peaks()
    s = inputs.WORKLOADS[HEADLINE]
    x = inputs.make_v1(s, seed=rank_seed(args.seed, rank), device=dev)
    out = torch.empty((s.B, s.T, s.H, 2 * s.d), dtype=torch.bfloat16, device=dev)
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def launch():
        binding.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"],
                       x["lam_k2"], s.layer_index, out=out)

    # The step is one C-ABI call; it is captured once into a CUDA graph and
    # replayed, so that the host-side argument checks and tensor-map encoding
    # of the call (tens of microseconds against a ~0.1 ms kernel) never leave
    # the GPU idle inside a timed step.  The graph holds exactly the call's
    # one kernel launch.
    launch()                       # first call: per-device set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launch()
    launches_per_step = binding.last_launch_count()

    def step():
        graph.replay()

    # Clock spin-up: an idle GPU starts below its maximum SM clock and takes a
    # fraction of a second under load to reach it; the step runs untimed for
    # SPINUP_S seconds before the W warm-up steps so that the K timed steps
    # see steady clocks (recorded in config).
    t_end = time.perf_counter() + SPINUP_S
    while time.perf_counter() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        flush.add_(1)
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    section(f"headline {HEADLINE}")
    times = time_steps(step, args.steps, flush)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(times), world, dev)
    if binding.device_error():
        raise RuntimeError("a kernel reported a device-side wait timeout")
    flops = v1_flops(s)
    value = job_throughput(flops, args.steps, world, total_ms)
    avg_ms = sum(times) / len(times)
    med_ms, min_ms = statistics.median(times), min(times)
    tokens_per_s = s.B * s.T * args.steps * world / (total_ms * 1e-3)
    achieved = flops / (avg_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    tr = TRAFFIC_RECORDS.get("prefill_v1_d64")
    traffic = tr["bytes_per_launch"] if tr and tr["src_sha"] == src_sha(
        "differential_attention_causal_gb300/csrc/k_prefill.cu") else None

    # end to end through the C-ABI call on host buffers (diffattn_v1_fwd_host): the
    # pinned H2D of the step's inputs, the forward and the D2H of the result, all
    # inside the events; the call overlaps them chunk by chunk of batch entries.
    host = {k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in x.items()
            if k in ("q", "k", "v", "lam_q1", "lam_k1", "lam_q2", "lam_k2")}
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws_host = torch.empty(binding.v1_fwd_host_workspace_size(s.B, s.T, s.H, s.d), dtype=torch.uint8, device=dev)

    def e2e_step():
        binding.v1_fwd_host(host["q"], host["k"], host["v"], host["lam_q1"], host["lam_k1"], host["lam_q2"],
                            host["lam_k2"], s.layer_index, hout, ws_host)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(5, min(args.steps, 50))
    section("e2e diffattn_v1_fwd_host")
    et = time_steps(e2e_step, e2e_steps, flush)
    h2d = sum(host[n].numel() * host[n].element_size() for n in host)
    d2h = hout.numel() * hout.element_size()
    e2e_ms = max_over_ranks(sum(et) / len(et), world, dev)
    e2e_val = job_throughput(flops, 1, world, e2e_ms)

    aux = {} if args.no_aux else run_aux(args, dev, peaks, peak_kind, binding)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "ms_per_step_median": round(med_ms, 5), "ms_per_step_min": round(min_ms, 5),
        "tokens_per_s": round(tokens_per_s), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, N(0,0.1) lambda vectors; seed + rank per rank)",
        "config": {"workload": HEADLINE, "B": s.B, "T": s.T, "H": s.H, "d": s.d, "dv": 2 * s.d,
                   "layer_index": s.layer_index, "causal": True,
                   "l2": "256 MiB buffer written between timed steps (flush)",
                   "spinup": f"the step run untimed for {SPINUP_S} s before the warm-up steps (clock ramp)",
                   "launch": "the C-ABI call captured once into a CUDA graph (one kernel) and replayed per step",
                   "flop_count": "12d per causal pair (two QK, two PV)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"bf16 dense burst ({peak_kind})", "kernel": "prefill_onepass<64,128,V1>"},
        "e2e": {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if aux:
        line["aux"] = aux
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, s, out, dev, budget_s=args.cpu_seconds, seed=args.seed,
                                            per_config=not args.no_aux)
    return line


def run_aux(args, dev, peaks, peak_kind, binding) -> dict:
    aux = {}
    flush = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    section("aux v1_fp32_tiny")
    # DIFF V1 fp32, the tiny parity workload: a latency figure (fp32 on CUDA cores), no roofline claim
    s = inputs.WORKLOADS["v1_fp32_B1_T64_H2_d32"]
    x = inputs.make_v1(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.T, s.H, 2 * s.d), dtype=torch.float32, device=dev)
    f = lambda: binding.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"],  # noqa
                               x["lam_q2"], x["lam_k2"], s.layer_index, out=out)
    for _ in range(10):
        f()
    t = time_steps(f, 100, None)
    # the same call captured in a CUDA graph: the kernel without the host-side call overhead
    f()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        f()
    for _ in range(10):
        graph.replay()
    tg = time_steps(graph.replay, 100, None)
    aux["v1_fp32_tiny"] = {"workload": "v1_fp32_B1_T64_H2_d32", "ms_median": round(statistics.median(t), 5),
                           "ms_min": round(min(t), 5), "kernel_ms_median": round(statistics.median(tg), 5),
                           "launches": 1,
                           "note": "fp32 on CUDA cores; ms_*: the C-ABI call (host checks included), "
                                   "kernel_ms: replayed from a CUDA graph; latency-bound, no roofline claim"}
    del x, out
    section("aux v2_prefill")
    # DIFF V2 prefill
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.T, s.Hq // 2, s.D), dtype=torch.bfloat16, device=dev)
    f = lambda: binding.v2_fwd(x["q"], x["k"], x["v"], x["lam"], out=out)  # noqa: E731
    for _ in range(3):
        f()
    t = time_steps(f, 10, flush)
    ms = sum(t) / len(t)
    tf = v2_flops(s) / (ms * 1e-3) / 1e12
    aux["v2_prefill"] = {"workload": "v2_bf16_B8_T4096_Hq32_Hkv8_D128", "ms": round(ms, 4),
                         "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                         "tokens_per_s": round(s.B * s.T / (ms * 1e-3)), "peak_kind": peak_kind}
    del x, out
    section("aux v1_long")
    # DIFF V1 long context, d = 128 / dv = 256 (two-pass kernel)
    s = inputs.WORKLOADS["v1_bf16_B1_T32768_H12_d128"]
    x = inputs.make_v1(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.T, s.H, 2 * s.d), dtype=torch.bfloat16, device=dev)
    f = lambda: binding.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"],  # noqa
                               x["lam_q2"], x["lam_k2"], s.layer_index, out=out)
    for _ in range(3):
        f()
    t = time_steps(f, 5, flush)
    ms = sum(t) / len(t)
    tf = v1_flops(s) / (ms * 1e-3) / 1e12
    aux["v1_long"] = {"workload": "v1_bf16_B1_T32768_H12_d128", "ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                      "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                      "tokens_per_s": round(s.B * s.T / (ms * 1e-3)), "kernel": "prefill_v1_twopass<128>",
                      "peak_kind": peak_kind}
    del x, out
    section("aux v2_decode")
    # DIFF V2 decode (8.6 GB cache >> L2: no flush needed)
    s = inputs.WORKLOADS["v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128"]
    x = inputs.make_decode(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.Hq // 2, s.D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(binding.decode_workspace_size(s.B, s.L, s.Hq, s.Hkv, s.D), dtype=torch.uint8, device=dev)
    f = lambda: binding.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"], out=out, workspace=ws)  # noqa
    for _ in range(3):
        f()
    t = time_steps(f, 20, None)
    ms = sum(t) / len(t)
    gbs = decode_bytes(s) / (ms * 1e-3) / 1e9
    aux["v2_decode"] = {"workload": "v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128", "ms": round(ms, 4),
                        "GB/s": round(gbs, 1), "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                        "frac_8TBs": round(gbs / 8000.0, 4), "tokens_per_s": round(s.B / (ms * 1e-3)),
                        "launches": 2, "peak_kind": peak_kind}
    del x, out, ws
    torch.cuda.empty_cache()
    section("aux v2_decode_varlen")
    # DIFF V2 decode, per-sequence lengths uniform on 1..L (the same cache allocation)
    s = inputs.WORKLOADS["v2_decode_varlen_bf16_B64_L32768_Hq64_Hkv8_D128"]
    x = inputs.make_decode(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.Hq // 2, s.D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(binding.decode_workspace_size(s.B, s.L, s.Hq, s.Hkv, s.D), dtype=torch.uint8, device=dev)
    f = lambda: binding.v2_decode_varlen(x["q"], x["k_cache"], x["v_cache"], x["lam"], x["cache_lens"],  # noqa
                                         out=out, workspace=ws)
    for _ in range(3):
        f()
    t = time_steps(f, 20, flush)
    ms = sum(t) / len(t)
    lens = x["cache_lens"].cpu().tolist()
    gbs = decode_varlen_bytes(s, lens) / (ms * 1e-3) / 1e9
    aux["v2_decode_varlen"] = {"workload": "v2_decode_varlen_bf16_B64_L32768_Hq64_Hkv8_D128", "ms": round(ms, 4),
                               "cached_rows": int(sum(lens)), "GB/s": round(gbs, 1),
                               "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                               "tokens_per_s": round(s.B / (ms * 1e-3)), "launches": 3, "l2_flush": True,
                               "peak_kind": peak_kind}
    del x, out, ws
    torch.cuda.empty_cache()
    section("aux v1_decode")
    # DIFF V1 decode, d = 128 (6.4 GB of k1, k2, v cache >> L2)
    s = inputs.WORKLOADS["v1_decode_bf16_B32_L16384_H12_d128"]
    x = inputs.make_v1_decode(s, seed=args.seed, device=dev)
    out = torch.empty((s.B, s.H, 2 * s.d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(binding.v1_decode_workspace_size(s.B, s.L, s.H, s.d), dtype=torch.uint8, device=dev)
    f = lambda: binding.v1_decode(x["q1"], x["q2"], x["k1_cache"], x["k2_cache"], x["v_cache"],  # noqa
                                  x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"], s.layer_index,
                                  out=out, workspace=ws)
    for _ in range(3):
        f()
    t = time_steps(f, 20, None)
    ms = sum(t) / len(t)
    gbs = v1_decode_bytes(s) / (ms * 1e-3) / 1e9
    aux["v1_decode"] = {"workload": "v1_decode_bf16_B32_L16384_H12_d128", "ms": round(ms, 4),
                        "GB/s": round(gbs, 1), "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                        "tokens_per_s": round(s.B / (ms * 1e-3)), "launches": 2, "peak_kind": peak_kind}
    del x, out, ws
    torch.cuda.empty_cache()
    section("aux prologue")
    # prologue (rotary q, k in place + projected lambda) on the V2 prefill workload
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=args.seed, device=dev)
    C, P = (s.Hq // 2) * s.D, s.Hq // 2
    lp = inputs.make_lambda_proj(s.B, s.T, C, P, "bf16", seed=args.seed, device=dev)
    lam = torch.empty((s.B, s.T, P), dtype=torch.float32, device=dev)
    f = lambda: binding.prologue(q=x["q"], k=x["k"], x=lp["x"], w_lam=lp["w_lam"], lam=lam)  # noqa: E731
    for _ in range(3):
        f()
    ms = sum(t := time_steps(f, 10, flush)) / len(t)
    nbytes = 2 * (x["q"].numel() + x["k"].numel()) * 2 + lp["x"].numel() * 2 + lp["w_lam"].numel() * 2 + lam.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    aux["prologue"] = {"workload": "v2_bf16_B8_T4096_Hq32_Hkv8_D128, x (B,T,2048), w (2048,16)", "ms": round(ms, 4),
                       "GB/s": round(gbs, 1), "frac_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
                       "bytes": int(nbytes), "launches": 2, "peak_kind": peak_kind}
    section("aux v2_prefill_with_prologue")
    # the V2 attention call with its prologue, two ways: rotary q, k + lambda
    # logits, then the prefill (3 launches), against lambda logits, then the
    # prefill with q rotated tile by tile inside it (k + table, prefill: 3 launches)
    out = torch.empty((s.B, s.T, s.Hq // 2, s.D), dtype=torch.bfloat16, device=dev)

    def two_call():
        binding.prologue(q=x["q"], k=x["k"], x=lp["x"], w_lam=lp["w_lam"], lam=lam)
        binding.v2_fwd(x["q"], x["k"], x["v"], lam, out=out)

    def fused():
        binding.prologue(x=lp["x"], w_lam=lp["w_lam"], lam=lam)
        binding.v2_fwd_rope(x["q"], x["k"], x["v"], lam, out=out)

    res = {}
    for name, fn in (("two_call", two_call), ("fused", fused)):
        for _ in range(3):
            fn()
        t = time_steps(fn, 10, flush)
        res[name] = (sum(t) / len(t), statistics.median(t))
    tf = v2_flops(s) / (res["fused"][1] * 1e-3) / 1e12
    aux["v2_prefill_with_prologue"] = {
        "workload": "v2_bf16_B8_T4096_Hq32_Hkv8_D128, x (B,T,2048), w (2048,16)",
        "two_call_ms": round(res["two_call"][0], 4), "two_call_ms_median": round(res["two_call"][1], 4),
        "fused_ms": round(res["fused"][0], 4), "fused_ms_median": round(res["fused"][1], 4),
        "saved_ms_median": round(res["two_call"][1] - res["fused"][1], 4),
        "fused_attention_TFLOP/s_incl_prologue": round(tf, 1), "launches": 3,
        "note": "two_call: prologue (rotary q, k; lambda logits) + v2_fwd; fused: lambda logits + "
                "v2_fwd_rope (rotary k, then the prefill rotating each Q tile in shared memory)"}
    del x, lp, lam, out
    torch.cuda.empty_cache()
    section("aux paired_prefill")
    # Paired Head Attention (interleaved head pairs, one causal softmax) on the V2 prefill's query heads
    s = inputs.WORKLOADS["paired_bf16_B8_T4096_H32_D128"]
    x = inputs.make_paired(s, seed=args.seed, device=dev)
    out = torch.empty_like(x["q"])
    f = lambda: binding.paired_fwd(x["q"], x["k"], x["v"], out=out)  # noqa: E731
    for _ in range(3):
        f()
    ms = sum(t := time_steps(f, 10, flush)) / len(t)
    tf = paired_flops(s) / (ms * 1e-3) / 1e12
    aux["paired_prefill"] = {"workload": "paired_bf16_B8_T4096_H32_D128", "ms": round(ms, 4),
                             "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                             "flop_count": "4D per head pair and causal pair of the 2T interleaved positions",
                             "launches": 1, "peak_kind": peak_kind}
    del x, out
    torch.cuda.empty_cache()
    section("aux backward")
    # backward (training): DIFF V1 on the headline workload, DIFF V2 on the prefill workload
    s = inputs.WORKLOADS[HEADLINE]
    x = inputs.make_v1(s, seed=args.seed, device=dev)
    dout = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=args.seed, device=dev)
    a = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"],
         s.layer_index)
    _, saved = binding.v1_fwd_train(*a)
    ws = torch.empty(binding.lib().diffattn_v1_bwd_workspace_size(s.B, s.T, s.H, s.d, 1), dtype=torch.uint8,
                     device=dev)
    f = lambda: binding.v1_bwd(*a, dout, saved, workspace=ws)  # noqa: E731
    for _ in range(3):
        f()
    ms = sum(t := time_steps(f, 10, flush)) / len(t)
    ftr = lambda: binding.v1_fwd_train(*a)  # noqa: E731
    ms_ft = sum(t := time_steps(ftr, 10, flush)) / len(t)
    tf = v1_bwd_flops(s) / (ms * 1e-3) / 1e12
    aux["v1_backward"] = {"workload": HEADLINE, "ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                          "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                          "flop_count": "28d per causal pair (two attention backwards)",
                          "fwd_train_ms": round(ms_ft, 4), "launches": 4, "peak_kind": peak_kind}
    del x, dout, saved, ws
    section("aux v1_long_backward")
    # backward of the long-context DIFF V1 workload (d = 128, dv = 256: split kernels)
    s = inputs.WORKLOADS["v1_bf16_B1_T32768_H12_d128"]
    x = inputs.make_v1(s, seed=args.seed, device=dev)
    dout = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=args.seed, device=dev)
    a = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"],
         s.layer_index)
    _, saved = binding.v1_fwd_train(*a)
    ws = torch.empty(binding.lib().diffattn_v1_bwd_workspace_size(s.B, s.T, s.H, s.d, 1), dtype=torch.uint8,
                     device=dev)
    f = lambda: binding.v1_bwd(*a, dout, saved, workspace=ws)  # noqa: E731
    for _ in range(2):
        f()
    ms = sum(t := time_steps(f, 3, flush)) / len(t)
    ftr = lambda: binding.v1_fwd_train(*a)  # noqa: E731
    ms_ft = sum(t := time_steps(ftr, 3, flush)) / len(t)
    tf = v1_bwd_flops(s) / (ms * 1e-3) / 1e12
    aux["v1_long_backward"] = {"workload": "v1_bf16_B1_T32768_H12_d128", "ms": round(ms, 3), "TFLOP/s": round(tf, 1),
                               "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                               "flop_count": "28d per causal pair (two attention backwards)",
                               "fwd_train_ms": round(ms_ft, 3), "launches": 5, "peak_kind": peak_kind}
    del x, dout, saved, ws
    torch.cuda.empty_cache()
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    x = inputs.make_v2(s, seed=args.seed, device=dev)
    dout = inputs.make_grad_out((s.B, s.T, s.Hq // 2, s.D), "bf16", seed=args.seed, device=dev)
    _, saved = binding.v2_fwd_train(x["q"], x["k"], x["v"], x["lam"])
    ws = torch.empty(binding.lib().diffattn_v2_bwd_workspace_size(s.B, s.T, s.Hq, s.Hkv, s.D, 1), dtype=torch.uint8,
                     device=dev)
    f = lambda: binding.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout, saved, workspace=ws)  # noqa: E731
    for _ in range(3):
        f()
    ms = sum(t := time_steps(f, 5, flush)) / len(t)
    ftr = lambda: binding.v2_fwd_train(x["q"], x["k"], x["v"], x["lam"])  # noqa: E731
    ms_ft = sum(t := time_steps(ftr, 5, flush)) / len(t)
    tf = v2_bwd_flops(s) / (ms * 1e-3) / 1e12
    aux["v2_backward"] = {"workload": "v2_bf16_B8_T4096_Hq32_Hkv8_D128", "ms": round(ms, 4),
                          "TFLOP/s": round(tf, 1), "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                          "flop_count": "10D per query head and causal pair", "fwd_train_ms": round(ms_ft, 4),
                          "launches": 3, "peak_kind": peak_kind}
    del x, dout, saved, ws
    torch.cuda.empty_cache()
    if binding.device_error():
        raise RuntimeError("a kernel reported a device-side wait timeout")
    return aux


# ------------------------------------------------------ the oracle (CPU)

def _oracle_inputs(x) -> dict:
    """fp64 contiguous host copies of the V1 inputs (done once, outside any timing)."""
    import numpy as np
    out = {}
    for k in ("q1", "q2", "k1", "k2", "v", "lam_q1", "lam_k1", "lam_q2", "lam_k2"):
        out[k] = np.ascontiguousarray(x[k].detach().to("cpu").double().numpy())
    return out


def _oracle_rows_time(x_cpu, s, rows) -> float:
    return _oracle_rows(x_cpu, s, rows)[0]


def _oracle_rows(x_cpu, s, rows):
    """(wall seconds, output rows) of the V1 oracle on the listed rows."""
    import oracle
    t0 = time.perf_counter()
    y = oracle.v1_fwd(x_cpu["q1"], x_cpu["q2"], x_cpu["k1"], x_cpu["k2"], x_cpu["v"], x_cpu["lam_q1"],
                      x_cpu["lam_k1"], x_cpu["lam_q2"], x_cpu["lam_k2"], s.layer_index, rows=rows)
    return time.perf_counter() - t0, y


def _rows_flops(rows, s) -> float:
    import numpy as np
    t = (np.asarray(rows) // s.H) % s.T
    return float(((t + 1) * 12 * s.d).sum())


def cpu_baseline(x, s, out, dev, budget_s: float = 15.0, seed: int = 0, per_config: bool = True) -> dict:
    """Time the fp64 oracle on a bounded random sample of the headline rows,
    compare those rows with the timed GPU output, and time the oracle on the
    other workloads (in full where it finishes in seconds, else on a stated
    sample with the fraction of the causal work it covers)."""
    import numpy as np
    import oracle
    oracle.build()
    x_cpu = _oracle_inputs(x)
    rng = np.random.default_rng(seed)
    nall = s.B * s.T * s.H
    probe = rng.choice(nall, size=min(512, nall), replace=False)
    dt = _oracle_rows_time(x_cpu, s, probe)
    per_row = dt / len(probe)          # random rows: their mean cost is the workload's mean
    n = int(min(nall, max(len(probe), budget_s / max(per_row, 1e-9))))
    rows = rng.choice(nall, size=n, replace=False)
    dt, ref = _oracle_rows(x_cpu, s, rows)
    val = _rows_flops(rows, s) / dt / 1e12
    got = out.reshape(-1, 2 * s.d)[torch.from_numpy(rows).to(out.device)].double().cpu().numpy()
    err = float(np.abs(got - ref).max())
    rl2 = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    res = {"value": val, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
           "sample": f"{n} of {nall} output rows (b, t, head) of {HEADLINE}, uniform without replacement; "
                     f"{dt:.1f} s wall; value = algorithmic 12d-per-pair FLOPs of the sample / wall time",
           "headline_parity": {"rows": n, "max_abs": err, "rel_l2": rl2, "bound": "max abs <= 2e-2, rel L2 <= 5e-3",
                               "ok": bool(err <= 2e-2 and rl2 <= 5e-3),
                               "what": "the timed step's output against the oracle on the sampled rows"}}
    if per_config:
        res["configs"] = oracle_per_config(dev, seed)
    return res


def oracle_per_config(dev, seed: int) -> dict:
    """The fp64 oracle timed on the other workloads, on this host's cores."""
    import numpy as np
    import oracle
    cores = oracle.default_threads()
    res = {}
    # DIFF V1 fp32 tiny workload: in full
    s = inputs.WORKLOADS["v1_fp32_B1_T64_H2_d32"]
    x = _oracle_inputs(inputs.make_v1(s, seed=seed))
    t0 = time.perf_counter()
    oracle.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"],
                  s.layer_index)
    dt = time.perf_counter() - t0
    res["v1_fp32_B1_T64_H2_d32"] = {"s": round(dt, 6), "covered": 1.0, "cores": cores,
                                    "GFLOP/s": round(v1_flops(s) / dt / 1e9, 3)}
    # DIFF V2 decode: in full, one batch entry per call (its cache copied out
    # and widened to fp64 outside the timed calls)
    s = inputs.WORKLOADS["v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128"]
    xd = inputs.make_decode(s, seed=seed, device=dev)
    tot = 0.0
    for b in range(s.B):
        xb = {k: xd[k][b:b + 1].double().cpu().numpy() for k in ("q", "k_cache", "v_cache", "lam")}
        t0 = time.perf_counter()
        oracle.v2_decode(xb["q"], xb["k_cache"], xb["v_cache"], xb["lam"])
        tot += time.perf_counter() - t0
    del xd, xb
    torch.cuda.empty_cache()
    res["v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128"] = {
        "s": round(tot, 3), "covered": 1.0, "cores": cores, "GB/s": round(decode_bytes(s) / tot / 1e9, 3),
        "note": "all B x Hq/2 rows, one batch entry per call"}
    # DIFF V2 prefill and long-context DIFF V1: a sample of rows of batch entry 0
    rng = np.random.default_rng(seed)
    s = inputs.WORKLOADS["v2_bf16_B8_T4096_Hq32_Hkv8_D128"]
    xd = inputs.make_v2(s, seed=seed, device=dev)
    xb = {k: xd[k][0:1].double().cpu().numpy() for k in ("q", "k", "v", "lam")}
    del xd
    P = s.Hq // 2
    rows = rng.choice(s.T * P, size=32768, replace=False)
    t0 = time.perf_counter()
    oracle.v2_fwd(xb["q"], xb["k"], xb["v"], xb["lam"], rows=rows)
    dt = time.perf_counter() - t0
    pairs = float(((rows // P) + 1).sum()) * 2          # two query heads per output row
    frac = pairs / (s.B * s.Hq * s.T * (s.T + 1) / 2)
    res["v2_bf16_B8_T4096_Hq32_Hkv8_D128"] = {
        "s": round(dt, 3), "covered": frac, "cores": cores,
        "TFLOP/s": round(pairs * 4 * s.D / dt / 1e12, 5),
        "sample": "32768 random output rows (t, pair) of batch entry 0"}
    s = inputs.WORKLOADS["v1_bf16_B1_T32768_H12_d128"]
    xd = inputs.make_v1(s, seed=seed, device=dev)
    xb = {k: (xd[k][:, :, 0:1].double().cpu().numpy() if k in ("q1", "q2", "k1", "k2", "v")
              else xd[k].double().cpu().numpy()) for k in ("q1", "q2", "k1", "k2", "v", "lam_q1", "lam_k1",
                                                           "lam_q2", "lam_k2")}
    del xd
    torch.cuda.empty_cache()
    rows = rng.choice(s.T, size=4096, replace=False)
    t0 = time.perf_counter()
    oracle.v1_fwd(xb["q1"], xb["q2"], xb["k1"], xb["k2"], xb["v"], xb["lam_q1"], xb["lam_k1"], xb["lam_q2"],
                  xb["lam_k2"], s.layer_index, rows=rows)
    dt = time.perf_counter() - t0
    pairs = float((rows + 1).sum())
    frac = pairs / (s.B * s.H * s.T * (s.T + 1) / 2)
    res["v1_bf16_B1_T32768_H12_d128"] = {
        "s": round(dt, 3), "covered": frac, "cores": cores,
        "TFLOP/s": round(pairs * 12 * s.d / dt / 1e12, 5),
        "sample": "4096 random rows t of diff head 0"}
    return res


def run_reference(args, rank: int, world: int) -> dict | None:
    """The oracle as the reference arm: fp64 plain C on the host cores."""
    import numpy as np
    import oracle
    if rank != 0:
        return None
    oracle.build()
    s = inputs.WORKLOADS[HEADLINE]
    x = _oracle_inputs(inputs.make_v1(s, seed=args.seed, device="cpu"))
    nall = s.B * s.T * s.H
    rng = np.random.default_rng(args.seed)
    probe = rng.choice(nall, size=256, replace=False)
    dt = _oracle_rows_time(x, s, probe)
    per_row = dt / len(probe)
    budget = max(0.05, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    n = int(max(16, min(nall, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        _oracle_rows_time(x, s, rng.choice(nall, size=n, replace=False))
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        rows = rng.choice(nall, size=n, replace=False)
        tot_t += _oracle_rows_time(x, s, rows)
        tot_f += _rows_flops(rows, s)
    val = tot_f / tot_t / 1e12
    sample = (f"each step: {n} of {nall} random output rows of {HEADLINE}; value = algorithmic "
              f"12d-per-pair FLOPs of the rows / wall time")
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "B": s.B, "T": s.T, "H": s.H, "d": s.d, "dv": 2 * s.d,
                   "layer_index": s.layer_index},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------ single cases (profiling)

CASES = {
    "v1": ("v1", "v1_bf16_B4_T2048_H16_d64"),
    "v1_long": ("v1", "v1_bf16_B1_T32768_H12_d128"),
    "v2": ("v2", "v2_bf16_B8_T4096_Hq32_Hkv8_D128"),
    # the V2 forward with the rotary embedding folded in, on a quarter of the
    # prefill batch (profiler-sized): rotary k, then the prefill
    "v2_rope_b2": ("v2_rope", None),
    "decode": ("decode", "v2_decode_bf16_B64_L32768_Hq64_Hkv8_D128"),
    # the decode workload with 8 of its 64 sequences: 1.07 GB of cache, small
    # enough for multi-pass profiler captures, still far larger than L2
    "decode_b8": ("decode", None),
    "decode_varlen": ("decode_varlen", "v2_decode_varlen_bf16_B64_L32768_Hq64_Hkv8_D128"),
    "v1_decode": ("v1_decode", "v1_decode_bf16_B32_L16384_H12_d128"),
    # backward of the headline V1 workload / a quarter of the V2 prefill workload (profiler-sized)
    "v1_bwd": ("v1_bwd", "v1_bf16_B4_T2048_H16_d64"),
    "v2_bwd_b2": ("v2_bwd", None),
    # the long-context V1 backward (d = 128) on a quarter of its length, profiler-sized
    "v1_long_bwd_t8k": ("v1_bwd", None),
    "prologue": ("prologue", "v2_bf16_B8_T4096_Hq32_Hkv8_D128"),
    "paired": ("paired", "paired_bf16_B8_T4096_H32_D128"),
    # the V1 decode and the ragged-length decode workloads with 4 / 8 of their
    # sequences (0.8 / 1.07 GB of cache: profiler-sized, still far larger than L2)
    "v1_decode_b4": ("v1_decode", None),
    "decode_varlen_b8": ("decode_varlen", None),
    # a quarter of its batch, for multi-pass profiler captures
    "paired_b2": ("paired", None),
    # pinned host <-> device copy rates per NUMA node (the end-to-end figure's link)
    "host_link": ("host_link", None),
}


def host_link(launches: int):
    """Pinned host <-> device copy rates behind the end-to-end figure, with the
    host buffer first touched by a process bound to each NUMA node's CPUs."""
    def read(path):
        try:
            with open(path) as f:
                return f.read().strip()
        except OSError:
            return None
    nodes = {}
    base = "/sys/devices/system/node"
    for n in sorted(os.listdir(base)) if os.path.isdir(base) else []:
        if n.startswith("node") and n[4:].isdigit():
            nodes[n] = read(os.path.join(base, n, "cpulist"))
    bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader"], capture_output=True,
                         text=True).stdout.strip().splitlines()
    gpu_node = read(f"/sys/bus/pci/devices/{bus[0].strip().lower()}/numa_node") if bus else None
    code = r"""
import os, sys, torch
cpus = sys.argv[1]
if cpus != "all":
    sel = set()
    for part in cpus.split(","):
        a, _, b = part.partition("-")
        sel.update(range(int(a), int(b or a) + 1))
    os.sched_setaffinity(0, sel)
n = 256 << 20
h = torch.empty(n, dtype=torch.uint8).pin_memory()
h.fill_(1)
d = torch.empty(n, dtype=torch.uint8, device="cuda")
def rate(fn, k):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(k):
        fn()
    b.record()
    b.synchronize()
    return n * k / (a.elapsed_time(b) * 1e-3) / 1e9
print(rate(lambda: d.copy_(h, non_blocking=True), int(sys.argv[2])),
      rate(lambda: h.copy_(d, non_blocking=True), int(sys.argv[2])))
"""
    res = {}
    for name, cpus in [("all", "all")] + list(nodes.items()):
        r = subprocess.run([sys.executable, "-c", code, cpus or "all", str(max(3, launches))], capture_output=True,
                           text=True)
        v = r.stdout.split()
        res[name] = {"cpus": cpus, "h2d_GBps": round(float(v[0]), 1), "d2h_GBps": round(float(v[1]), 1)} \
            if len(v) == 2 else {"cpus": cpus, "error": r.stderr[-300:]}
    print(json.dumps({"case": "host_link", "numa_nodes": nodes, "gpu_numa_node": gpu_node, "copies": res}))


def run_case(name: str, launches: int):
    from differential_attention_causal_gb300 import binding
    if name == "host_link":
        host_link(launches)
        return
    kind, wl = CASES[name]
    dev = torch.device("cuda", 0)
    if wl:
        s = inputs.WORKLOADS[wl]
    elif kind in ("v2_bwd", "v2_rope"):
        s = inputs.V2Shape(2, 4096, 32, 8, 128, "bf16")
    elif kind == "v1_bwd":
        s = inputs.V1Shape(1, 8192, 12, 128, 27, "bf16")
    elif kind == "paired":
        s = inputs.PairedShape(2, 4096, 32, 128, "bf16")
    elif kind == "v1_decode":
        s = inputs.V1DecodeShape(4, 16384, 12, 128, 27, "bf16")
    elif kind == "decode_varlen":
        s = inputs.DecodeShape(8, 32768, 64, 8, 128, "bf16", True)
    else:
        s = inputs.DecodeShape(8, 32768, 64, 8, 128, "bf16")
    x = inputs.make(s, seed=0, device=dev)
    if kind == "v1":
        f = lambda: binding.v1_fwd(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"],  # noqa
                                   x["lam_q2"], x["lam_k2"], s.layer_index)
    elif kind == "v2":
        f = lambda: binding.v2_fwd(x["q"], x["k"], x["v"], x["lam"])  # noqa: E731
    elif kind == "v2_rope":
        f = lambda: binding.v2_fwd_rope(x["q"], x["k"], x["v"], x["lam"])  # noqa: E731
    elif kind == "paired":
        f = lambda: binding.paired_fwd(x["q"], x["k"], x["v"])  # noqa: E731
    elif kind == "decode_varlen":
        f = lambda: binding.v2_decode_varlen(x["q"], x["k_cache"], x["v_cache"], x["lam"],  # noqa: E731
                                             x["cache_lens"])
    elif kind == "prologue":
        lp = inputs.make_lambda_proj(s.B, s.T, (s.Hq // 2) * s.D, s.Hq // 2, "bf16", seed=0, device=dev)
        f = lambda: binding.prologue(q=x["q"], k=x["k"], x=lp["x"], w_lam=lp["w_lam"])  # noqa: E731
    elif kind == "v1_bwd":
        a = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"],
             s.layer_index)
        dout = inputs.make_grad_out((s.B, s.T, s.H, 2 * s.d), "bf16", seed=0, device=dev)
        _, saved = binding.v1_fwd_train(*a)
        f = lambda: binding.v1_bwd(*a, dout, saved)  # noqa: E731
    elif kind == "v2_bwd":
        dout = inputs.make_grad_out((s.B, s.T, s.Hq // 2, s.D), "bf16", seed=0, device=dev)
        _, saved = binding.v2_fwd_train(x["q"], x["k"], x["v"], x["lam"])
        f = lambda: binding.v2_bwd(x["q"], x["k"], x["v"], x["lam"], dout, saved)  # noqa: E731
    elif kind == "v1_decode":
        f = lambda: binding.v1_decode(x["q1"], x["q2"], x["k1_cache"], x["k2_cache"], x["v_cache"],  # noqa
                                      x["lam_q1"], x["lam_k1"], x["lam_q2"], x["lam_k2"], s.layer_index)
    else:
        f = lambda: binding.v2_decode(x["q"], x["k_cache"], x["v_cache"], x["lam"])  # noqa: E731
    for _ in range(launches):
        f()
    torch.cuda.synchronize()
    if binding.device_error():
        raise RuntimeError("a kernel reported a device-side wait timeout")
    line = {"case": name, "launches": launches, "ok": True}
    if kind == "decode_varlen":   # the lengths are drawn on the device: report what they sum to
        line["alg_bytes_per_launch"] = decode_varlen_bytes(s, x["cache_lens"].tolist())
    elif kind == "v1_decode":
        line["alg_bytes_per_launch"] = v1_decode_bytes(s)
    print(json.dumps(line))


# -------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-aux", action="store_true", help="skip the V2 prefill / decode measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="run one kernel case --launches times and exit (for profilers)")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.launches)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch.distributed as dist
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=dev)
    try:
        line = run_ours(args, rank, world, dev)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
