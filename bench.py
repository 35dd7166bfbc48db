"""Benchmark of the MoE layer forward pass on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward (router, permute, grouped gate/up and down GEMMs, shared experts,
combine) over one resident batch of the named workload; the default workload is the
Mixtral-shaped bf16 layer (N=4096, d=4096, d_ff=14336, E=8, top-2).  Weights (2.8 GB) exceed the
126 MB L2, so no flush is needed between steps.  `value` is tokens/s over all ranks from CUDA
events; `e2e` repeats the measurement through the same C ABI with every step's batch copied in
from pinned host memory and its output copied back (the copies on their own streams, double
buffered, overlapping the neighbouring steps' layers).  `roofline` reports the dominant kernel (the
routed gate/up grouped GEMM) against the measured bf16 peak.  `cpu_baseline` times the CPU oracle
on a bounded sub-batch of the same layer.  Under torchrun (N > 1) every rank runs its own replica
(the layer needs no exchange between GPUs).  The W4A16 workload runs moe_forward_w4a16 on expert
weights quantised once by the library before timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402
from sparse_conditional_moe_b300 import accounting  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_id_for_smi(torch, local: int) -> str:
    """nvidia-smi --id of the device torch uses (its UUID, so CUDA_VISIBLE_DEVICES is honoured)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


# ------------------------------------------------------------------ CPU oracle leg

def cpu_oracle_rate(spec, layer_host: dict, budget_s: float, max_steps: int = 0):
    """Oracle forward over consecutive sub-batches of the layer until budget_s elapses.
    Returns (tokens/s, tokens processed, seconds, sub-batch size, cores)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    code = oracle.BF16 if spec.dtype == "bf16" else oracle.F32
    sub = max(1, min(spec.N, cores))
    x = layer_host["x"]
    done, t_used, steps = 0, 0.0, 0
    start = 0
    while True:
        L = dict(layer_host)
        L["x"] = x[start:start + sub]
        if spec.w4a16:
            t_used += _oracle_w4_batch(spec, L)
        else:
            t0 = time.perf_counter()
            oracle.forward_naive(L, spec.k, code, cf=spec.capacity_factor)
            t_used += time.perf_counter() - t0
        done += L["x"].shape[0]
        steps += 1
        start = (start + sub) % max(1, spec.N - sub + 1)
        if t_used >= budget_s or (max_steps and steps >= max_steps):
            break
    return done / t_used, done, t_used, sub, cores


_W4_ORACLE_WEIGHTS = {}


def _oracle_w4_batch(spec, L) -> float:
    """The W4A16 layer on one sub-batch with the oracle: routing, capacity, then every token's
    experts on the oracle's own quantised weights (quantised once, outside the timed parts).
    Returns the seconds spent in the timed parts."""
    import concurrent.futures as cf
    import oracle
    cache = _W4_ORACLE_WEIGHTS.setdefault(id(L["W_gate"]), {})

    def trip(prefix, e):
        if (prefix, e) not in cache:
            cache[(prefix, e)] = tuple(oracle.quantize_w4(L[prefix + n][e])
                                       for n in ("_gate", "_up", "_down"))
        return cache[(prefix, e)]

    t0 = time.perf_counter()
    idx, w, _, _ = oracle.route(L["x"], L["W_r"], L["b_r"], spec.k, oracle.BF16,
                                bias_mode=spec.bias_mode if L["b_r"] is not None else None)
    n = L["x"].shape[0]
    keep = oracle.keep_naive(idx, spec.E, oracle.capacity(n, spec.k, spec.E,
                                                          spec.capacity_factor))
    t_route = time.perf_counter() - t0
    for e in np.unique(idx):                       # untimed: weight preparation
        trip("W", int(e))
    shared = [trip("Ws", s) for s in range(spec.n_shared)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max(1, min(n, len(os.sched_getaffinity(0))))) as ex:
        list(ex.map(lambda t: oracle.moe_token_w4(L["x"][t], w[t], keep[t],
                                                 [trip("W", int(e)) for e in idx[t]], shared, 1),
                    range(n)))
    return t_route + time.perf_counter() - t0


# ------------------------------------------------------------------ several ranks (replicas)

def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank runs its own replica over its own batch, and the job
    is done when the last one is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: the tokens of all ranks over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def metric_name(spec) -> str:
    if spec == moe_synth.MIXTRAL:
        return "MoE layer forward tokens/s (Mixtral-shaped bf16 layer, 1 GPU)"
    return f"MoE layer forward tokens/s ({spec.name})"


def host_layer(dev: dict) -> dict:
    return {k: (None if v is None else v.cpu()) for k, v in dev.items()}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=moe_synth.MIXTRAL.name,
                    choices=sorted(moe_synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the batch size N (smaller cases for profiling; not a bench line)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count E (smaller cases for profiling; not a bench line)")
    ap.add_argument("--backward", type=int, default=10,
                    help="timed moe_backward iterations after the forward measurement (0: none)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU-oracle budget for the cpu_baseline field (0 to skip)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    spec = moe_synth.WORKLOADS[args.workload]
    if args.tokens > 0:
        spec = spec.with_(N=args.tokens, name=f"{spec.name}_N{args.tokens}")
    if args.experts > 0:
        spec = spec.with_(E=args.experts, k=min(spec.k, args.experts),
                          name=f"{spec.name}_E{args.experts}")
    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        return run_reference(args, spec, rank, world)

    import torch
    import torch.distributed as dist
    from sparse_conditional_moe_b300 import moe

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    cfg = moe.cfg_from_spec(spec)
    w4 = moe.quantize_layer_w4(dev) if spec.w4a16 else None
    host_copy = None
    if w4 is not None:
        # the forward reads the 4-bit copies only: keep host bf16 weights for the oracle leg
        # (if it runs) and free the device ones
        if args.cpu_seconds > 0 and rank == 0:
            host_copy = host_layer(dev)
        for n in ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
            if dev.get(n) is not None:
                dev[n] = torch.empty(0, dtype=torch.bfloat16, device="cuda")
        torch.cuda.empty_cache()
    lay = moe.MoELayer(cfg, dev, w4=w4)
    xs = [dev["x"], moe_synth.make_x(spec, seed=1000 + rank, device="cuda")]
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for i in range(args.warmup):
        lay.forward(xs[i % 2])
    torch.cuda.synchronize()
    if lay.device_error() != 0:
        raise RuntimeError("device error during warm-up")
    st = lay.stats()
    kept_rows, touched = st["kept_rows"], st["touched_experts"]

    # ---------------- device-timed region (inputs resident in HBM)
    # Each step records two events, around the routed gate/up GEMM (the dominant kernel, whose
    # roofline is reported from these); the full per-phase breakdown comes from a separate
    # traced pass, so seven event records per step do not add to the timed work of small,
    # launch-bound layers.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gu_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
             for _ in range(args.steps)]
    clocks = ClockSampler(gpu_id_for_smi(torch, local))
    clocks.start()
    time.sleep(0.15)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        lay.forward(xs[i % 2], events=[None, None, gu_ev[i][0], gu_ev[i][1], None, None, None])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, "cuda")
    if lay.device_error() != 0:
        raise RuntimeError("device error during the timed region")
    ms_step = elapsed_ms / args.steps

    # ---------------- per-phase breakdown (traced pass, not part of the timed region)
    trace_steps = max(1, min(args.steps, 50))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_TRACE_EVENTS)]
          for _ in range(trace_steps)]
    for i in range(trace_steps):
        lay.forward(xs[i % 2], events=ev[i])
    torch.cuda.synchronize()
    value = job_rate(spec.N, world, ms_step)

    phases = ["route", "permute", "gateup", "down", "shared", "combine"]
    ph_ms = {p: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(trace_steps))
             for j, p in enumerate(phases)}

    # ---------------- roofline of the dominant kernel (routed gate/up grouped GEMM)
    act_b = 2 if spec.dtype == "bf16" else 4
    w_b = accounting.W4_BYTES_PER_WEIGHT if spec.w4a16 else act_b
    gu_flops = accounting.gateup_flops(spec.d, spec.d_ff, kept_rows)
    gu_ms_timed = statistics.mean(a.elapsed_time(b) for a, b in gu_ev)
    gu_s = gu_ms_timed / 1e3
    peak_t = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    achieved_t = gu_flops / gu_s / 1e12
    work = accounting.layer_work(spec.N, spec.d, spec.d_ff, spec.E, spec.k, spec.n_shared,
                                 spec.d_ff_shared, act_b, kept_rows, touched, weight_bytes=w_b)
    layer_tflops = work.flops / (ms_step / 1e3) / 1e12
    layer_gbs = work.bytes / (ms_step / 1e3) / 1e9
    roof_s = work.roofline_s(peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
    traffic = read_traffic("gateup", spec.name)
    # the dominant kernel's rate from the timed region, the other phases from the traced pass
    phase_roof = phase_rooflines(spec, act_b, w_b, kept_rows, touched,
                                 dict(ph_ms, gateup=gu_ms_timed), peaks)

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its batch in from pinned host memory and its output back.  The copies run
    # on their own streams with two device buffers each way, so step i's upload and step i-2's
    # download overlap step i-1's layer (events keep each buffer's uses in order).
    x_host = [x.cpu().pin_memory() for x in xs]
    out_host = [torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(xs[0]) for _ in range(2)]
    out_dev = [torch.empty_like(lay.out) for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    e2e_steps = max(3, min(args.steps, 50))

    def run_e2e(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        ev_d2h = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev_out[i - 2])          # x_dev[b] read by step i-2
                x_dev[b].copy_(x_host[i % 2], non_blocking=True)
                ev_in[i].record(up)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_d2h[i - 2])          # out_dev[b] copied out by step i-2
            lay.forward(x_dev[b], out=out_dev[b])
            ev_out[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_out[i])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                ev_d2h[i].record(down)
        return ev_d2h[n - 1]

    run_e2e(3)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    last = run_e2e(e2e_steps)
    down.wait_event(last)
    e1.record(down)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, "cuda")
    e2e_value = job_rate(spec.N, world, e2e_ms)

    # router 2, permute 4, m-tile plan 1 (not on the W4A16 path), routed 2, shared 2, combine 1
    # ---------------- backward pass (bf16 layers whose fp32 weight gradients fit comfortably)
    bwd = None
    grad_bytes = 4.0 * (3 * spec.E * spec.d * spec.d_ff + 3 * spec.n_shared * spec.d * spec.d_ff_shared)
    if (args.backward > 0 and not spec.w4a16 and spec.dtype == "bf16" and grad_bytes <= 24e9
            and spec.d % 64 == 0 and spec.d_ff % 128 == 0):
        dout = torch.randn(lay.out.shape, device="cuda").to(torch.bfloat16)
        lay.forward(xs[0])
        for _ in range(2):
            lay.backward(dout)
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(args.backward):
            lay.backward(dout)
        b1.record(stream)
        torch.cuda.synchronize()
        if lay.device_error() != 0:
            raise RuntimeError("device error in the backward pass")
        bwd_ms = b0.elapsed_time(b1) / args.backward
        # expert GEMM work of the backward: 2x the forward's (data and weight gradients)
        bwd_flops = 2.0 * (accounting.gateup_flops(spec.d, spec.d_ff, kept_rows)
                           + accounting.down_flops(spec.d, spec.d_ff, kept_rows)
                           + 6.0 * spec.d * spec.d_ff_shared * spec.N * spec.n_shared)
        bwd = {"ms": bwd_ms, "tokens_per_s": spec.N * world / (bwd_ms / 1e3),
               "expert_tflops": bwd_flops / (bwd_ms / 1e3) / 1e12, "iterations": args.backward,
               "note": "moe_backward after one forward, all gradients fp32; the expert GEMMs do 2x "
                       "the forward's work (gate/up recomputed once more on top)"}

    launches_per_step = 2 + 4 + (0 if spec.w4a16 else 1) + 2 + (2 if spec.n_shared > 0 else 0) + 1
    gemm_kernel = ("grouped W4A16 gate/up SwiGLU (CUDA cores, FFMA2)" if spec.w4a16
                   else "grouped gate/up SwiGLU GEMM (tcgen05)")

    # ---------------- CPU oracle on a bounded sub-batch (rank 0 only)
    cpu = None
    if rank == 0 and args.cpu_seconds > 0:
        rate, done, secs, sub, cores = cpu_oracle_rate(spec, host_copy or host_layer(dev),
                                                       args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{done} tokens of {spec.name} in consecutive sub-batches of {sub} "
                         f"(each its own batch), {secs:.1f} s of CPU work"
                         + (" (weights quantised by the oracle beforehand, untimed)"
                            if spec.w4a16 else "")}

    if rank == 0:
        line = {
            "metric": metric_name(spec),
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if act_b == 2 else "f32",
            "data": "synthetic (seeded N(0,1) activations, N(0,1/d_in) weights)",
            "config": {"workload": spec.name, "N": spec.N, "d": spec.d, "d_ff": spec.d_ff,
                       "E": spec.E, "k": spec.k, "n_shared": spec.n_shared,
                       "capacity_factor": spec.capacity_factor,
                       "weights": "w4a16 (int4 codes + fp32 scale per 128)" if spec.w4a16
                       else spec.dtype,
                       "l2": "no flush: weights of %.2f GB exceed the 126 MB L2" %
                             (3 * spec.E * spec.d * spec.d_ff * w_b / 1e9),
                       "parallelism": f"replicas x{world}"},
            "layer": {"tflops": layer_tflops, "hbm_gbs_alg": layer_gbs,
                      "roofline_ms": roof_s * 1e3, "roofline_frac": roof_s * 1e3 / ms_step,
                      "kept_rows": kept_rows, "touched_experts": touched,
                      "gateup_ms_timed_region": gu_ms_timed, "phase_ms": ph_ms, "phase_roofline": phase_roof, "backward": bwd},
            "roofline": ({"kernel": gemm_kernel, "bound": "tensor",
                          "achieved": achieved_t, "peak": peak_t, "unit": "TFLOP/s",
                          "frac": achieved_t / peak_t, "traffic": traffic,
                          "frac_of_burst": achieved_t / peaks["bf16_tflops"],
                          "peak_source": f"{peak_src} bf16 sustained (kernel timed inside a "
                                         f"continuous loop); burst {peaks['bf16_tflops']}"}
                         if phase_roof["gateup"]["unit"] == "TFLOP/s" else
                         {"kernel": gemm_kernel, "bound": "hbm",
                          "achieved": phase_roof["gateup"]["achieved"], "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": phase_roof["gateup"]["frac"],
                          "traffic": None if spec.w4a16 else traffic,
                          "peak_source": f"{peak_src} HBM copy bandwidth"}),
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "h2d_bytes_per_step": spec.N * spec.d * act_b,
                    "d2h_bytes_per_step": spec.N * spec.d * act_b},
            "gpu_launches": launches_per_step * args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def phase_rooflines(spec, act_b, w_b, kept_rows, touched, ph_ms, peaks):
    """Achieved rate of every phase against its own bound (algorithmic work only): the GEMM
    phases in TFLOP/s against the bf16 peak, the data-movement phases in GB/s against HBM.
    w_b: bytes per expert weight (the activation size, or 0.53125 for W4A16)."""
    d, F, E, N, S, Fs = spec.d, spec.d_ff, spec.E, spec.N, spec.n_shared, spec.d_ff_shared
    tf_peak, gb_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), peaks["hbm_gbs"]
    w_bytes = w_b * d * F
    work = {
        # x read + W_r read
        "route": ("GB/s", N * d * act_b + 4.0 * d * E),
        # x rows read + grouped rows written (+ indices)
        "permute": ("GB/s", 2.0 * kept_rows * d * act_b + 16.0 * N * spec.k),
        "gateup": ("TFLOP/s", accounting.gateup_flops(d, F, kept_rows)),
        "down": ("TFLOP/s", accounting.down_flops(d, F, kept_rows)),
        "shared": ("TFLOP/s", 6.0 * d * Fs * N * S),
        # grouped rows + shared rows read, out written
        "combine": ("GB/s", (kept_rows + S * N) * d * act_b + N * d * act_b),
    }
    if spec.N <= 1024:   # decode-sized: the GEMMs stream weights, HBM is their bound
        work["gateup"] = ("GB/s", 2.0 * w_bytes * touched + kept_rows * (d + F) * act_b)
        work["down"] = ("GB/s", 1.0 * w_bytes * touched + kept_rows * (d + F) * act_b)
        work["shared"] = ("GB/s", 3.0 * w_b * d * Fs * S + N * (d + Fs) * act_b * 2)
    out = {}
    for ph, (unit, amount) in work.items():
        ms = ph_ms.get(ph, 0.0)
        if ms <= 0 or amount <= 0:
            continue
        rate = amount / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
        peak = tf_peak if unit == "TFLOP/s" else gb_peak
        out[ph] = {"ms": ms, "achieved": rate, "unit": unit, "frac": rate / peak}
    return out


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if its source hash is current."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in ("grouped_gemm_tc.cu", "tc_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "sparse_conditional_moe_b300", "csrc", f), "rb").read())
    h = h.hexdigest()[:16]
    for ln in open(path):
        parts = [p.strip() for p in ln.strip().strip("|").split("|")]
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[2] == h:
            try:
                return float(parts[3])
            except ValueError:
                return None
    return None


def run_reference(args, spec, rank, world):
    """The CPU oracle timed on this machine's host cores on the same workload and metric."""
    if rank != 0:
        return
    import torch
    layer = moe_synth.make_layer(spec, seed=0, device="cpu")
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_rate(spec, layer, 0.0, max_steps=1)
    rates = []
    t0 = time.perf_counter()
    total, secs_total = 0, 0.0
    for _ in range(args.steps):
        rate, done, secs, sub, cores = cpu_oracle_rate(spec, layer, budget)
        total += done
        secs_total += secs
    wall = time.perf_counter() - t0
    value = total / secs_total
    line = {
        "impl": "reference", "metric": metric_name(spec), "value": value,
        "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * spec.N / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": spec.name, "N": spec.N, "d": spec.d, "d_ff": spec.d_ff,
                   "E": spec.E, "k": spec.k},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{total} tokens in sub-batches of {sub}, {secs_total:.1f} s "
                                   f"of oracle time ({wall:.1f} s wall)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    del torch
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
