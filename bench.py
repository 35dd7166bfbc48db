"""Benchmark of the MoE layer forward pass on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward (router, permute, grouped gate/up and down GEMMs, shared experts,
combine) over one resident batch of the named workload.  The default workload, and the headline
`value`, is the DeepSeek-V3-shaped prefill layer (N=8192, d=7168, d_ff=2048, E=256, top-8, one
shared expert): the largest layer of the workload set that fits one GPU.  Its weights (22.5 GB)
exceed the 126 MB L2, so no flush is needed between steps.  `value` is tokens/s over all ranks
from CUDA events around the K timed steps; `e2e` repeats the measurement through the same C ABI
with every step's batch copied in from pinned host memory and its output copied back;
`roofline` reports the dominant kernel (the routed gate/up grouped GEMM) against the measured
burst bf16 peak; `workloads` repeats the device-timed measurement, with the same K and W, on
the other layers of the set (Mixtral-shaped, DeepSeek-V3-shaped decode with bf16 and with
W4A16 expert weights, Qwen3-30B-A3B-shaped skewed); `cpu_baseline` times the CPU oracle on a
bounded sample of the headline layer.  Under torchrun (N > 1) every rank runs its own replica
(the layer needs no exchange between GPUs).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
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
HEADLINE = moe_synth.DSV3_PREFILL
# the layer whose backward is timed in a full run (its backward is checked at full size)
BACKWARD_WORKLOAD = moe_synth.MIXTRAL
SIDE_WORKLOADS = (moe_synth.MIXTRAL, moe_synth.DSV3_DECODE, moe_synth.DSV3_DECODE_W4,
                  moe_synth.QWEN3_SKEWED)
# the library forks the shared experts of bf16 batches of at most this many tokens onto its
# side stream, so the per-phase events on the caller's stream do not bracket them
SIDE_STREAM_MAX_TOKENS = 128


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class _Nvml:
    """The few NVML calls the clock sampler needs, through ctypes on the driver's libnvidia-ml."""

    def __init__(self, uuid: str):
        L = ctypes.CDLL("libnvidia-ml.so.1")
        self.L = L
        rc = (getattr(L, "nvmlInit_v2", None) or L.nvmlInit)()
        if rc != 0:
            raise RuntimeError(f"nvmlInit returned {rc}")
        self.h = ctypes.c_void_p()
        rc = L.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError(f"nvmlDeviceGetHandleByUUID({uuid}) returned {rc}")
        self._reasons = (getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None)
                         or L.nvmlDeviceGetCurrentClocksThrottleReasons)
        self.max_mhz = self.clock(getattr(L, "nvmlDeviceGetMaxClockInfo"))

    def clock(self, fn=None) -> float:
        v = ctypes.c_uint()
        rc = (fn or self.L.nvmlDeviceGetClockInfo)(self.h, 1, ctypes.byref(v))   # 1 = SM clock
        if rc != 0:
            raise RuntimeError(f"clock query returned {rc}")
        return float(v.value)

    def sample(self):
        mw, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.L.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw)) != 0:
            mw.value = 0
        if self._reasons(self.h, ctypes.byref(rs)) != 0:
            rs.value = 0
        return self.clock(), mw.value / 1000.0, int(rs.value)

    def close(self):
        self.L.nvmlShutdown()


class ClockSampler:
    """SM clocks and throttle reasons sampled every few milliseconds during a timed region,
    through NVML (nvidia-smi polling as a fallback)."""
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))

    def __init__(self, uuid: str, period_s: float = 0.004):
        self.uuid = uuid
        self.period = period_s
        self.samples = []      # (sm_mhz, max_mhz, power_w, reasons bitmask)
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._proc = None
        self.nvml_error = None

    def start(self):
        try:
            self._nvml = _Nvml(self.uuid)
        except Exception as e:   # noqa: BLE001 -- fall back to nvidia-smi polling
            self.nvml_error = f"{type(e).__name__}: {e}"
            self._nvml = None
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return
        try:
            fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,"
                      "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.uuid}", f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._read_smi, daemon=True)
            self._thread.start()
        except (OSError, ValueError):
            self._proc = None

    def _poll(self):
        nv = self._nvml
        while not self._stop.is_set():
            try:
                sm, pw, rs = nv.sample()
                self.samples.append((sm, nv.max_mhz, pw, rs))
            except Exception:   # noqa: BLE001 -- a failed poll is a missing sample
                pass
            time.sleep(self.period)

    def _read_smi(self):
        for ln in self._proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                bits = sum(b for (_, b), v in zip(self.REASONS, parts[3:7]) if v.lower() == "active")
                self.samples.append((float(parts[0]), float(parts[1]), float(parts[2]), bits))
            except ValueError:
                continue

    def stop(self) -> dict:
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._nvml is not None:
            try:
                self._nvml.close()
            except Exception:   # noqa: BLE001
                pass
        if not self.samples:
            out = {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                   "reasons": ["no clock samples (NVML and nvidia-smi unavailable)"]}
            if self.nvml_error:
                out["nvml_error"] = self.nvml_error
            return out
        reasons = sorted({n for n, b in self.REASONS for s in self.samples if s[3] & b})
        out = {"sm_mhz": statistics.median(s[0] for s in self.samples),
               "sm_min_mhz": min(s[0] for s in self.samples),
               "sm_max_mhz": max(s[1] for s in self.samples),
               "power_w_max": max(s[2] for s in self.samples),
               "samples": len(self.samples),
               "source": "nvml" if self._nvml is not None else "nvidia-smi",
               "reasons": reasons}
        if self.nvml_error:
            out["nvml_error"] = self.nvml_error
        return out


def gpu_uuid(torch, local: int) -> str:
    """The NVML/nvidia-smi id of the device torch uses (its UUID, so CUDA_VISIBLE_DEVICES is
    honoured)."""
    u = str(torch.cuda.get_device_properties(local).uuid)
    return u if u.startswith("GPU-") else "GPU-" + u


# ------------------------------------------------------------------ CPU oracle leg

def cpu_oracle_rate(spec, layer_host: dict, budget_s: float, max_steps: int = 0, sub: int = 0):
    """Oracle forward over consecutive sub-batches of the layer until budget_s elapses (each
    sub-batch is routed as a batch of its own).  Returns (tokens/s, tokens, seconds, sub-batch
    size, cores)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    code = oracle.BF16 if spec.dtype == "bf16" else oracle.F32
    sub = sub or max(1, min(spec.N, cores))
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


def cpu_oracle_one_core(spec, layer_host: dict, tokens: int = 2):
    """The oracle on one thread over `tokens` tokens (OpenMP restricted to one thread for the
    call), extrapolated linearly to tokens/s of one core."""
    import oracle
    try:
        gomp = ctypes.CDLL("libgomp.so.1")
        prev = gomp.omp_get_max_threads()
        gomp.omp_set_num_threads(1)
    except OSError:
        return None
    try:
        rate, done, secs, sub, _ = cpu_oracle_rate(spec, layer_host, 0.0, max_steps=1, sub=tokens)
    finally:
        gomp.omp_set_num_threads(prev)
    return {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} tokens of {spec.name} on one thread ({secs:.1f} s), extrapolated "
                      f"linearly to tokens/s"}


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


def cpu_sample_note(spec, sub: int) -> str:
    note = f"consecutive sub-batches of {sub} tokens, each routed as its own batch"
    if spec.capacity_factor > 0:
        c = int(np.ceil(spec.capacity_factor * sub * spec.k / spec.E))
        note += f" (so with its own capacity C = {c}, not the full batch's)"
    return note


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
    return f"MoE layer forward tokens/s ({spec.name})"


def config_of(spec, world: int) -> dict:
    w_b = accounting.W4_BYTES_PER_WEIGHT if spec.w4a16 else (2 if spec.dtype == "bf16" else 4)
    return {"workload": spec.name, "N": spec.N, "d": spec.d, "d_ff": spec.d_ff, "E": spec.E,
            "k": spec.k, "n_shared": spec.n_shared, "capacity_factor": spec.capacity_factor,
            "weights": "w4a16 (int4 codes + fp32 scale per 128)" if spec.w4a16 else spec.dtype,
            "l2": "no flush: weights of %.2f GB exceed the 126 MB L2"
                  % (3 * spec.E * spec.d * spec.d_ff * w_b / 1e9),
            "parallelism": f"replicas x{world}"}


def host_layer(dev: dict) -> dict:
    return {k: (None if v is None else v.cpu()) for k, v in dev.items()}


def count_kernel_launches(torch, lay, x) -> int:
    """Kernels one forward launches: the kernel nodes of a CUDA graph captured from it (-1 if
    the graph cannot be inspected)."""
    try:
        from cuda.bindings import runtime as rt
        g = torch.cuda.CUDAGraph(keep_graph=True)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                lay.forward(x)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        raw = g.raw_cuda_graph()
        graph = raw if isinstance(raw, rt.cudaGraph_t) else rt.cudaGraph_t(init_value=int(raw))
        err, _, n = rt.cudaGraphGetNodes(graph, 0)
        if err != rt.cudaError_t.cudaSuccess:
            return -1
        err, nodes, n = rt.cudaGraphGetNodes(graph, n)
        if err != rt.cudaError_t.cudaSuccess:
            return -1
        kernels = 0
        for nd in nodes[:n]:
            err, t = rt.cudaGraphNodeGetType(nd)
            if err == rt.cudaError_t.cudaSuccess and t == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                kernels += 1
        del g
        return kernels
    except Exception as e:   # noqa: BLE001 -- reported as unknown, never fatal to the bench
        print(f"kernel count unavailable: {e}", file=sys.stderr)
        return -1


# ------------------------------------------------------------------ one workload

def backward_eligible(spec) -> bool:
    """moe_backward covers bf16 layers with d a multiple of 64 and d_ff, d_ff_shared multiples of
    128 (not W4A16 weights)."""
    return (spec.dtype == "bf16" and not spec.w4a16 and spec.d % 64 == 0 and spec.d_ff % 128 == 0
            and (spec.n_shared == 0 or spec.d_ff_shared % 128 == 0))


def measure_backward(spec, lay, x, kept_rows, iters, peaks, torch, world):
    """moe_backward after one forward: 2 warm-up passes, then `iters` passes between CUDA events
    on the launching stream.  Algorithmic expert work of a backward pass: the data and weight
    gradients of the three expert matrices, 12 d d_ff per kept row (twice the forward's 6; the
    pass also recomputes gate/up, 4 d d_ff per row, not counted), and the same for the shared
    experts over every token."""
    dout = torch.randn(lay.out.shape, device="cuda").to(torch.bfloat16)
    lay.forward(x)
    for _ in range(2):
        lay.backward(dout)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(iters):
        lay.backward(dout)
    b1.record(stream)
    torch.cuda.synchronize()
    if lay.device_error() != 0:
        raise RuntimeError(f"device error in the backward pass ({spec.name})")
    ms = b0.elapsed_time(b1) / iters
    flops = 12.0 * spec.d * spec.d_ff * kept_rows + 12.0 * spec.d * spec.d_ff_shared * spec.N * spec.n_shared
    tflops = flops / (ms / 1e3) / 1e12
    return {"ms": ms, "tokens_per_s": spec.N * world / (ms / 1e3), "iterations": iters,
            "expert_tflops": tflops, "tensor_frac": tflops / peaks["bf16_tflops"],
            "work": f"12*d*d_ff*kept_rows (+ shared) = {flops:.4g} flop",
            "note": "moe_backward after one forward: dx, dW_r, db and the expert weight gradients, "
                    "all fp32; gate/up recomputed (not counted)"}


def measure(spec, args, peaks, torch, dist, world, rank, local, headline: bool,
            backward: bool = False):
    """Device-timed forward of one workload: K steps after W warm-up steps, events around the
    routed gate/up and down GEMMs of every timed step, clocks sampled during the region.
    The headline workload also gets the end-to-end measurement and the CPU oracle leg;
    `backward` adds a timed moe_backward (measure_backward)."""
    from sparse_conditional_moe_b300 import moe
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    cfg = moe.cfg_from_spec(spec)
    w4 = moe.quantize_layer_w4(dev) if spec.w4a16 else None
    host_copy = None
    want_cpu = headline and rank == 0 and args.cpu_seconds > 0
    if w4 is not None:
        # the forward reads the 4-bit copies only: keep host bf16 weights for the oracle leg
        if want_cpu:
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
        raise RuntimeError(f"device error during warm-up ({spec.name})")
    st = lay.stats()
    kept_rows, touched = st["kept_rows"], st["touched_experts"]

    # ---------------- device-timed region (inputs resident in HBM)
    # Each step records four events: around the routed gate/up GEMM (the dominant kernel, whose
    # roofline is reported from these) and around the routed down GEMM.  The other per-phase
    # times come from a separate traced pass.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(torch, local))
    clocks.start()
    time.sleep(0.05)
    barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        lay.forward(xs[i % 2], events=[None, None, ev[i][0], ev[i][1], ev[i][2], None, None])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    region_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(region_ms, world, "cuda")
    if lay.device_error() != 0:
        raise RuntimeError(f"device error during the timed region ({spec.name})")
    ms_step = elapsed_ms / args.steps
    gu_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    dn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)

    # ---------------- per-phase breakdown (traced pass, not part of the timed region)
    trace_steps = max(1, min(args.steps, 20))
    tev = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_TRACE_EVENTS)]
           for _ in range(trace_steps)]
    for i in range(trace_steps):
        lay.forward(xs[i % 2], events=tev[i])
    torch.cuda.synchronize()
    phases = ["route", "permute", "gateup", "down", "shared", "combine"]
    ph_ms = {p: statistics.mean(tev[i][j].elapsed_time(tev[i][j + 1]) for i in range(trace_steps))
             for j, p in enumerate(phases)}
    forked = (spec.dtype == "bf16" and spec.n_shared > 0 and spec.N <= SIDE_STREAM_MAX_TOKENS)
    if forked or spec.n_shared == 0:
        ph_ms.pop("shared")

    act_b = 2 if spec.dtype == "bf16" else 4
    w_b = accounting.W4_BYTES_PER_WEIGHT if spec.w4a16 else act_b
    work = accounting.layer_work(spec.N, spec.d, spec.d_ff, spec.E, spec.k, spec.n_shared,
                                 spec.d_ff_shared, act_b, kept_rows, touched, weight_bytes=w_b)
    roof_s = work.roofline_s(peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9)
    phase_roof = phase_rooflines(spec, act_b, w_b, kept_rows, touched,
                                 dict(ph_ms, gateup=gu_ms, down=dn_ms), peaks)
    out = {
        "workload": spec.name, "value": job_rate(spec.N, world, ms_step), "unit": "tokens/s",
        "ms_per_step": ms_step, "timed_region_ms": region_ms,
        "layer": {"tflops": work.flops / (ms_step / 1e3) / 1e12,
                  "hbm_gbs_alg": work.bytes / (ms_step / 1e3) / 1e9,
                  "roofline_ms": roof_s * 1e3, "roofline_frac": roof_s * 1e3 / ms_step,
                  "bound": work.bound(peaks["bf16_tflops"] * 1e12, peaks["hbm_gbs"] * 1e9),
                  "kept_rows": kept_rows, "touched_experts": touched},
        "gateup": phase_roof["gateup"], "down": phase_roof["down"],
        "phase_ms": ph_ms, "phase_roofline": phase_roof,
        "shared_phase": ("forked onto the library's side stream (overlaps the routed phases; "
                         "not bracketed by the caller-stream events)") if forked else None,
        "clocks": clk,
    }
    if backward and args.backward > 0 and backward_eligible(spec):
        out["backward"] = measure_backward(spec, lay, xs[0], kept_rows, args.backward, peaks,
                                           torch, world)
    if not headline:
        del lay, dev, xs, w4
        torch.cuda.empty_cache()
        return out

    out["gpu_launches_per_step"] = count_kernel_launches(torch, lay, xs[0])

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its batch in from pinned host memory and its output back.  The copies run
    # on their own streams with two device buffers each way, so step i's upload and step i-2's
    # download overlap step i-1's layer (events keep each buffer's uses in order).
    x_host = [x.cpu().pin_memory() for x in xs]
    out_host = [torch.empty(lay.out.shape, dtype=lay.out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(xs[0]) for _ in range(2)]
    out_dev = [torch.empty_like(lay.out) for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

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

    run_e2e(max(3, args.warmup))
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    last = run_e2e(args.steps)
    down.wait_event(last)
    e1.record(down)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    out["e2e"] = {"value": job_rate(spec.N, world, e2e_ms), "unit": "tokens/s",
                  "h2d_bytes_per_step": x_host[0].numel() * x_host[0].element_size(),
                  "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size()}

    # ---------------- CPU oracle on a bounded sample (rank 0 only)
    if want_cpu:
        hl = host_copy or host_layer(dev)
        del lay, dev, xs
        torch.cuda.empty_cache()
        rate, done, secs, sub, cores = cpu_oracle_rate(spec, hl, args.cpu_seconds)
        out["cpu_baseline"] = {
            "value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tokens of {spec.name} in {cpu_sample_note(spec, sub)}; "
                      f"{secs:.1f} s of CPU work"
                      + (" (weights quantised by the oracle beforehand, untimed)"
                         if spec.w4a16 else "")}
        out["cpu_baseline_one_core"] = cpu_oracle_one_core(spec, hl)
    return out


def phase_rooflines(spec, act_b, w_b, kept_rows, touched, ph_ms, peaks):
    """Achieved rate of every phase against its own bound (algorithmic work only).  A GEMM phase
    has both a tensor bound (flops / burst bf16 peak) and an HBM bound (weights of the touched
    experts + rows read and written, / HBM bandwidth); the larger ideal time binds, and the phase
    is reported in that bound's unit, with the other bound's fraction beside it.  The
    data-movement phases are HBM-bound.  w_b: bytes per expert weight (the activation size, or
    0.53125 for W4A16)."""
    d, F, E, N, S, Fs = spec.d, spec.d_ff, spec.E, spec.N, spec.n_shared, spec.d_ff_shared
    tf_peak, gb_peak = peaks["bf16_tflops"], peaks["hbm_gbs"]
    w_bytes = w_b * d * F
    rows_io = kept_rows * (d + F) * act_b
    gemm = {   # phase: (flops, bytes)
        "gateup": (accounting.gateup_flops(d, F, kept_rows), 2.0 * w_bytes * touched + rows_io),
        "down": (accounting.down_flops(d, F, kept_rows), 1.0 * w_bytes * touched + rows_io),
        "shared": (6.0 * d * Fs * N * S, 3.0 * w_b * d * Fs * S + 2.0 * N * (d + Fs) * act_b * S),
    }
    moves = {
        # x read + W_r read
        "route": N * d * act_b + 4.0 * d * E,
        # x rows read + grouped rows written (+ indices)
        "permute": 2.0 * kept_rows * d * act_b + 16.0 * N * spec.k,
        # grouped rows + shared rows read, out written
        "combine": (kept_rows + S * N) * d * act_b + N * d * act_b,
    }
    out = {}
    for ph, ms in ph_ms.items():
        if ms <= 0:
            continue
        sec = ms / 1e3
        if ph in gemm:
            flops, nbytes = gemm[ph]
            if flops <= 0:
                continue
            t_tensor, t_hbm = flops / (tf_peak * 1e12), nbytes / (gb_peak * 1e9)
            tensor = {"achieved": flops / sec / 1e12, "unit": "TFLOP/s"}
            tensor["frac"] = tensor["achieved"] / tf_peak
            hbm = {"achieved": nbytes / sec / 1e9, "unit": "GB/s"}
            hbm["frac"] = hbm["achieved"] / gb_peak
            if t_tensor >= t_hbm:
                out[ph] = {"ms": ms, "bound": "tensor", **tensor, "hbm_frac": hbm["frac"],
                           "flops": flops, "bytes": nbytes}
            else:
                out[ph] = {"ms": ms, "bound": "hbm", **hbm, "tensor_frac": tensor["frac"],
                           "flops": flops, "bytes": nbytes}
        elif ph in moves:
            rate = moves[ph] / sec / 1e9
            out[ph] = {"ms": ms, "bound": "hbm", "achieved": rate, "unit": "GB/s",
                       "frac": rate / gb_peak, "bytes": moves[ph]}
    return out


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("grouped_gemm_pair.cu", "tc_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "sparse_conditional_moe_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary (scaled from
    the captured case to the full launch), if the summary's source hash is current."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash()
    for ln in open(path):
        parts = [p.strip() for p in ln.strip().strip("|").split("|")]
        if len(parts) >= 5 and parts[0] == kernel and parts[1] == workload and parts[2] == h:
            try:
                return float(parts[3]) * float(parts[4])
            except ValueError:
                return None
    return None


def roofline_of(spec, res, peaks, peak_src):
    """The dominant kernel (the routed gate/up launch) against the bound that binds it."""
    g = res["gateup"]
    kern = ("routed grouped W4A16 gate/up SwiGLU (TMA + mma.sync)" if spec.w4a16
            else "routed grouped gate/up SwiGLU GEMM (tcgen05, CTA pairs)")
    traffic = None if spec.w4a16 else read_traffic("gateup", spec.name)
    common = {"kernel": kern, "achieved": g["achieved"], "unit": g["unit"], "frac": g["frac"],
              "traffic": traffic, "ms_per_launch": g["ms"],
              "work_per_launch": {"flop": g["flops"], "bytes": g["bytes"],
                                  "flop_formula": "4*d*d_ff*kept_rows",
                                  "bytes_formula": "2*d*d_ff*w_bytes*touched_experts + "
                                                   "kept_rows*(d + d_ff)*act_bytes"}}
    if g["bound"] == "tensor":
        return {"bound": "tensor", "peak": peaks["bf16_tflops"], **common,
                "hbm_frac": g["hbm_frac"],
                "peak_source": f"{peak_src} bf16 burst (cuBLAS bf16 GEMM, best of 10)"}
    return {"bound": "hbm", "peak": peaks["hbm_gbs"], **common, "tensor_frac": g["tensor_frac"],
            "tensor_peak": peaks["bf16_tflops"],
            "peak_source": f"{peak_src} HBM copy bandwidth (tensor: bf16 burst)"}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE.name, choices=sorted(moe_synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the batch size N (smaller cases for profiling; not a bench line)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count E (smaller cases for profiling; not a bench line)")
    ap.add_argument("--backward", type=int, default=5,
                    help="timed moe_backward passes after the forward measurement of the "
                         "Mixtral-shaped layer (also when it is run alone, at any --tokens / "
                         "--experts); 0: none")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure the named workload only (no `workloads` object)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU-oracle budget for the cpu_baseline field (0 to skip)")
    args = ap.parse_args()
    if args.impl == "ours" and args.warmup < 3:
        ap.error("at least 3 warm-up steps")

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

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    single = args.no_workloads or args.tokens > 0 or args.experts > 0
    res = measure(spec, args, peaks, torch, dist, world, rank, local, headline=True,
                  backward=spec.name.startswith(BACKWARD_WORKLOAD.name))
    side = {}
    if not single:
        for s in SIDE_WORKLOADS:
            if s.name == spec.name:
                continue
            r = measure(s, args, peaks, torch, dist, world, rank, local, headline=False,
                        backward=s.name == BACKWARD_WORKLOAD.name)
            side[s.name] = {"ms_per_step": r["ms_per_step"], "value": r["value"],
                            "unit": "tokens/s", "gateup": r["gateup"], "down": r["down"],
                            "layer_roofline_frac": r["layer"]["roofline_frac"],
                            "layer_bound": r["layer"]["bound"],
                            "kept_rows": r["layer"]["kept_rows"],
                            "touched_experts": r["layer"]["touched_experts"],
                            "phase_ms": r["phase_ms"], "shared_phase": r["shared_phase"],
                            "clocks": {k: r["clocks"].get(k) for k in
                                       ("sm_mhz", "sm_min_mhz", "samples", "reasons")},
                            "config": config_of(s, world)}
            if r.get("backward"):
                side[s.name]["backward"] = r["backward"]

    if rank == 0:
        per_step = res.get("gpu_launches_per_step", -1)
        line = {
            "metric": metric_name(spec),
            "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if spec.dtype == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1) activations, N(0,1/d_in) weights)",
            "config": config_of(spec, world),
            "layer": dict(res["layer"], phase_ms=res["phase_ms"],
                          phase_roofline=res["phase_roofline"], shared_phase=res["shared_phase"],
                          timed_region_ms=res["timed_region_ms"]),
            "roofline": roofline_of(spec, res, peaks, peak_src),
            "clocks": res["clocks"],
            "e2e": res["e2e"],
            "gpu_launches": per_step * args.steps if per_step > 0 else None,
            "gpu_launches_per_step": per_step,
            "cpu_baseline": res.get("cpu_baseline"),
            "cpu_baseline_one_core": res.get("cpu_baseline_one_core"),
            "workloads": side or None,
        }
        if res.get("backward"):
            line["backward"] = res["backward"]
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args, spec, rank, world):
    """The CPU oracle timed on this machine's host cores on the same workload and metric.  Each step
    is one sub-batch of the workload (as many tokens as the box has cores, routed as a batch of
    its own); ms_per_step is the measured time of one such step."""
    if rank != 0:
        return
    layer = moe_synth.make_layer(spec, seed=0, device="cpu")
    for _ in range(args.warmup):
        cpu_oracle_rate(spec, layer, 0.0, max_steps=1)
    step_s, total = [], 0
    sub = cores = 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rate, done, secs, sub, cores = cpu_oracle_rate(spec, layer, 0.0, max_steps=1)
        step_s.append(time.perf_counter() - t0)
        total += done
    value = total / sum(step_s)
    line = {
        "impl": "reference", "metric": metric_name(spec), "value": value,
        "unit": "tokens/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(step_s), "tokens_per_step": sub,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle experts, fp32 router)", "data": "synthetic",
        "config": config_of(spec, 1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{total} tokens of {spec.name}: {args.steps} steps, each "
                                   f"{cpu_sample_note(spec, sub)}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
