"""Benchmark of the MoE layer forward on B300: tokens/s and each expert FFN's roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|mixtral|...] [--impl ours|reference]

One step = one moe_forward call: the whole layer (router + top-k, dispatch + permute, grouped
expert FFN, combine, auxiliary value) over one batch of the workload's seeded synthetic inputs,
with weights and inputs resident in HBM. Each rank (one process per GPU, launched by torchrun for N > 1) runs
an independent replica of the layer on its own batch: there is no exchange on this path, so the
scaling is weak and `value` is the tokens of all ranks over the slowest rank's time.

By default (`--workload all`) the run times all five workloads one after another, each for K
steps after W warm-up steps, and prints ONE line: the Mixtral-shape layer is the headline (its
keys at the top level) and every workload's own measurements sit under `workloads`.

Each measurement carries:
  e2e          the same metric through the C-ABI pipeline (moe_pipeline_submit) with host
               buffers: every step copies its pinned h in and its y (plus aux) out inside the
               timed region, the copies of neighbouring steps overlapping the layer computation;
  roofline     the dominant kernel (the grouped expert FFN, launched twice per step: GEMM1 and
               GEMM2) over its CUDA-event duration, recorded by moe_forward_events on the
               launching stream inside the timed region: algorithmic flops against the bf16
               tensor peak when the FFN's flops per HBM byte exceed the ridge point, else its
               algorithmic bytes against the measured HBM copy bandwidth (f32 layers: flops
               against the FP32 FFMA rate measured in the same run). The tensor peak is the burst
               figure unless the timed region ran under the power cap for a second or more, or
               with its median SM clock at most 0.8 of the maximum (then the sustained figure,
               itself measured under the cap); `frac_alt` gives the fraction against the other;
  cpu_baseline the double-precision oracle on this machine's host cores (rank 0, N = 1 only):
               routing over all T tokens plus the expert MLPs and combine of a token sample,
               extrapolated to T tokens;
  graph        the same step recorded once in a CUDA graph (Layer.capture) and replayed K times:
               the launch-bound shapes' time without host launch cost;
  clocks       nvidia-smi samples taken during the timed region;
  backward     K moe_backward calls after moe_forward_train (which keeps the first GEMM's
               pre-activations; f32 layers: after moe_forward, recomputing them), for an upstream
               gradient dy ~ N(0, 1) with auxiliary and z-loss weights: ms per step, tokens/s and
               the roofline of the whole backward (algorithmic work: the data and weight
               gradients of the expert GEMMs, twice the forward's flops); train_step times K
               forward + backward pairs.
--impl reference times the oracle itself (the method's plain statement) as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_70_b300 import workloads as wl  # noqa: E402

METRIC = "MoE layer tokens/s at 1 B300; % of bf16 TC peak (GEMM) or HBM BW (decode)"
HEADLINE = "mixtral"
ORDER = ["mixtral", "many_small", "switch", "decode", "micro"]
# DRAM bytes (read + write) per launch of the dominant kernel, averaged over its two launches
# (GEMM1, GEMM2), from ncu captures of the current kernels. `scale` says how the figure relates
# to the full workload: "full" = captured at the full shape; otherwise captured on a reduced case
# and scaled by the experts and rows processed (the traffic grows in proportion: weights once,
# activations once).
MEASURED_TRAFFIC = {
    "mixtral": {"bytes": 1.76e9, "scale": "ncu capture of a reduced case (T=2048, E=2, k=1: 2 of "
                                          "8 experts, 2048 of 8192 rows), scaled x4"},
    "switch": {"bytes": 1.39e9, "scale": "ncu capture of a reduced case (T=16384, E=64: half the "
                                         "experts and rows), scaled x2"},
    "decode": {"bytes": 1.42e9, "scale": "ncu capture of a reduced case (T=16, E=4: half the "
                                         "experts and rows), scaled x2"},
}
GEMM_KERNEL = "grouped_gemm_pair_kernel / grouped_gemm_tc_kernel"
F32_KERNEL = "ffn_f32_kernel (CUDA-core FFMA)"
# A timed region at least this long and capped by power is "sustained"; anything shorter, or
# without sw_power_cap in its clock samples, runs at the burst rate.
SUSTAINED_REGION_S = 1.0


def _peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return dict(bf16=p["bf16_tflops"], bf16_sustained=p["bf16_tflops_sustained"],
                    hbm=p["hbm_gbs"], source="measured")
    return dict(bf16=1800.0, bf16_sustained=1400.0, hbm=6400.0, source="fallback")


# ... or a region whose median SM clock sat at or below this fraction of the maximum under the
# power cap (the sustained peak was measured at 1170 of 2032 MHz).
SUSTAINED_CLOCK_FRAC = 0.8


def _tc_peak(peaks: dict, region_s: float, reasons, clocks: dict | None = None) -> tuple:
    """(peak, other peak, kind, other kind): the sustained tensor peak for a region that ran under
    the power cap for a second or more, or with its median SM clock pulled down to at most
    SUSTAINED_CLOCK_FRAC of the maximum; else the burst peak."""
    capped = "sw_power_cap" in set(reasons or ())
    low_clock = bool(clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz") and
                     clocks["sm_mhz"] <= SUSTAINED_CLOCK_FRAC * clocks["sm_max_mhz"])
    sustained = capped and (region_s >= SUSTAINED_REGION_S or low_clock)
    if sustained:
        return peaks["bf16_sustained"], peaks["bf16"], "bf16 sustained", "bf16 burst"
    return peaks["bf16"], peaks["bf16_sustained"], "bf16 burst", "bf16 sustained"


# weights of the auxiliary value and of the z-loss in the loss the backward differentiates
BWD_AUX_WEIGHT, BWD_ZLOSS_WEIGHT = 0.01, 0.001


def backward_roofline(w, bwd_ms: float, peaks: dict, region_s: float, reasons,
                      alu: dict | None = None, clocks: dict | None = None) -> dict:
    """The backward's roofline entry. Algorithmic flops: the expert GEMMs' data gradients (dX,
    dHact) and weight gradients, twice the forward's; algorithmic bytes: every expert's weights
    read and its weight gradients written once, plus h, dy and dh. The bound is the tensor peak
    when flops per byte exceed the ridge point, else the HBM copy bandwidth."""
    flops = 2 * w.expert_flops()
    es = 4 if w.dtype == "f32" else 2
    nbytes = 2 * w.weight_bytes() + 3 * w.T * w.d * es
    sec = bwd_ms * 1e-3
    tflops, gbs = flops / sec / 1e12, nbytes / sec / 1e9
    tc_peak, tc_alt, kind, alt_kind = _tc_peak(peaks, region_s, reasons, clocks)
    common = {"algorithmic_flops": flops, "algorithmic_bytes": nbytes,
              "flop_per_byte": flops / nbytes, "region_s": region_s}
    if w.dtype == "f32":  # CUDA-core FFMA against the measured FP32 rate
        rate = alu["tflops"]
        if flops / nbytes >= rate * 1e12 / (peaks["hbm"] * 1e9):
            return {"bound": "alu", "achieved": tflops, "peak": rate, "unit": "TFLOP/s",
                    "frac": tflops / rate, "peak_kind": alu["how"], "hbm_gbs": gbs, **common}
        return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": gbs / peaks["hbm"], "peak_kind": f"HBM copy ({peaks['source']})",
                "alu_tflops": tflops, **common}
    if flops / nbytes >= tc_peak * 1e12 / (peaks["hbm"] * 1e9):
        return {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": tflops / tc_peak, "peak_kind": f"{kind} ({peaks['source']})",
                "frac_alt": tflops / tc_alt, "frac_alt_kind": alt_kind, "hbm_gbs": gbs, **common}
    return {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": gbs / peaks["hbm"], "peak_kind": f"HBM copy ({peaks['source']})",
            "tensor_tflops": tflops, **common}


def roofline(w, ffn_ms: float, peaks: dict, region_s: float, reasons, alu: dict | None = None,
             traffic: dict | None = None, clocks: dict | None = None) -> dict:
    """The expert FFN's roofline entry.

    w: the workload (its algorithmic flops and bytes); ffn_ms: the FFN's live duration per step
    (both launches); peaks: tensor (burst, sustained) and HBM peaks; region_s / reasons: length
    of the timed region and the clock-event reasons seen in it; alu: {"tflops": measured FP32
    FFMA rate, "how": ...} for f32 layers; traffic: {"bytes": DRAM bytes per launch, "scale": how
    it was taken} or None.
    """
    flops, nbytes = w.expert_flops(), w.ffn_bytes()
    launches = 2
    tflops = flops / (ffn_ms * 1e-3) / 1e12
    gbs = nbytes / (ffn_ms * 1e-3) / 1e9
    intensity = flops / nbytes
    tc_peak, tc_alt, tc_kind, alt_kind = _tc_peak(peaks, region_s, reasons, clocks)
    common = {"flop_per_byte": intensity, "launches_per_step": launches,
              "algorithmic_flops_per_launch": flops / launches,
              "algorithmic_bytes_per_launch": nbytes / launches,
              "traffic": traffic["bytes"] if traffic else None,
              "traffic_source": traffic["scale"] if traffic else None,
              "region_s": region_s}
    if w.dtype == "f32":
        rate = alu["tflops"]
        if intensity >= rate * 1e12 / (peaks["hbm"] * 1e9):
            return {"bound": "alu", "kernel": F32_KERNEL, "achieved": tflops, "peak": rate,
                    "unit": "TFLOP/s", "frac": tflops / rate, "peak_kind": alu["how"],
                    "hbm_gbs": gbs, **common}
        return {"bound": "hbm", "kernel": F32_KERNEL, "achieved": gbs, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": gbs / peaks["hbm"],
                "peak_kind": f"HBM copy ({peaks['source']})", "alu_tflops": tflops, **common}
    ridge = tc_peak * 1e12 / (peaks["hbm"] * 1e9)
    if intensity >= ridge:
        return {"bound": "tensor", "kernel": GEMM_KERNEL, "achieved": tflops, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": tflops / tc_peak,
                "peak_kind": f"{tc_kind} ({peaks['source']})", "frac_alt": tflops / tc_alt,
                "frac_alt_kind": alt_kind, "hbm_gbs": gbs, **common}
    return {"bound": "hbm", "kernel": GEMM_KERNEL, "achieved": gbs, "peak": peaks["hbm"],
            "unit": "GB/s", "frac": gbs / peaks["hbm"],
            "peak_kind": f"HBM copy ({peaks['source']})", "tensor_tflops": tflops,
            "tensor_frac": tflops / tc_peak, "tensor_peak_kind": tc_kind, **common}


class Clocks:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
            os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


class OracleRun:
    """The oracle (double, OpenMP over rows) on the host cores for one workload: routing (router,
    top-k, gates, dispatch, aux) over all T tokens, then the expert MLPs and combine over the first
    n tokens; a run's tokens/s is T / (routing time + the n tokens' time scaled to T tokens)."""

    def __init__(self, w, inputs: dict):
        import oracle
        self.oracle = oracle
        self.w, self.inputs = w, inputs
        self.threads = oracle.max_threads()

    def run(self, n: int) -> dict:
        oracle, w, inputs = self.oracle, self.w, self.inputs
        t0 = time.perf_counter()
        r = oracle.route(w, inputs)
        t_route = time.perf_counter() - t0
        keep = None if r["capacity"] < 0 else (r["slot_of"] >= 0).reshape(w.T, w.k)
        toks = torch.arange(n, dtype=torch.int64).numpy()
        t1 = time.perf_counter()
        oracle.forward_rows(toks, inputs["h"], r["idx"], r["g"], inputs["W1"], inputs.get("W3"),
                            inputs["W2"], inputs.get("b1"), inputs.get("b2"), oracle.act_code(w),
                            keep=keep)
        t_rows = time.perf_counter() - t1
        total = t_route + t_rows * w.T / n
        return {"value": w.T / total, "unit": "tokens/s", "cores": self.threads, "kind": "oracle",
                "sample": f"{w.name}: routing (router, top-k, gates, dispatch, aux) over all {w.T} "
                          f"tokens in {t_route:.2f} s, expert MLPs + combine over the first {n} "
                          f"tokens in {t_rows:.2f} s, scaled to {w.T} tokens: {total:.1f} s of "
                          f"double-precision work on {self.threads} threads",
                "seconds": t_route + t_rows}

    def calibrate(self, budget_s: float) -> int:
        """The token count n whose run takes about budget_s (between a half and all of it)."""
        n = 1
        t = self.run(n)["seconds"]
        while t < budget_s / 8 and n < self.w.T:
            n = min(self.w.T, n * 4)
            t = self.run(n)["seconds"]
        if t < budget_s / 2 and n < self.w.T:
            n = min(self.w.T, max(n + 1, int(n * (budget_s * 0.75) / max(t, 1e-3))))
        return n


def _cpu_baseline(w, inputs: dict, budget_s: float = 12.0) -> dict:
    """The oracle on a bounded sample of workload w (see OracleRun), about budget_s seconds."""
    o = OracleRun(w, inputs)
    out = o.run(o.calibrate(budget_s / 2))
    out.pop("seconds")
    return out


def run_reference(args, todo) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = todo[0] if len(todo) == 1 else wl.WORKLOADS[HEADLINE]
    inputs = wl.generate(w)
    # every step: routing over all T tokens plus the expert MLPs of a token sample, sized once so
    # that all warm-up and timed steps together take about two minutes
    o = OracleRun(w, inputs)
    n = o.calibrate(max(0.02, 120.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        o.run(n)
    t0 = time.perf_counter()
    vals = [o.run(n) for _ in range(args.steps)]
    dt = time.perf_counter() - t0
    value = len(vals) / sum(1.0 / v["value"] for v in vals)   # T tokens per step, harmonic mean
    cb = dict(vals[-1])
    cb.pop("seconds")
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * w.T / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, N(0,1/fan_in))",
            "config": _config(w, args.gpus), "wall_s": dt, "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config(w, world: int) -> dict:
    return {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "E": w.E, "k": w.k, "act": w.act,
            "gate": w.gate, "per_rank_tokens": w.T, "parallelism": f"replicas x{world}",
            "l2": "working set smaller than L2: each step bracketed by its own events, L2 "
                  "flushed between steps (256 MB written outside the events)" if _l2_resident(w)
                  else
                  f"inputs larger than L2 ({w.weight_bytes() / 1e9:.3f} GB of expert weights read "
                  "every step), steps back to back"}


def _l2_resident(w) -> bool:
    """Whether the layer's weights and activations fit in the 126 MB L2 (then steps are timed
    one at a time with L2 flushed in between)."""
    es = 4 if w.dtype == "f32" else 2
    return w.weight_bytes() + w.T * w.d * es * 2 + w.P * (2 * w.d + w.f) * es < 126e6


def _ffma_rate(local: int) -> dict:
    """The FP32 FFMA rate of this GPU, measured by libmoe's probe kernel (CUDA events)."""
    from sparse_mixture_experts_70_b300 import binding as B
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    blocks, threads, iters = sms * 4, 512, 4096
    flops = B.moe_fp32_ffma_probe(blocks, threads, iters, out)   # warm-up, and the flop count
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = math.inf
    for _ in range(5):
        e0.record()
        B.moe_fp32_ffma_probe(blocks, threads, iters, out)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    rate = flops / (best * 1e-3) / 1e12
    return {"tflops": rate, "how": f"FP32 FFMA, measured: moe_fp32_ffma_probe ({blocks} blocks x "
                                   f"{threads} threads, 8 chains x {iters * 16} FMAs), best of 5"}


def bench_workload(w, args, peaks, D, B, local, world, alu=None, cpu_budget_s=0.0) -> dict:
    """One workload: K timed moe_forward calls (+ live FFN events), the host-buffer pipeline,
    the CUDA-graph replay; returns its measurement entry (rank 0 reads it)."""
    cfg = B.config_for(w)
    inputs = wl.generate(w)
    dev = {k: (v.cuda().contiguous() if v is not None else None) for k, v in inputs.items()}
    T, d = w.T, w.d
    stream = torch.cuda.current_stream()
    layer = B.Layer(cfg, dev)          # weights resident, workspace and outputs preallocated
    h = dev["h"]

    for _ in range(args.warmup):
        layer.forward(h, stream)
    torch.cuda.synchronize()
    st = B.moe_device_status(layer.ws)
    if st != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after warm-up: {B.status_string(st)}")

    # A layer whose working set fits in L2 (the micro shape) is timed step by step with L2
    # flushed in between (a 256 MB buffer written between the step's events, queued on the same
    # stream); the larger layers stream more than L2 holds every step and run back to back.
    flush = (torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if _l2_resident(w)
             else None)

    def new_events(n):
        """n pairs of timing events, created (first record) outside any timed region."""
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(n)]
        for e0, e1 in pairs:
            e0.record(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        return pairs

    def timed(step, n, stream_):
        """ms per step of n calls of step(i) on stream_ (mean; events on stream_). With L2
        flushes, every step is bracketed by its own events and the flush kernel runs between
        steps, outside them; the host queues all n steps before waiting once."""
        if flush is None:
            (t0, t1), = new_events(1)
            t0.record(stream_)
            for i in range(n):
                step(i)
            t1.record(stream_)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / n
        pairs = new_events(n)
        for i in range(n):
            flush.zero_()
            pairs[i][0].record(stream_)
            step(i)
            pairs[i][1].record(stream_)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in pairs) / n

    # Timed region: K calls of moe_forward (the call a user makes); each also records two events
    # on its stream around the expert-FFN launches, the dominant kernel's live duration.
    evs = new_events(args.steps)
    with Clocks(local) as clk:
        D.barrier()
        torch.cuda.synchronize()
        ms = timed(lambda i: layer.forward(h, stream, ffn_events=evs[i]), args.steps, stream)
        D.barrier()
    clocks = clk.summary()
    ffn_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
    st = B.moe_device_status(layer.ws)
    if st != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after timed region: {B.status_string(st)}")

    # end to end through the C-ABI pipeline with host buffers (pinned): every step copies its h in
    # and its y + aux out; the copies of neighbouring steps overlap the layer computation
    h_host = inputs["h"].pin_memory()
    y_host = torch.empty((T, d), dtype=w.torch_dtype).pin_memory()
    aux_host = torch.empty(1, dtype=torch.float32).pin_memory()
    pipe = B.Pipeline(cfg, layer.w, stream=stream)
    for _ in range(args.warmup):
        pipe.submit(h_host, y_host, aux_host)
    if pipe.device_status() != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after e2e warm-up")

    def e2e_step(i):
        pipe.submit(h_host, y_host, aux_host)
        if flush is not None or i == args.steps - 1:
            pipe.join(stream)

    D.barrier()
    e_ms = timed(e2e_step, args.steps, stream)
    if pipe.device_status() != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after e2e region")
    pipe.close()

    # the same step recorded once in a CUDA graph and replayed (host launch cost removed)
    graph = layer.capture(dev["h"])
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    D.barrier()
    g_ms = timed(lambda i: graph.replay(), args.steps, torch.cuda.current_stream())
    if B.moe_device_status(layer.ws) != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after graph region")
    del graph
    bwd = (bench_backward(w, args, layer, h, stream, peaks, D, B, local, timed, alu)
           if not args.no_backward else None)
    del flush

    ms, e_ms, ffn_ms, g_ms = D.max_over_ranks([ms, e_ms, ffn_ms, g_ms], device="cuda")
    launches_per_step = B.moe_forward_launch_count(cfg)
    region_s = ms * args.steps * 1e-3
    traffic = None if args.override else MEASURED_TRAFFIC.get(w.name)
    entry = {
        "value": D.job_tokens_per_s(T, world, ms),
        "unit": "tokens/s",
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "dtype": w.dtype,
        "config": _config(w, world),
        "breakdown_ms": {"expert_ffn": ffn_ms, "router_dispatch_combine_aux": ms - ffn_ms},
        "roofline": roofline(w, ffn_ms, peaks, region_s, clocks.get("reasons"), alu, traffic,
                             clocks),
        "e2e": {"value": D.job_tokens_per_s(T, world, e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": T * d * inputs["h"].element_size(),
                "d2h_bytes_per_step": T * d * layer.y.element_size() + 4},
        "gpu_launches": launches_per_step * args.steps,
        "graph": {"value": D.job_tokens_per_s(T, world, g_ms), "unit": "tokens/s",
                  "ms_per_step": g_ms},
        "clocks": clocks,
    }
    if bwd is not None:
        entry["backward"] = bwd
    del layer, dev
    torch.cuda.empty_cache()
    if world == 1 and cpu_budget_s > 0:
        entry["cpu_baseline"] = _cpu_baseline(w, inputs, budget_s=cpu_budget_s)
    return entry


def bench_backward(w, args, layer, h, stream, peaks, D, B, local, timed, alu=None) -> dict:
    """The backward of workload w for a seeded dy ~ N(0, 1): K moe_backward calls after one
    moe_forward_train of h (the routing they differentiate at and the saved pre-activations;
    f32 layers: moe_forward, the backward recomputing them), then K training steps (forward +
    backward); returns the measurement entry."""
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 1000)
    dy = torch.randn((w.T, w.d), generator=g, device="cuda").to(w.torch_dtype)
    f32 = w.dtype == "f32"
    fwd = (lambda: layer.forward(h, stream)) if f32 else (lambda: layer.forward_train(h, stream))
    fwd()
    bwd = lambda i: layer.backward(h, dy, BWD_AUX_WEIGHT, BWD_ZLOSS_WEIGHT, stream)  # noqa: E731

    def train(i):
        fwd()
        bwd(i)

    for i in range(args.warmup):
        bwd(i)
    torch.cuda.synchronize()
    if B.moe_device_status(layer.ws) != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after backward warm-up")
    with Clocks(local) as clk:
        D.barrier()
        torch.cuda.synchronize()
        ms = timed(bwd, args.steps, stream)
        D.barrier()
    clocks = clk.summary()
    for i in range(args.warmup):
        train(i)
    torch.cuda.synchronize()
    D.barrier()
    t_ms = timed(train, args.steps, stream)
    if B.moe_device_status(layer.ws) != B.MOE_OK:
        raise SystemExit(f"{w.name}: device status after the backward regions")
    ms, t_ms = D.max_over_ranks([ms, t_ms], device="cuda")
    world = D.env()[1]
    launches = B.moe_backward_launch_count(layer.cfg, not f32)
    fwd_launches = B.moe_forward_launch_count(layer.cfg)
    del layer.bws, layer.grads
    layer.bws = layer.grads = None
    return {"value": D.job_tokens_per_s(w.T, world, ms), "unit": "tokens/s",
            "ms_per_step": ms, "steps": args.steps,
            "pre_activations": "recomputed" if f32 else "saved by the forward",
            "aux_weight": BWD_AUX_WEIGHT, "zloss_weight": BWD_ZLOSS_WEIGHT,
            "roofline": backward_roofline(w, ms, peaks, ms * args.steps * 1e-3,
                                          clocks.get("reasons"), alu, clocks),
            "gpu_launches": launches * args.steps, "launches_per_step": launches,
            "train_step": {"value": D.job_tokens_per_s(w.T, world, t_ms), "unit": "tokens/s",
                           "ms_per_step": t_ms,
                           "what": ("moe_forward + moe_backward" if f32 else
                                    "moe_forward_train + moe_backward") + ", one call each",
                           "gpu_launches": (launches + fwd_launches) * args.steps},
            "clocks": clocks}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="all", choices=["all"] + list(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward measurement")
    ap.add_argument("--override", default="",
                    help="reshape the workload for profiling, e.g. T=2048,E=2,k=1 (not a bench line)")
    args = ap.parse_args()
    names = ORDER if args.workload == "all" else [args.workload]
    todo = [wl.WORKLOADS[n] for n in names]
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        todo = [w.with_(name=w.name + "_override",
                        **{k_: (float(v) if "." in v or "e" in v else int(v))
                           for k_, v in kv.items()}) for w in todo]
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args, todo)
        return

    from sparse_mixture_experts_70_b300 import binding as B
    from sparse_mixture_experts_70_b300 import dist as D

    rank, world, local = D.env()
    torch.cuda.set_device(local)
    if world > 1:
        D.init("nccl", torch.device("cuda", local))

    peaks = _peaks()
    alu = _ffma_rate(local) if any(w.dtype == "f32" for w in todo) else None
    entries = {}
    for w in todo:
        headline = w.name.split("_override")[0] == HEADLINE or len(todo) == 1
        budget = 0.0 if args.no_cpu_baseline else (12.0 if headline else 3.0)
        entries[w.name] = bench_workload(w, args, peaks, D, B, local, world, alu, budget)
    if rank != 0:
        D.shutdown()
        return

    head_name = next((n for n in entries if n.split("_override")[0] == HEADLINE),
                     next(iter(entries)))
    head = entries[head_name]
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": head["dtype"],
        "data": "synthetic (seeded; h ~ N(0,1), weights ~ N(0, 1/fan_in))",
        "config": head["config"],
        "breakdown_ms": head["breakdown_ms"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "gpu_launches_all_workloads": sum(e["gpu_launches"] for e in entries.values()),
        "graph": head["graph"],
        "clocks": head["clocks"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if "backward" in head:
        line["backward"] = head["backward"]
    if alu is not None:
        line["fp32_ffma_tflops"] = alu
    if len(entries) > 1:
        line["workloads"] = entries
    print(json.dumps(line), flush=True)
    D.shutdown()


if __name__ == "__main__":
    main()
