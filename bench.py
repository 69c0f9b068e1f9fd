"""Benchmark of the MoE layer forward on B300: tokens/s and the grouped expert GEMM's roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixtral] [--impl ours|reference]

One step = one moe_forward call: the whole layer (router + top-k, dispatch + permute, grouped
expert FFN, combine, auxiliary value) over one batch of the workload's seeded synthetic inputs,
with weights and inputs resident in HBM. Each rank (one process per GPU, launched by torchrun for N > 1) runs
an independent replica of the layer on its own batch: there is no exchange on this path, so the
scaling is weak and `value` is the tokens of all ranks over the slowest rank's time.

The JSON line also carries:
  e2e          the same metric through the C-ABI pipeline (moe_pipeline_submit) with host
               buffers: every step copies its pinned h in and its y (plus aux) out inside the
               timed region, the copies of neighbouring steps overlapping the layer computation;
  roofline     the dominant kernel (the grouped expert GEMM, launched twice per step: GEMM1 and
               GEMM2) over its CUDA-event duration, recorded by moe_forward_events on the
               launching stream inside the timed region: algorithmic flops against the measured
               bf16 tensor peak when the FFN's flops per HBM byte exceed the ridge point of the
               measured peaks, else its algorithmic bytes against the measured HBM bandwidth;
  cpu_baseline the double-precision oracle on this machine's host cores, on a bounded token
               sample of the same workload (rank 0, N = 1 only);
  graph        the same step recorded once in a CUDA graph (Layer.capture) and replayed K times:
               the launch-bound shapes' time without host launch cost;
  clocks       nvidia-smi samples taken during the timed region.
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
# DRAM bytes (read + write) per launch of the dominant kernel, from the ncu capture summarised in
# profiles/grouped_gemm_pair_T2048_E2_k1.md (a reduced case: 2 of 8 experts, 2048 of 8192 rows),
# scaled to the full Mixtral-shape launch by the experts and rows processed (traffic grows in
# proportion: weights once, activations once). Average of GEMM1 (2.19 GB) and GEMM2 (1.34 GB).
MEASURED_TRAFFIC = {"mixtral": 1.76e9}
GEMM_KERNEL = "grouped_gemm_pair_kernel / grouped_gemm_tc_kernel"
F32_KERNEL = "ffn_f32_kernel (CUDA-core FFMA)"


def _peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return dict(bf16=p["bf16_tflops"], bf16_sustained=p["bf16_tflops_sustained"],
                    hbm=p["hbm_gbs"], source="measured")
    return dict(bf16=1800.0, bf16_sustained=1400.0, hbm=6400.0, source="fallback")


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


def _cpu_baseline(w, budget_s: float = 12.0) -> dict:
    """The oracle (double, OpenMP over rows) on a bounded prefix of the workload's tokens."""
    import oracle
    threads = oracle.max_threads()
    inputs = wl.generate(w)

    def run(n):
        sub = w.with_(T=n)
        part = dict(inputs)
        part["h"] = inputs["h"][:n].contiguous()
        t0 = time.perf_counter()
        oracle.reference(sub, part)
        return time.perf_counter() - t0

    n = 1
    t = run(n)
    while t < budget_s / 8 and n < w.T:
        n = min(w.T, n * 4)
        t = run(n)
    if t < budget_s / 2 and n < w.T:
        n = min(w.T, max(n + 1, int(n * (budget_s / 2) / max(t, 1e-3))))
        t = run(n)
    return {"value": n / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {w.T} tokens of the {w.name} workload, full layer "
                      f"(router, top-k, gates, dispatch, expert MLPs, combine, aux) in double, "
                      f"{t:.1f} s"}


def run_reference(args, w) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    # each step a bounded token sample sized so that all warm-up and timed steps together take
    # about two minutes (a run of the sample takes between half and all of its budget)
    per_step = 120.0 / max(args.steps + args.warmup, 1)
    cb = _cpu_baseline(w, budget_s=max(0.02, per_step))
    n_tok = int(cb["sample"].split()[1])
    sub = w.with_(T=n_tok)
    inputs = wl.generate(w)
    part = dict(inputs)
    part["h"] = inputs["h"][:n_tok].contiguous()
    for _ in range(args.warmup):
        oracle.reference(sub, part)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.reference(sub, part)
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, N(0,1/fan_in))",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "f": w.f, "E": w.E, "k": w.k,
                       "act": w.act, "gate": w.gate, "sample_tokens": n_tok},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="mixtral", choices=list(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--override", default="",
                    help="reshape the workload for profiling, e.g. T=2048,E=2,k=1 (not a bench line)")
    args = ap.parse_args()
    w = wl.WORKLOADS[args.workload]
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        w = w.with_(name=w.name + "_override",
                    **{k_: (float(v) if "." in v or "e" in v else int(v)) for k_, v in kv.items()})
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        run_reference(args, w)
        return

    from sparse_mixture_experts_70_b300 import binding as B
    from sparse_mixture_experts_70_b300 import dist as D

    rank, world, local = D.env()
    torch.cuda.set_device(local)
    if world > 1:
        D.init("nccl", torch.device("cuda", local))

    peaks = _peaks()
    cfg = B.config_for(w)
    inputs = wl.generate(w)
    dev = {k: (v.cuda().contiguous() if v is not None else None) for k, v in inputs.items()}
    T, k, E, d = w.T, w.k, w.E, w.d
    stream = torch.cuda.current_stream()
    layer = B.Layer(cfg, dev)          # weights resident, workspace and outputs preallocated
    h = dev["h"]

    for _ in range(args.warmup):
        layer.forward(h, stream)
    torch.cuda.synchronize()
    st = B.moe_device_status(layer.ws)
    if st != B.MOE_OK:
        raise SystemExit(f"device status after warm-up: {B.status_string(st)}")

    # Timed region: K calls of moe_forward (the call a user makes); each also records two events
    # on its stream around the expert-FFN launches, the dominant kernel's live duration.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        D.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            layer.forward(h, stream, ffn_events=evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
        D.barrier()
    clocks = clk.summary()
    ms = start.elapsed_time(stop) / args.steps
    ffn_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
    st = B.moe_device_status(layer.ws)
    if st != B.MOE_OK:
        raise SystemExit(f"device status after timed region: {B.status_string(st)}")

    # end to end through the C-ABI pipeline with host buffers (pinned): every step copies its h in
    # and its y + aux out; the copies of neighbouring steps overlap the layer computation
    h_host = inputs["h"].pin_memory()
    y_host = torch.empty((T, d), dtype=w.torch_dtype).pin_memory()
    aux_host = torch.empty(1, dtype=torch.float32).pin_memory()
    pipe = B.Pipeline(cfg, layer.w, stream=stream)
    for _ in range(args.warmup):
        pipe.submit(h_host, y_host, aux_host)
    if pipe.device_status() != B.MOE_OK:
        raise SystemExit("device status after e2e warm-up")
    e_start = torch.cuda.Event(enable_timing=True)
    e_stop = torch.cuda.Event(enable_timing=True)
    D.barrier()
    e_start.record(stream)
    for _ in range(args.steps):
        pipe.submit(h_host, y_host, aux_host)
    pipe.join(stream)
    e_stop.record(stream)
    torch.cuda.synchronize()
    e_ms = e_start.elapsed_time(e_stop) / args.steps
    if pipe.device_status() != B.MOE_OK:
        raise SystemExit("device status after e2e region")
    pipe.close()

    # the same step recorded once in a CUDA graph and replayed (host launch cost removed)
    graph = layer.capture(dev["h"])
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    g_start = torch.cuda.Event(enable_timing=True)
    g_stop = torch.cuda.Event(enable_timing=True)
    D.barrier()
    g_start.record()
    for _ in range(args.steps):
        graph.replay()
    g_stop.record()
    torch.cuda.synchronize()
    g_ms = g_start.elapsed_time(g_stop) / args.steps
    if B.moe_device_status(layer.ws) != B.MOE_OK:
        raise SystemExit("device status after graph region")
    del graph

    ms, e_ms, ffn_ms, g_ms = D.max_over_ranks([ms, e_ms, ffn_ms, g_ms], device="cuda")
    if rank != 0:
        D.shutdown()
        return

    # The expert FFN's roofline: tensor-bound when its arithmetic intensity (flops per HBM byte
    # it must move) is above the ridge point of the measured peaks, else HBM-bound (decode).
    flops, nbytes = w.expert_flops(), w.ffn_bytes()
    tflops = flops / (ffn_ms * 1e-3) / 1e12
    gbs = nbytes / (ffn_ms * 1e-3) / 1e9
    intensity = flops / nbytes
    ridge = peaks["bf16_sustained"] * 1e12 / (peaks["hbm"] * 1e9)
    traffic = MEASURED_TRAFFIC.get(w.name if not args.override else "")
    if w.dtype == "f32":
        # f32 experts run as FFMA chains on the CUDA cores: the compute roof is the FP32 ALU rate,
        # SMs x 128 FP32 lanes x 2 flop x the maximum SM clock (derived, not measured)
        sms = torch.cuda.get_device_properties(local).multi_processor_count
        mhz = clocks.get("sm_max_mhz") or 2032.0
        alu = sms * 128 * 2 * mhz * 1e6 / 1e12
        if intensity >= alu * 1e12 / (peaks["hbm"] * 1e9):
            roofline = {"bound": "alu", "kernel": F32_KERNEL, "achieved": tflops, "peak": alu,
                        "unit": "TFLOP/s", "frac": tflops / alu,
                        "peak_kind": f"FP32 FFMA, {sms} SMs x 128 lanes x 2 x {mhz:.0f} MHz "
                                     "(derived)", "traffic": traffic,
                        "flop_per_byte": intensity, "hbm_gbs": gbs}
        else:
            roofline = {"bound": "hbm", "kernel": F32_KERNEL, "achieved": gbs,
                        "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                        "peak_kind": f"HBM copy ({peaks['source']})", "traffic": traffic,
                        "flop_per_byte": intensity, "alu_tflops": tflops}
    elif intensity >= ridge:
        roofline = {"bound": "tensor", "kernel": GEMM_KERNEL, "achieved": tflops,
                    "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                    "frac": tflops / peaks["bf16_sustained"],
                    "peak_kind": f"bf16 sustained ({peaks['source']})",
                    "frac_of_burst": tflops / peaks["bf16"], "traffic": traffic,
                    "flop_per_byte": intensity, "hbm_gbs": gbs}
    else:
        roofline = {"bound": "hbm", "kernel": GEMM_KERNEL, "achieved": gbs, "peak": peaks["hbm"],
                    "unit": "GB/s", "frac": gbs / peaks["hbm"],
                    "peak_kind": f"HBM copy ({peaks['source']})", "traffic": traffic,
                    "flop_per_byte": intensity, "tensor_tflops": tflops}
    # the library's own count of the kernels one moe_forward launches for this config
    launches_per_step = B.moe_forward_launch_count(cfg)
    line = {
        "metric": METRIC,
        "value": D.job_tokens_per_s(T, world, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded; h ~ N(0,1), weights ~ N(0, 1/fan_in))",
        "config": {"workload": w.name, "T": T, "d": d, "f": w.f, "E": E, "k": k,
                   "act": w.act, "gate": w.gate, "per_rank_tokens": T,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({w.weight_bytes() / 1e9:.2f} GB of expert "
                         "weights read every step)"},
        "breakdown_ms": {"expert_ffn": ffn_ms, "router_dispatch_combine_aux": ms - ffn_ms},
        "roofline": roofline,
        "e2e": {"value": D.job_tokens_per_s(T, world, e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": T * d * inputs["h"].element_size(),
                "d2h_bytes_per_step": T * d * layer.y.element_size() + 4},
        "gpu_launches": launches_per_step * args.steps,
        "graph": {"value": D.job_tokens_per_s(T, world, g_ms), "unit": "tokens/s",
                  "ms_per_step": g_ms},
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(w)
    print(json.dumps(line), flush=True)
    D.shutdown()


if __name__ == "__main__":
    main()
