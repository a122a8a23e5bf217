"""Prefill throughput of the dense decoder-layer stack on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one prefill call through the whole stack: every layer's seven
projections, RoPE, attention and SwiGLU over one batch of synthetic input
(seeded, the shapes and distributions of the workload; random weights).
The default workload is the Llama-3.2-3B shape at pp512 (28 layers,
d=3072, 24/8 heads of 128, ffn 8192, 512 new tokens, empty prefix).

* ``value``: tokens/s with weights, caches and the hidden batch resident in
  HBM (device-I/O entry point), timed with CUDA events over exactly K steps
  after W warm-up steps; weights (5.6 GB) exceed the 129 MB L2, so no flush.
* ``e2e``: the same through the host-I/O entry point (pinned host hidden
  batch in, host out; the copies are inside the timed region).
* ``roofline``: the dominant kernel, its algorithmic FLOP (or bytes) per
  launch over its average CUDA-event duration (measured in a pass right
  after the timed region, with per-kernel events on the call's stream),
  against the measured bf16 peak (burst for a timed region shorter than a
  second, else sustained) or, for a workload whose GEMMs stream weights
  (batch below the ridge of the two peaks), the measured HBM bandwidth.
  ``kernels`` gives every kernel kind's achieved TFLOP/s and GB/s.
* ``cpu_baseline``: the fp64 CPU oracle on a bounded sample (the first
  layers of the same workload), extrapolated to the whole stack.

Under torchrun (N > 1) every rank runs an independent replica on its own
GPU (the stack does not shard: no collectives); ``value`` is all ranks'
tokens over the slowest rank's time.  ``--impl reference`` times the CPU
oracle instead (rank 0 only).
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

import synth  # noqa: E402

DEFAULT_WORKLOAD = "llama3.2-3b-pp512"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops(dims):
    """Algorithmic FLOP of one call, per kernel kind and in total."""
    B, s, d, F = dims.batch, dims.start_pos, dims.d_model, dims.ffn_dim
    qw, kvw = dims.q_width, dims.kv_width
    per = {
        "qkv": 2.0 * B * d * (qw + 2 * kvw),
        "attn": 4.0 * dims.n_heads * dims.head_dim * (B * s + B * (B + 1) / 2),
        "wo": 2.0 * B * qw * d,
        "gateup": 2.0 * B * d * 2 * F,
        "down": 2.0 * B * F * d,
    }
    return per, dims.n_layers * sum(per.values())


def weight_bytes_per_layer(dims):
    d, F, qw, kvw = dims.d_model, dims.ffn_dim, dims.q_width, dims.kv_width
    return 2 * (d * (qw + 2 * kvw) + qw * d + 2 * F * d + F * d) + 4 * 2 * d


def algo_bytes(dims):
    """Bytes each kernel kind must move at least once per launch: weights and
    cache rows read, activations read and written (float32 4, bf16 2), once."""
    B, s, d, F, hd = dims.batch, dims.start_pos, dims.d_model, dims.ffn_dim, dims.head_dim
    qw, kvw = dims.q_width, dims.kv_width
    ss = 4 * B * (d // 64)  # row sum-of-squares partials
    return {
        # weights, a, ss in; q and the new k/v rows out
        "qkv": 2 * d * (qw + 2 * kvw) + 2 * B * d + ss + 2 * B * qw + 2 * 2 * B * kvw,
        # q in, every visible K/V row once, o out
        "attn": 2 * B * qw + 2 * 2 * (s + B) * kvw + 2 * B * qw,
        # weights, o in; residual in, h and a = bf16(h*g) and ss out
        "wo": 2 * qw * d + 2 * B * qw + 4 * B * d + 4 * B * d + 2 * B * d + ss,
        # weights, a and ss in; act out
        "gateup": 2 * 2 * F * d + 2 * B * d + ss + 2 * B * F,
        # weights, act in; residual in, x' and a and ss out
        "down": 2 * F * d + 2 * B * F + 4 * B * d + 4 * B * d + 2 * B * d + ss,
        # prep: x and the gain in, a and ss out; the (cos, sin) table out
        "prep": 4 * B * d + 4 * d + 2 * B * d + ss + 8 * B * (hd // 2),
    }


KERNEL_SOURCES = ("gemm_tc.cu", "sm100.cuh", "attn_tc.cu", "prep.cu", "tc.h", "kernels.h",
                  "common.cuh", "fastmath.cuh")


def kernel_source_sha():
    """sha256 prefix of the kernel sources, to tell whether a profile is current."""
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_decoder_layer_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kind, workload):
    """DRAM bytes per launch of one kernel from the committed ncu summary, or
    None when that summary was taken on other kernel sources or workload."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            kv = dict(line.split(None, 1) for line in f
                      if line.strip() and not line.startswith("#"))
    except (OSError, ValueError):
        return None
    if kv.get("source_sha", "").strip() != kernel_source_sha():
        return None
    if kv.get("workload", "").strip() != workload or kind not in kv:
        return None
    return int(kv[kind])


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_layers_timed(dims, layers, pk, pv, hidden, budget_s):
    """Time the oracle layer by layer on the full batch until `budget_s` is spent."""
    import oracle
    x = np.asarray(hidden, np.float64)
    t0 = time.perf_counter()
    n = 0
    while n < dims.n_layers:
        x, _, _ = oracle.prefill_dense_stack(x, [layers[n]], [pk[n]], [pv[n]], dims.start_pos,
                                             dims.n_heads, dims.n_kv_heads, dims.head_dim,
                                             dims.rope_theta, dims.rms_eps)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return time.perf_counter() - t0, n


def run_reference(args, dims, rank):
    """The CPU oracle as the reference arm: each step is the oracle on the
    first `layers` layers of the workload at the full batch, extrapolated."""
    if rank != 0:
        return
    import oracle
    sample_layers = 1
    layers = [synth.draw_layer(dims, l) for l in range(sample_layers)]
    pk, pv = zip(*[synth.draw_prefix(dims, l) for l in range(sample_layers)])
    hidden = synth.draw_hidden(dims)

    def step():
        oracle.prefill_dense_stack(hidden, layers, list(pk), list(pv), dims.start_pos,
                                   dims.n_heads, dims.n_kv_heads, dims.head_dim,
                                   dims.rope_theta, dims.rms_eps)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps * dims.n_layers / sample_layers
    value = dims.batch / dt
    sample = (f"fp64 oracle, first {sample_layers} of {dims.n_layers} layers at B={dims.batch}, "
              f"time x{dims.n_layers // sample_layers} (layers are identical in cost)")
    out = {
        "impl": "reference", "metric": "prefill tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, **_cfg(dims)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def _cfg(dims):
    return {"layers": dims.n_layers, "d_model": dims.d_model, "n_heads": dims.n_heads,
            "n_kv_heads": dims.n_kv_heads, "head_dim": dims.head_dim, "ffn_dim": dims.ffn_dim,
            "batch": dims.batch, "start_pos": dims.start_pos, "rope_theta": dims.rope_theta}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.CONFIGS))
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers (small cases for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    dims = synth.CONFIGS[args.workload]
    if args.layers:
        dims = dims.replace(n_layers=args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, dims, rank)
        return

    import torch
    import torch.distributed as dist
    from dense_decoder_layer_gb300 import pds
    from dense_decoder_layer_gb300.stack import DenseStack

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    layers, pk, pv, hidden = synth.draw_workload(dims)
    st = DenseStack(dims, dims.start_pos + dims.batch, dims.batch)
    st.load_layers(layers)
    st.load_prefix(pk, pv)
    stream = torch.cuda.current_stream()
    x_dev = torch.from_numpy(hidden).cuda()
    out_dev = torch.empty_like(x_dev)
    B, s = dims.batch, dims.start_pos

    from dense_decoder_layer_gb300 import replicas

    barrier = replicas.barrier

    def step():
        st.prefill_device(x_dev, s, out_dev)

    for _ in range(args.warmup):
        step()
    st.sync()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    st.sync()
    ms, value = replicas.aggregate(e0.elapsed_time(e1), B * args.steps)
    ms_per_step = ms / args.steps

    # end to end through the host-I/O entry point (pinned host buffers)
    h_in = torch.from_numpy(hidden).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    for _ in range(2):
        st.prefill(h_in, s, out=h_out)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        st.prefill(h_in, s, out=h_out)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    e2e_ms, e2e_value = replicas.aggregate(max(e0.elapsed_time(e1), wall * 1e3), B * args.steps)

    # per-kernel durations: same steps with events around every kernel
    pds.pds_plan_set_timing(st.plan, True)
    pds.pds_plan_kernel_times(st.plan, stream.cuda_stream, reset=True)
    for _ in range(args.steps):
        step()
    kt = pds.pds_plan_kernel_times(st.plan, stream.cuda_stream, reset=True)
    pds.pds_plan_set_timing(st.plan, False)
    per_flop, total_flop = flops(dims)
    per_bytes = algo_bytes(dims)
    peaks, peak_src = read_peaks()
    # A kernel timed inside a timed region shorter than a second runs at the
    # burst clocks: its denominator is the burst peak (the sustained one is
    # printed beside it).
    timed_s = ms_per_step * args.steps / 1e3
    burst = timed_s < 1.0
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sust = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_tf = peak_burst if burst else peak_sust
    peak_gbs = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kernels = {}
    for kind, (n, tot) in kt.items():
        if n == 0:
            continue
        avg_ms = tot / n
        k = {"launches": n, "avg_us": avg_ms * 1e3, "share": None,
             "gbs": per_bytes[kind] / (avg_ms / 1e3) / 1e9}
        if kind in per_flop:
            k["tflops"] = per_flop[kind] / (avg_ms / 1e3) / 1e12
        k["hbm_frac"] = k["gbs"] / peak_gbs
        kernels[kind] = k
    tot_all = sum(v[1] for v in kt.values()) or 1.0
    for kind, k in kernels.items():
        k["share"] = kt[kind][1] / tot_all
    gemm_kinds = [k for k in ("qkv", "wo", "gateup", "down") if k in kernels]
    dom = max(gemm_kinds, key=lambda k: kt[k][1])
    gemm_ms = sum(kt[k][1] for k in gemm_kinds) / args.steps
    gemm_flop = dims.n_layers * sum(per_flop[k] for k in gemm_kinds)
    # a GEMM of M rows does M flop per weight byte: below the ridge of the
    # measured peaks (flop per byte at which both peaks meet) it streams
    # weights and is bound by HBM, above it by the tensor cores
    ridge = peak_tf * 1e12 / (peak_gbs * 1e9)
    hbm_bound = dims.batch < ridge
    if hbm_bound:
        roofline = {
            "kernel": f"gemm_{dom}", "bound": "hbm",
            "achieved": kernels[dom]["gbs"], "peak": peak_gbs, "unit": "GB/s",
            "frac": kernels[dom]["gbs"] / peak_gbs,
            "peak_source": f"{peak_src} hbm_gbs",
        }
    else:
        roofline = {
            "kernel": f"gemm_{dom}", "bound": "tensor",
            "achieved": kernels[dom]["tflops"], "peak": peak_tf, "unit": "TFLOP/s",
            "frac": kernels[dom]["tflops"] / peak_tf,
            "peak_source": f"{peak_src} {'bf16_tflops (burst)' if burst else 'bf16_tflops_sustained'}"
                           f": timed region {timed_s:.2f} s",
            "frac_of_sustained": kernels[dom]["tflops"] / peak_sust,
        }
    roofline.update({
        "traffic": measured_traffic(dom, args.workload), "traffic_unit": "bytes per launch",
        "algorithmic_bytes": per_bytes[dom], "algorithmic_flop": per_flop[dom],
        "gemm_frac": gemm_flop / (gemm_ms / 1e3) / 1e12 / peak_tf,
        # the GEMMs' share of the replayed step: the step less the other
        # kernels' stand-alone times (launch gaps and overlaps go to the GEMMs)
        "gemm_frac_in_step": gemm_flop / ((ms_per_step - sum(
            kt[k][1] for k in kt if k not in gemm_kinds) / args.steps) / 1e3) / 1e12 / peak_tf,
        "end_to_end_frac": total_flop / (ms_per_step / 1e3) / 1e12 / peak_tf,
        # every byte a step must move at least once (weights, caches read,
        # activations in and out) over the step's time, against HBM
        "step_hbm_frac": dims.n_layers * sum(per_bytes[k] for k in per_flop) /
                         (ms_per_step / 1e3) / 1e9 / peak_gbs,
    })
    weight_bytes = dims.n_layers * weight_bytes_per_layer(dims)

    if rank != 0:
        return
    result = {
        "metric": "prefill tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1/in) bf16 weights, N(0,1) hidden)",
        "config": {"workload": args.workload, **_cfg(dims),
                   "l2": (f"inputs larger than L2: {weight_bytes / 1e9:.2f} GB of weights "
                          f"stream every step against a 129 MB L2, no flush"
                          if weight_bytes > 2 * 129e6 else
                          f"{weight_bytes / 1e6:.1f} MB of weights: L2-resident between steps"),
                   "parallelism": f"replicas x{world}"},
        "tflops": total_flop / (ms_per_step / 1e3) / 1e12,
        "us_per_token": ms_per_step * 1e3 / B,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": B * dims.d_model * 4,
                "d2h_bytes_per_step": B * dims.d_model * 4},
        "gpu_launches": args.steps * (2 + 5 * dims.n_layers),
        "roofline": roofline,
        "kernels": kernels,
        "clocks": clock_info,
    }
    if world == 1 and not args.no_cpu_baseline:
        dt, n = oracle_layers_timed(dims, layers, pk, pv, hidden, args.cpu_budget)
        per_call = dt / n * dims.n_layers
        result["cpu_baseline"] = {
            "value": B / per_call, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 oracle, first {n} of {dims.n_layers} layers at B={B}, "
                      f"{dt:.1f} s, extrapolated x{dims.n_layers}/{n} (layers identical in cost)"}
    print(json.dumps(result), flush=True)
    st.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
