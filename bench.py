#!/usr/bin/env python
"""Benchmark of the GB300 latent-MoE layer (one JSON line on stdout).

Workload (default): one decode step of the full layer -- T=1 token, hidden
8192, latent 4096, 256 experts top-8, expert intermediate 4096, MXFP4 W4A16
experts, bf16 pooler/unpooler, fp32 router -- on seeded synthetic inputs.
A "step" is one lmoe_forward (router, top-k, table, pooler, experts,
post_expert_norm, weighted sum, unpooler) over one batch of T tokens.

  value   tokens/s of the whole job (all ranks), inputs resident in HBM,
          device time from CUDA events, L2 flushed (512 MB write) between steps
          outside the timed events
  e2e     same metric with the x upload from pinned host memory and the
          output download inside the timed region: lmoe_forward_host (copy
          kernels over the host link) for the one-layer MXFP4 layer, else
          copy-engine transfers around the device call
  roofline  the dominant kernel (largest device time) timed live with per-launch
          CUDA events: algorithmic bytes per launch / mean launch duration,
          against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle, as it stands, on a bounded sample of the same
          workload on this host's cores

--impl reference times the CPU oracle (the only reference this layer has) on
the same workload and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank runs an independent replica (the layer is
not sharded at these sizes); value = tokens of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "latent-MoE layer tokens/s and HBM GB/s (frac of roofline) at T=1..4096"
EXPERT_BYTES = 26_738_688          # one expert: 3 matrices x (codes 8 MiB + scales 512 KiB)
EXPERT_BYTES_NVFP4 = 28_311_552    # NVFP4: 3 matrices x (codes 8 MiB + E4M3 scales 1 MiB) (+ 8 B global scales)
GATEUP_BYTES = 2 * EXPERT_BYTES // 3
PROJ_BYTES = 134_217_728           # pooler + unpooler bf16
# source files each measured kernel is built from (the ncu summary's source_sha256 covers these)
KERNEL_SOURCES = {
    "expert_fused": ("fused_experts.cu", "common.cuh"),
    "expert_gateup": ("experts.cu", "common.cuh"),
    "expert_down": ("experts.cu", "common.cuh"),
    "pool_tc_gemm": ("tc_gemm.cu", "tc.cuh", "common.cuh"),
    "unpool_tc_gemm": ("tc_gemm.cu", "tc.cuh", "common.cuh"),
    "expert_gateup_tc": ("tc_experts.cu", "tc.cuh", "common.cuh"),
    "expert_down_tc": ("tc_experts.cu", "tc.cuh", "common.cuh"),
    "pool_gemv": ("gemv.cu", "common.cuh"),
    "unpool_gemv": ("gemv.cu", "common.cuh"),
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_name(d: synth.Dims, name: str) -> str:
    s = " (skewed routing: +3.0 logit bias on experts 0..15)" if d.skewed else ""
    return (f"latent-MoE layer {name}: T={d.T}, hidden {d.H}, latent {d.L}, {d.E} experts top-{d.k}, "
            f"intermediate {d.I}, MXFP4 W4A16 experts, bf16 pooler/unpooler, fp32 router{s}")


def kernel_work(kernel: str, d: synth.Dims, touched: int):
    """Algorithmic (bytes, flops) of one launch of `kernel` on workload d:
    every operand read once, every result written once, 2 flops per MAC."""
    T, H, L, I, k = d.T, d.H, d.L, d.I, d.k
    R = T * k
    if kernel == "expert_fused":  # gate/up + SwiGLU and down in one launch
        return (touched * EXPERT_BYTES + 2 * T * L + 2 * 2 * R * I + 4 * R * L + 4 * R * (L // 32),
                2 * R * 3 * I * L)
    if kernel.startswith("expert_gateup"):
        return touched * GATEUP_BYTES + 2 * T * L + 2 * R * I, 2 * R * 2 * I * L
    if kernel.startswith("expert_down"):
        return touched * (EXPERT_BYTES - GATEUP_BYTES) + 2 * R * I + 4 * R * L, 2 * R * L * I
    if kernel.startswith("pool_"):
        return 2 * L * H + 2 * T * H + 2 * T * L, 2 * T * L * H
    if kernel.startswith("unpool_"):
        return 2 * H * L + 2 * T * L + 2 * T * H, 2 * T * H * L
    return None


def profile_name(kernel: str, config: str) -> str:
    return os.path.join(ROOT, "profiles", f"{kernel}_{config}.txt")


def traffic_from_profiles(kernel: str, config: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary for
    this workload, if it was taken on the current kernel source."""
    p = profile_name(kernel, config)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and not line.startswith("#"):
            key, v = line.split(":", 1)
            vals[key.strip()] = v.strip()
    if vals.get("source_sha256") != kernel_source_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, ()):
        h.update(open(os.path.join(ROOT, "latent_moe_layer_fp32_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples (the JSON line carries their summary); LMOE_CLOCKS_DIR keeps them somewhere chosen
        self.path = os.path.join(os.environ.get("LMOE_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"lmoe_clocks_rank{index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus, backend=None):
    """One process per GPU (torchrun): rank, world and local rank from the
    environment.  The ranks are independent replicas; the process group only
    carries the barrier and the max over ranks of the timed region (nccl on
    GPUs; gloo for the host-side tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = backend or os.environ.get("LMOE_DIST_BACKEND", "nccl")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank: float, seconds: float):
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    total = allreduce_max(world, seconds)
    return units_per_rank * world / total, total


def cpu_oracle_rate(d, hw, x, min_seconds=10.0, max_reps=1000, block_norms=None, nvfp4=False):
    """Tokens/s of the CPU oracle on repeated whole-layer (or whole-block) evaluations of `x`."""
    import oracle
    o = oracle.get()
    reps, t0 = 0, time.perf_counter()
    while reps < max_reps:
        if block_norms is not None:
            o.block_forward(d, x, hw, block_norms)
        elif nvfp4:
            o.forward_nvfp4(d, x, hw)
        else:
            o.forward(d, x, hw)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    return reps * d.T / dt, o.threads, reps, dt


def run_reference(args, d, name, world, rank):
    if rank != 0:
        return
    hw = synth.make_weights(d)
    x = synth.make_x(d)
    import oracle
    o = oracle.get()
    for _ in range(args.warmup):
        o.forward(d, x, hw)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        o.forward(d, x, hw)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * d.T / total
    sample = f"{name}: the whole layer for T={d.T} token(s) per step, full layer shape"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": workload_name(d, name), "T": d.T, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": o.threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_stage(args, d, name, lm, dev):
    """One dense projection call per step on its own (inputs resident, L2
    flushed between steps): the pooler (lmoe_pool) or the post-expert path
    ending in the unpooler (lmoe_norm_combine_unpool: ssq, combine, unpool)."""
    import torch

    def bf_dev(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    T, H, L, k, E = d.T, d.H, d.L, d.k, d.E
    dims = lm.dims_of(T, H, L, d.I, E, k, d.eps)
    ws = torch.empty(lm.lmoe_workspace_bytes(dims), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    if args.stage == "pool":
        x = bf_dev(synth.make_x(d))
        pw = bf_dev(synth.normal_bf16(0, synth.TID_POOLER, (L, H), 0.0, (1.0 / H) ** 0.5))
        x_lat = torch.empty(T, L, dtype=torch.bfloat16, device=dev)

        def call():
            lm.lmoe_pool(dims, x, pw, x_lat, ws)
    else:
        y = torch.from_numpy(synth.normal_f32(0, 21, (T * k, L), 0.0, 1.0)).to(dev)
        # routing: token t takes experts (t + j * E / k) mod E, equal weights (a valid top-k table)
        t_ = np.arange(T)[:, None]
        j_ = np.arange(k)[None, :]
        idx = torch.from_numpy(((t_ + j_ * (E // k)) % E).astype(np.int32)).to(dev)
        tw = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=dev)
        g = bf_dev(synth.normal_bf16(0, synth.TID_GAIN, (E, L), 1.0, 0.1 ** 0.5))
        uw = bf_dev(synth.normal_bf16(0, synth.TID_UNPOOLER, (H, L), 0.0, (1.0 / L) ** 0.5))
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

        def call():
            lm.lmoe_norm_combine_unpool(dims, y, idx, tw, g, uw, out, ws)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
        n = lm.lmoe_last_launch_count()
        names = [lm.lmoe_last_launch_name(j) for j in range(n)]
        per = [[] for _ in range(n)]
        for _ in range(args.steps):
            for j, v in enumerate(per_launch_ms(lm, call, n, 1, flush)):
                per[j] += v
        rc = lm.lmoe_status_check(ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc}: {lm.lmoe_error_string(rc)}")
    pk = peaks()
    kern = names[-1]
    ms = statistics.mean(per[-1])
    nbytes, flops = kernel_work(kern, d, 0)
    print(json.dumps({"stage": args.stage, "config": name, "kernel": kern, "launch_ms": ms,
                      "tflops": flops / (ms / 1e3) / 1e12, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / pk[
                          "bf16_tflops"], "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "peak_source": pk["source"],
                      "kernels_ms": {names[j]: statistics.mean(per[j]) for j in range(n)}}), flush=True)


PER_CONFIG = ["verify_t4", "verify_t8", "verify_t4_skewed", "verify_t8_skewed", "batched_t64", "prefill_t4096"]


def layer_work(d: synth.Dims, touched: int):
    """Algorithmic bytes and flops of one layer step: the decode roofline's
    bytes (touched expert slices + pooler + unpooler weights) and the tensor
    flops (experts, pooler, unpooler; 2 per MAC)."""
    T, H, L, I, k = d.T, d.H, d.L, d.I, d.k
    nbytes = touched * EXPERT_BYTES + PROJ_BYTES
    flops = 2 * T * k * (2 * I * L + L * I) + 2 * 2 * T * H * L
    return nbytes, flops


def layer_fraction(d, touched, ms, pk, tc_peak):
    """The layer's roofline fraction: HBM bytes for a bandwidth-bound step,
    tensor flops against the bf16 peak for a compute-bound one (whichever
    roof the step's arithmetic intensity puts it under)."""
    nbytes, flops = layer_work(d, touched)
    balance = tc_peak * 1e12 / (pk["hbm_gbs"] * 1e9)
    if flops / nbytes > balance:
        ach = flops / (ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s", "frac": ach / tc_peak,
                "algorithmic_flops": flops}
    ach = nbytes / (ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
            "algorithmic_bytes": nbytes}


def dominant_roofline(d, touched, kern_ms, pk, tc_peak, traffic_key):
    """The modelled launch with the largest mean device time, against the
    roof its own arithmetic intensity puts it under."""
    cand = [(ms, n) for n, ms in kern_ms.items() if kernel_work(n, d, touched) is not None]
    dom_ms, dom = max(cand)
    dom_bytes, dom_flops = kernel_work(dom, d, touched)
    balance = tc_peak * 1e12 / (pk["hbm_gbs"] * 1e9)
    if dom_flops / dom_bytes > balance:
        roof = {"bound": "tensor", "achieved": dom_flops / (dom_ms / 1e3) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s", "algorithmic_flops_per_launch": dom_flops}
    else:
        roof = {"bound": "hbm", "achieved": dom_bytes / (dom_ms / 1e3) / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"traffic": traffic_from_profiles(dom, traffic_key), "kernel": dom,
                 "algorithmic_bytes_per_launch": dom_bytes, "launch_ms": dom_ms,
                 "peak_source": pk["source"] + ("" if roof["bound"] == "hbm" else
                                                (" burst" if tc_peak == pk["bf16_tflops"] else " sustained"))})
    return roof


def time_steps(call, steps, flush):
    """Device time of `steps` calls, each after an L2 flush outside the timed events."""
    import torch
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        e0[i].record()
        call()
        e1[i].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(e0, e1)]


def per_launch_ms(lm, call, n_launch, reps, flush):
    """Mean device time of each kernel launch of one call (CUDA events between launches)."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_launch)]
    per = [[] for _ in range(n_launch)]
    lm.lmoe_profile_events(evs)
    try:
        for _ in range(reps):
            flush.zero_()
            call()
            torch.cuda.synchronize()
            for j in range(n_launch):  # events 2j, 2j+1 bracket launch j on its own stream
                per[j].append(evs[2 * j].elapsed_time(evs[2 * j + 1]))
    finally:
        lm.lmoe_profile_events(None)
    return per


def run_per_config(args, lm, w_dev, hw, dev, flush, pk, want_cpu):
    """Every other workload config of the layer, timed like the headline one
    (plain lmoe_forward, inputs resident, L2 flushed between steps): ms per
    step, tokens/s, the layer's roofline fraction, the dominant kernel's
    roofline and the CPU oracle on a bounded token sample."""
    import torch
    res = {}
    steps = max(5, min(args.steps, 20))
    for name in PER_CONFIG:
        d = synth.CONFIGS[name]
        bias = synth.make_router_bias(d)
        w = dict(w_dev)
        w["router_bias"] = None if bias is None else torch.from_numpy(bias).to(dev)
        wts = lm.weights_of(w)
        dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
        ws = torch.empty(lm.lmoe_workspace_bytes(dims), dtype=torch.uint8, device=dev)
        x_np = synth.make_x(d)
        x = torch.from_numpy(x_np.view(np.int16)).to(dev).view(torch.bfloat16)
        out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=dev)

        def call():
            lm.lmoe_forward(dims, wts, x, out, ws)
        for _ in range(max(3, args.warmup)):
            call()
        rc = lm.lmoe_status_check(ws)
        if rc != 0:
            raise RuntimeError(f"{name}: device status {rc}: {lm.lmoe_error_string(rc)}")
        n_launch = lm.lmoe_last_launch_count()
        names = [lm.lmoe_last_launch_name(j) for j in range(n_launch)]
        lay = lm.lmoe_workspace_layout(dims)
        offs = ws[lay.expert_offsets:lay.expert_offsets + 4 * (d.E + 1)].view(torch.int32).cpu().numpy()
        touched = int(np.count_nonzero(np.diff(offs)))
        step_ms = time_steps(call, steps, flush)
        ms = float(np.mean(step_ms))
        per = per_launch_ms(lm, call, n_launch, 5, flush)
        kern_ms = {}
        for j, nm in enumerate(names):  # a name may repeat (e.g. two tensor-core GEMMs): keep both
            key = nm if nm not in kern_ms else f"{nm}#{j}"
            kern_ms[key] = statistics.mean(per[j])
        tc_peak = pk["bf16_tflops"]
        entry = {"workload": workload_name(d, name), "T": d.T, "touched_experts": touched, "ms_per_step": ms,
                 "tokens_per_s": d.T / (ms / 1e3), "launches_per_step": n_launch,
                 "step_ms_percentiles": {"p10": float(np.percentile(step_ms, 10)),
                                         "median": float(np.median(step_ms)),
                                         "p90": float(np.percentile(step_ms, 90))},
                 "layer_roofline": layer_fraction(d, touched, ms, pk, tc_peak),
                 "roofline": dominant_roofline(d, touched, {k.split("#")[0] if "#" in k else k: v
                                                            for k, v in kern_ms.items()}, pk, tc_peak, name),
                 "kernels_ms": kern_ms}
        if want_cpu:
            # the layer is token-independent: the oracle on a bounded sample of the step's tokens
            ns = min(d.T, 8)
            S = np.linspace(0, d.T - 1, ns).astype(np.int64)
            dS = synth.with_tokens(d, ns)
            hws = dict(hw)
            hws["router_bias"] = bias
            rate, cores, reps, dt = cpu_oracle_rate(dS, hws, np.ascontiguousarray(x_np[S]), min_seconds=2.0)
            entry["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                     "sample": f"{reps} whole-layer evaluations of {ns} of the step's {d.T} "
                                               f"token(s) ({dt:.1f} s)"}
        res[name] = entry
        del ws
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode_t1", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--routed", action="store_true",
                    help="time lmoe_forward_routed on a seeded caller-supplied routing (uniform expert ids, "
                         "weights summing to 1) instead of lmoe_forward")
    ap.add_argument("--layers", type=int, default=1,
                    help="a step runs this many layers back to back, each layer's output the next one's input "
                         "and each layer with its own device copy of the weights")
    ap.add_argument("--graph", action="store_true", help="capture one step in a CUDA graph and replay it")
    ap.add_argument("--nvfp4", action="store_true",
                    help="NVFP4 expert weights (E4M3 scale per 16 elements, fp32 global scale per expert matrix) "
                         "through lmoe_forward_nvfp4")
    ap.add_argument("--block", action="store_true",
                    help="time the sandwich block around the layer (lmoe_block_forward: pre-norm, layer, "
                         "post-norm and residual) instead of the layer alone")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --config (by default the decode_t1 run also times every other workload "
                         "config of the layer and reports them under per_config)")
    ap.add_argument("--stage", choices=["pool", "unpool"], default=None,
                    help="time one dense projection call alone (for profiling); prints a stage line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    name = args.config
    d = synth.CONFIGS[name]
    world, rank, local = dist_setup(args.gpus)

    if args.impl == "reference":
        run_reference(args, d, name, world, rank)
        return

    import torch
    import latent_moe_layer_fp32_gb300 as lm
    lm.build()
    lm.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.stage:
        run_stage(args, d, name, lm, dev)
        return

    if args.nvfp4 and (args.block or args.routed):
        raise SystemExit("--nvfp4 times lmoe_forward_nvfp4; it does not combine with --block or --routed")
    if args.nvfp4:
        global EXPERT_BYTES, GATEUP_BYTES
        EXPERT_BYTES = EXPERT_BYTES_NVFP4
        GATEUP_BYTES = 2 * EXPERT_BYTES // 3
    hw = synth.make_weights_nvfp4(d) if args.nvfp4 else synth.make_weights(d)
    x = synth.make_x(d)

    def to_dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    w = {k: to_dev(v) for k, v in hw.items()}
    n_layers = max(1, args.layers)
    # each layer gets its own copy of the weights, so no layer finds another's in L2
    w_layers = [w] + [{k: (None if v is None else v.clone()) for k, v in w.items()} for _ in range(n_layers - 1)]
    wts_layers = [lm.weights_of(wl) for wl in w_layers]
    wts = wts_layers[0]
    dims = lm.dims_of(d.T, d.H, d.L, d.I, d.E, d.k, d.eps)
    ws_bytes = lm.lmoe_block_workspace_bytes(dims) if args.block else lm.lmoe_workspace_bytes(dims)
    # the one-layer MXFP4 layer takes its end-to-end step through lmoe_forward_host (tokens and output
    # in pinned host memory); its workspace also holds the two staging buffers
    host_api = not (args.nvfp4 or args.block or args.routed or args.graph or args.layers > 1)
    if host_api:
        ws_bytes = max(ws_bytes, lm.lmoe_host_workspace_bytes(dims))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    x_dev = to_dev(x)
    out = torch.empty(d.T, d.H, dtype=torch.bfloat16, device=dev)
    block_norms = synth.make_block_norms(d) if args.block else None
    if args.block and args.routed:
        raise SystemExit("--block runs the block's own router; it does not combine with --routed")
    if args.nvfp4:
        nv_layers = [lm.nvfp4_of(wl) for wl in w_layers]

        def forward(xd, o, layer=0):
            lm.lmoe_forward_nvfp4(dims, wts_layers[layer], nv_layers[layer], xd, o, ws)
    elif args.block:
        nw_dev = {k: to_dev(v) for k, v in block_norms.items()}
        norms = lm.norms_of(nw_dev, d.eps)

        def forward(xd, o, layer=0):
            lm.lmoe_block_forward(dims, wts_layers[layer], norms, xd, o, ws)
    elif args.routed:
        rng = np.random.default_rng(1234)
        r_idx = rng.integers(0, d.E, size=(d.T, d.k), dtype=np.int32)
        r_w = rng.uniform(0.05, 1.0, size=(d.T, d.k)).astype(np.float32)
        r_w /= r_w.sum(1, keepdims=True)
        r_idx_dev, r_w_dev = to_dev(r_idx), to_dev(r_w.astype(np.float32))

        def forward(xd, o, layer=0):
            lm.lmoe_forward_routed(dims, wts_layers[layer], xd, r_idx_dev, r_w_dev, o, ws)
    else:
        def forward(xd, o, layer=0):
            lm.lmoe_forward(dims, wts_layers[layer], xd, o, ws)
    mid = torch.empty_like(out)

    def layers(xd, o):
        # layer i reads the previous layer's output; the last one writes o
        cur = xd
        for i in range(n_layers):
            dst = o if (n_layers - 1 - i) % 2 == 0 else mid
            forward(cur, dst, i)
            cur = dst
    graph = None
    if args.graph:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layers(x_dev, out)  # first-use setup happens outside the capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layers(x_dev, out)

    def step(xd, o):
        if graph is not None:
            graph.replay()  # captured on x_dev and out
        else:
            layers(xd, o)
    x_host = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = torch.empty(d.T, d.H, dtype=torch.bfloat16).pin_memory()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(x_dev, out)
        rc = lm.lmoe_status_check(ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc}: {lm.lmoe_error_string(rc)}")
        launches_per_step = lm.lmoe_last_launch_count()
        names = [lm.lmoe_last_launch_name(j) for j in range(launches_per_step)]
        lay = lm.lmoe_workspace_layout(dims)
        offs = ws[lay.expert_offsets:lay.expert_offsets + 4 * (d.E + 1)].view(torch.int32).cpu().numpy()
        touched = int(np.count_nonzero(np.diff(offs)))

        # ---- device-resident timed region ----
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        clk = Clocks(local).__enter__()
        time.sleep(0.5)  # nvidia-smi needs a moment before its first sample
        torch.cuda.synchronize()
        barrier(world)
        try:
            for i in range(args.steps):
                flush.zero_()
                e0[i].record()
                step(x_dev, out)
                e1[i].record()
            torch.cuda.synchronize()
        finally:
            clk.__exit__(None, None, None)
        barrier(world)
        step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
        # a step of n_layers layers moves each of its T tokens through n_layers layers:
        # the metric counts token-layers, so one- and many-layer steps compare directly
        value, total_s = job_throughput(world, d.T * n_layers * args.steps, sum(step_ms) / 1e3)
        clocks = clk.summary()

        # ---- end to end: host input upload and output download inside the timed region ----
        def e2e_step():
            if host_api:  # the public call for host buffers: copy kernels over the host link
                lm.lmoe_forward_host(dims, wts, x_host, out_host, ws)
            else:
                x_dev.copy_(x_host, non_blocking=True)
                step(x_dev, out)
                out_host.copy_(out, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        for i in range(args.steps):
            flush.zero_()
            e0[i].record()
            e2e_step()
            e1[i].record()
        torch.cuda.synchronize()
        barrier(world)
        e2e_value, e2e_s = job_throughput(world, d.T * n_layers * args.steps,
                                          sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / 1e3)

        # ---- dominant kernel, per-launch events ----
        per_launch = per_launch_ms(lm, lambda: forward(x_dev, out), launches_per_step,
                                   max(5, min(args.steps, 20)), flush)
        rc = lm.lmoe_status_check(ws)
        if rc != 0:
            raise RuntimeError(f"device status {rc}: {lm.lmoe_error_string(rc)}")

    pk = peaks()
    layer_bytes = touched * EXPERT_BYTES + PROJ_BYTES
    # every layer of a step streams about the same bytes (its own touched experts)
    layer_gbs = layer_bytes * n_layers * args.steps / total_s / 1e9

    # dominant kernel: the modelled launch with the largest mean device time
    kern_ms = {names[j]: statistics.mean(v) for j, v in enumerate(per_launch)}
    step_ms_mean = 1e3 * total_s / args.steps
    tc_peak = pk["bf16_tflops"] if step_ms_mean < 50 or not pk.get("bf16_tflops_sustained") \
        else pk["bf16_tflops_sustained"]
    roof = dominant_roofline(d, touched, kern_ms, pk, tc_peak, name + ("_nvfp4" if args.nvfp4 else ""))
    # the layer's own fraction: HBM bytes at decode, tensor flops at prefill
    layer_roof = layer_fraction(d, touched, step_ms_mean / n_layers, pk, tc_peak)
    if args.nvfp4 and layer_roof["bound"] == "hbm":
        layer_roof["achieved"] = layer_bytes / (step_ms_mean / n_layers / 1e3) / 1e9
        layer_roof["frac"] = layer_roof["achieved"] / layer_roof["peak"]
        layer_roof["algorithmic_bytes"] = layer_bytes

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based generator; random weights of the layer's shape)",
        "config": {"workload": workload_name(d, name) + (" (caller-supplied routing: seeded uniform ids, "
                                                          "lmoe_forward_routed)" if args.routed else "") +
                   (" inside the sandwich block (pre-norm, fp32 router input, post-norm, residual; "
                    "lmoe_block_forward)" if args.block else "") +
                   (" with NVFP4 experts (E4M3 scale per 16 elements, fp32 global scale per matrix; "
                    "lmoe_forward_nvfp4)" if args.nvfp4 else "") +
                   (f", {n_layers} layers per step" if n_layers > 1 else "") + (", CUDA graph" if args.graph else ""),
                   "T": d.T, "touched_experts": touched, "layers_per_step": n_layers,
                   "l2": "flushed between steps (512 MB device write outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "ms_per_layer": 1e3 * total_s / args.steps / n_layers,
        "layer_hbm_gbs": layer_gbs, "layer_roofline_frac": layer_roof["frac"], "layer_roofline": layer_roof,
        "layer_bytes_per_step": layer_bytes,
        "roofline": roof,
        "kernels_ms": kern_ms,
        "step_ms_percentiles": {"p10": float(np.percentile(step_ms, 10)), "median": float(np.median(step_ms)),
                                "p90": float(np.percentile(step_ms, 90))},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": d.T * d.H * 2,
                "d2h_bytes_per_step": d.T * d.H * 2,
                "call": "lmoe_forward_host" if host_api else "copies + device call"},
        "gpu_launches": launches_per_step * n_layers * args.steps,
        "clocks": clocks,
    }
    plain = not (args.nvfp4 or args.block or args.routed or args.graph or n_layers > 1)
    if world == 1 and name == "decode_t1" and plain and not args.no_per_config:
        with torch.cuda.stream(stream):
            line["per_config"] = run_per_config(args, lm, w, hw, dev, flush, pk, not args.no_cpu_baseline)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, reps, dt = cpu_oracle_rate(d, hw, x, block_norms=block_norms, nvfp4=args.nvfp4)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{reps} whole-{'block' if args.block else 'layer'} evaluations of the T={d.T} workload ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
