"""Benchmark of the GQA attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill: the LLaMA-3-8B-shaped layer (B=1, H_q=32, H_kv=8, N=2048,
    d=128, bf16, causal) through gqa_attn_fwd, and
  * decode: one token per sequence against a bf16 K/V cache (B=64, H_q=12,
    H_kv=2, d=128, max_len=2048, seqlens ~ U[1, 2048]) through
    gqa_attn_decode (split-KV kernel + log-sum-exp combine).
`value` is the prefill throughput in TFLOP/s (4*B*H_q*N_q*N_kv*d, halved for
causal) over the prefill kernel's device time; the decode throughput in GB/s
(valid cache rows once per K/V head, plus q, o and seqlens) is reported in
the `decode` object. Inputs are rotated over enough copies that every step
reads operands that are not in the 129 MB L2. After the step, a ragged batch
of eight prompts (LLaMA-3-8B heads, 256-4096 tokens) is timed through
gqa_attn_fwd_varlen in a region of its own and reported in `varlen`.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With --gpus N > 1 it runs under torch.distributed.run, one replica per GPU
(no collective on the data path: the units are independent); rank 0 prints
the single JSON line.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill TFLOP/s & decode KV-cache GB/s on 1 GB300, as fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(rel):
    """Hash of a kernel source with comments and blank lines removed, so an
    edit of the comments alone leaves recorded counters valid."""
    with open(os.path.join(ROOT, rel)) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def recorded_traffic(kernel_src, name):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha") != source_sha(kernel_src):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = list(csv.reader(io.StringIO(self.out or "")))
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        top = max(sm)
        loaded = [x for x in sm if x >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device, world):
    """Elementwise maximum of per-rank timings over all ranks: the slowest
    replica sets the job's time (all ranks must call it)."""
    import torch
    vals = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    return vals.tolist()


def job_throughput(world, calls, units_per_call, total_ms, scale):
    """Whole-job throughput with fixed work per replica (weak scaling): the
    units all `world` ranks processed over the slowest rank's time, divided
    by `scale` (1e12 for TFLOP/s, 1e9 for GB/s)."""
    return world * calls * units_per_call / (total_ms * 1e-3) / scale


# --------------------------------------------------------------------------- ours

def run_ours(args):
    import torch
    import torch.distributed as dist

    from gqa_flash_attention_02_gb300 import inputs, ops

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    ops.load()
    peaks, peak_src = load_peaks()

    ps = inputs.LLAMA3_8B_LAYER
    ds = inputs.decode_shapes()[-1]
    # Rotate inputs so the operands of a step are evicted from L2 by the time
    # they come round again.
    q0, k0, v0 = inputs.prefill_inputs_for(ps)
    sl0, dq0, kc0, vc0 = inputs.decode_inputs_for(ds)
    step_in_bytes = (q0.numel() + k0.numel() + v0.numel()) * 2 + (kc0.numel() + vc0.numel()) * 2
    copies = max(2, math.ceil(3 * L2_BYTES / step_in_bytes))
    pre = [(q0.to(dev), k0.to(dev), v0.to(dev)) for _ in range(copies)]
    dec = [(sl0.to(dev), dq0.to(dev), kc0.to(dev), vc0.to(dev)) for _ in range(copies)]
    o_pre = torch.empty_like(pre[0][0])
    o_dec = torch.empty_like(dec[0][1])
    torch.cuda.synchronize()

    pre_flops = ps.flops
    n_valid = int(sl0.sum())
    dec_bytes = (n_valid * ds.H_kv * ds.d * 2 * 2 + 2 * dq0.numel() * 2 + 4 * ds.B)

    stream = torch.cuda.current_stream()

    # The timed region replays CUDA graphs of back-to-back calls, so neither
    # Python nor per-launch overhead on the host or the GPU front end sits
    # between the kernels (the e2e figure below goes through the plain API
    # calls with host buffers).
    def call_pre(i, s):
        q, k, v = pre[i % copies]
        ops.gqa_attn_fwd(q, k, v, o_pre, causal=True, scale=ps.scale, stream=s)

    def call_dec(i, s):
        sl, dq, kc, vc = dec[i % copies]
        ops.gqa_attn_decode(dq, kc, vc, sl, o_dec, scale=ds.scale, stream=s)

    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        for i in range(copies):   # workspace for the capture stream, outside any capture
            call_pre(i, cap)
            call_dec(i, cap)
    torch.cuda.synchronize()

    def capture(fn, first, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(first, first + count):
                fn(i, cap)
        return g

    # A chain graph holds `chain` back-to-back calls of one kernel over the
    # rotating copies (a multiple of `copies`, so replays continue the
    # rotation); K = reps * chain + rest calls are timed per kernel, the rest
    # as one more graph of `rest` back-to-back calls.
    K = args.steps
    chain = copies * max(1, 24 // copies)
    reps, rest = divmod(K, chain)
    chain_pre, chain_dec = capture(call_pre, 0, chain), capture(call_dec, 0, chain)
    rest_pre = capture(call_pre, 0, rest) if rest else None
    rest_dec = capture(call_dec, 0, rest) if rest else None
    torch.cuda.synchronize()

    def run_kernel(chain_g, rest_g):
        for _ in range(reps):
            chain_g.replay()
        if rest_g is not None:
            rest_g.replay()

    # The ragged batch (one call = the plan kernel + the prefill kernel) is
    # timed in a region of its own after the step, over its own rotating
    # copies.
    vs = inputs.varlen_batch_shape()
    vq0, vk0, vv0, vcq0, vck0 = inputs.varlen_inputs_for(vs)
    var_bytes = (vq0.numel() + vk0.numel() + vv0.numel()) * 2
    var_copies = max(2, math.ceil(3 * L2_BYTES / var_bytes))
    var = [(vq0.to(dev), vk0.to(dev), vv0.to(dev), vcq0.to(dev), vck0.to(dev))
           for _ in range(var_copies)]
    o_var = torch.empty_like(var[0][0])

    def call_var(i, s):
        q, k, v, cq, ck = var[i % var_copies]
        ops.gqa_attn_fwd_varlen(q, k, v, cq, ck, o_var, causal=True, scale=vs.scale, stream=s)

    with torch.cuda.stream(cap):
        for i in range(var_copies):
            call_var(i, cap)
    torch.cuda.synchronize()
    var_chain = var_copies * max(1, 8 // var_copies)
    chain_var = capture(call_var, 0, var_chain)
    var_reps = max(1, math.ceil(min(max(K, 4), 40) / var_chain))
    K_var = var_reps * var_chain
    chain_var.replay()

    for _ in range(max(1, math.ceil(args.warmup / chain))):  # at least W calls of each
        chain_pre.replay()
        chain_dec.replay()
    torch.cuda.synchronize()

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                      else local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ev[0].record(stream)
        run_kernel(chain_pre, rest_pre)     # K prefill launches
        ev[1].record(stream)
        run_kernel(chain_dec, rest_dec)     # K decode launches
        ev[2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        ev_var = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev_var[0].record(stream)
        for _ in range(var_reps):
            chain_var.replay()          # K_var ragged-batch calls
        ev_var[1].record(stream)
        torch.cuda.synchronize()
    tot_var = ev_var[0].elapsed_time(ev_var[1])
    tot_pre = ev[0].elapsed_time(ev[1])   # ms
    tot_dec = ev[1].elapsed_time(ev[2])
    gpu_err = ops.gqa_attn_get_device_error(stream=cap)  # the graphs' error word
    if gpu_err != 0:
        raise RuntimeError(f"device error during the bench: {ops.status_string(gpu_err)}")

    # ---- e2e through the public API with host buffers (pinned), copies timed
    hq, hk, hv = (t.pin_memory() for t in (q0, k0, v0))
    ho = torch.empty(o_pre.shape, dtype=o_pre.dtype).pin_memory()
    hsl, hdq, hkc, hvc = (t.pin_memory() for t in (sl0, dq0, kc0, vc0))
    hdo = torch.empty(o_dec.shape, dtype=o_dec.dtype).pin_memory()
    dq_, dk_, dv_ = (torch.empty_like(t, device=dev) for t in (q0, k0, v0))
    dsl_, ddq_, dkc_, dvc_ = (torch.empty_like(t, device=dev) for t in (sl0, dq0, kc0, vc0))
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step(evp):
        evp[0].record(stream)
        dq_.copy_(hq, non_blocking=True); dk_.copy_(hk, non_blocking=True)
        dv_.copy_(hv, non_blocking=True)
        ops.gqa_attn_fwd(dq_, dk_, dv_, o_pre, causal=True, scale=ps.scale, stream=stream)
        ho.copy_(o_pre, non_blocking=True)
        evp[1].record(stream)
        dsl_.copy_(hsl, non_blocking=True); ddq_.copy_(hdq, non_blocking=True)
        dkc_.copy_(hkc, non_blocking=True); dvc_.copy_(hvc, non_blocking=True)
        ops.gqa_attn_decode(ddq_, dkc_, dvc_, dsl_, o_dec, scale=ds.scale, stream=stream)
        hdo.copy_(o_dec, non_blocking=True)
        evp[2].record(stream)

    for _ in range(2):
        e2e_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()
    eev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        e2e_step(eev[i])
    torch.cuda.synchronize()
    e2e_pre = sum(e[0].elapsed_time(e[1]) for e in eev) / e2e_steps
    e2e_dec = sum(e[1].elapsed_time(e[2]) for e in eev) / e2e_steps

    # ---- max over ranks
    tot_pre, tot_dec, wall, e2e_pre, e2e_dec, tot_var = max_over_ranks(
        [tot_pre, tot_dec, wall, e2e_pre, e2e_dec, tot_var], dev, world)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    K = args.steps
    pre_ms = tot_pre / K
    dec_ms = tot_dec / K
    value = job_throughput(world, K, pre_flops, tot_pre, 1e12)
    dec_gbs = job_throughput(world, K, dec_bytes, tot_dec, 1e9)
    pre_ach = pre_flops / (pre_ms * 1e-3) / 1e12
    dec_ach = dec_bytes / (dec_ms * 1e-3) / 1e9
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    h2d_pre = (q0.numel() + k0.numel() + v0.numel()) * 2
    d2h_pre = o_pre.numel() * 2
    h2d_dec = sl0.numel() * 4 + (dq0.numel() + kc0.numel() + vc0.numel()) * 2
    d2h_dec = o_dec.numel() * 2
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(pre_ms + dec_ms, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded iid N(0,1) q/k/v, bf16; decode seqlens ~ U[1,2048])",
        "config": {
            "workload": "llama3_8b_prefill_layer + decode_b64",
            "prefill": {"B": ps.B, "H_q": ps.H_q, "H_kv": ps.H_kv, "N_q": ps.N_q,
                        "N_kv": ps.N_kv, "d": ps.d, "causal": ps.causal},
            "decode": {"B": ds.B, "H_q": ds.H_q, "H_kv": ds.H_kv, "max_len": ds.max_len,
                       "d": ds.d, "sum_seqlens": n_valid},
            "l2": f"inputs rotated over {copies} copies "
                  f"({copies * step_in_bytes / 2**20:.0f} MiB > 129 MiB L2)",
            "launch": "CUDA graphs: chains of back-to-back calls of each kernel over the rotating copies",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "prefill_tc_kernel<128, 0> (no lse output)",
            "achieved": round(pre_ach, 3),
            "peak": tc_peak,
            "unit": "TFLOP/s",
            "frac": round(pre_ach / tc_peak, 4),
            "peak_source": f"{peak_src} bf16_tflops (burst)",
            "traffic": recorded_traffic("gqa_flash_attention_02_gb300/csrc/prefill_tc.cu",
                                        "prefill_tc_kernel<128, 0>"),
        },
        "decode": {
            "value": round(dec_gbs, 2),
            "unit": "GB/s",
            "ms": round(dec_ms, 6),
            "roofline": {
                "bound": "hbm",
                "kernel": "decode_kernel<128,5> (persistent split-KV + in-kernel merge)",
                "achieved": round(dec_ach, 2),
                "peak": hbm_peak,
                "unit": "GB/s",
                "frac": round(dec_ach / hbm_peak, 4),
                "peak_source": f"{peak_src} hbm_gbs",
                "traffic": recorded_traffic("gqa_flash_attention_02_gb300/csrc/decode_splitkv.cu",
                                            "decode_kernel<128,5>"),
            },
            "e2e": {"value": round(dec_bytes / (e2e_dec * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d_dec, "d2h_bytes_per_step": d2h_dec},
        },
        "varlen": {
            "value": round(job_throughput(world, K_var, vs.flops, tot_var, 1e12), 3),
            "unit": "TFLOP/s",
            "ms": round(tot_var / K_var, 6),
            "calls": K_var,
            "gpu_launches": 2 * K_var,  # the plan kernel + the prefill kernel per call
            "config": {"workload": vs.name, "lens": list(vs.lens_q), "H_q": vs.H_q,
                       "H_kv": vs.H_kv, "d": vs.d, "causal": vs.causal,
                       "layout": "token-major [total][H][d], cu_seqlens on the device",
                       "l2": f"inputs rotated over {var_copies} copies "
                             f"({var_copies * var_bytes / 2**20:.0f} MiB)"},
            "roofline": {
                "bound": "tensor",
                "kernel": "varlen_plan_kernel + prefill_varlen_kernel<128, 0> (per call)",
                "achieved": round(vs.flops / (tot_var / K_var * 1e-3) / 1e12, 3),
                "peak": tc_peak,
                "unit": "TFLOP/s",
                "frac": round(vs.flops / (tot_var / K_var * 1e-3) / 1e12 / tc_peak, 4),
                "peak_source": f"{peak_src} bf16_tflops (burst)",
                "traffic": recorded_traffic("gqa_flash_attention_02_gb300/csrc/prefill_tc.cu",
                                            "prefill_varlen_kernel<128, 0>"),
            },
        },
        "e2e": {"value": round(pre_flops / (e2e_pre * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_pre, "d2h_bytes_per_step": d2h_pre},
        "gpu_launches": 2 * K,  # one prefill + one decode launch per step
        "wall_ms_per_step": round(wall * 1e3 / K, 6),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(ps)
    if world > 1:
        dist.destroy_process_group()
    return line


# --------------------------------------------------------------------------- oracle

def oracle_prefill_sample(ps, heads, threads):
    """Times the float64 CPU oracle on `heads` (b, h_q) heads of the workload.
    Returns (seconds, flops of that sample)."""
    import oracle
    from gqa_flash_attention_02_gb300 import inputs

    q, k, v = inputs.prefill_inputs_for(ps)
    oracle.build()
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, ps.causal, ps.scale, heads=(0, heads), n_threads=threads)
    dt = time.perf_counter() - t0
    return dt, ps.flops * heads / (ps.B * ps.H_q)


def cpu_baseline(ps, min_seconds=10.0, max_passes=64):
    """The oracle as it stands, timed on the host cores: whole passes over
    the prefill layer (every head, every row) until at least `min_seconds`
    of work, so the rate is not a sub-second sample."""
    import oracle
    from gqa_flash_attention_02_gb300 import inputs

    cores = os.cpu_count() or 1
    q, k, v = inputs.prefill_inputs_for(ps)
    oracle.build()
    heads = ps.B * ps.H_q
    passes, dt = 0, 0.0
    while passes == 0 or (dt < min_seconds and passes < max_passes):
        t0 = time.perf_counter()
        oracle.prefill(q, k, v, ps.causal, ps.scale, heads=(0, heads), n_threads=cores)
        dt += time.perf_counter() - t0
        passes += 1
    return {"value": round(passes * ps.flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} passes over the whole prefill layer ({heads} heads x "
                      f"{ps.N_q} rows), float64, OpenMP over heads, {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from gqa_flash_attention_02_gb300 import inputs

    ps = inputs.LLAMA3_8B_LAYER
    cores = os.cpu_count() or 1
    heads = max(1, min(ps.B * ps.H_q, cores))
    for _ in range(args.warmup):
        oracle_prefill_sample(ps, 1, 1)
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, flops = oracle_prefill_sample(ps, heads, cores)
        times.append(dt)
    tot = sum(times)
    value = args.steps * flops / tot / 1e12
    sample = (f"{heads} of {ps.B * ps.H_q} heads of the prefill layer per step, float64 "
              f"oracle, OpenMP over heads")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1), bf16 values widened to float64)",
        "config": {"workload": "llama3_8b_prefill_layer (head sample)",
                   "prefill": {"B": ps.B, "H_q": ps.H_q, "H_kv": ps.H_kv, "N_q": ps.N_q,
                               "N_kv": ps.N_kv, "d": ps.d, "causal": ps.causal}},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing leg (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
