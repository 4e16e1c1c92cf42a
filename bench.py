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


def _code_text(path):
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    return [ln for ln in lines if ln]


E2E_MODE = ("pipelined over steps: step i's H2D copies (one stream per input tensor), "
            "step i-1's kernel and step i-2's D2H copy overlap, two device buffers; "
            "serial_value: copies and kernel back to back on one stream")


def source_sha(rel):
    """Hash of a kernel source and of the local headers it includes
    (recursively, ``#include "..."`` next to the file), with comments and
    blank lines removed, so an edit of the comments alone leaves recorded
    counters valid while any code change, in the file or a header, voids
    them."""
    seen, parts, todo = set(), [], [os.path.join(ROOT, rel)]
    while todo:
        path = os.path.normpath(todo.pop(0))
        if path in seen or not os.path.exists(path):
            continue
        seen.add(path)
        lines = _code_text(path)
        parts.append("\n".join(lines))
        for ln in lines:
            m = re.match(r'\s*#\s*include\s+"([^"]+)"', ln)
            if m:
                todo.append(os.path.join(os.path.dirname(path), m.group(1)))
    return hashlib.sha256("\n\0".join(parts).encode()).hexdigest()[:16]


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

def decode_bytes(seqlens, shape):
    """Algorithmic bytes of one decode call: every valid cache row once per
    K/V head (K and V), plus q, o and seqlens."""
    n_valid = int(seqlens.sum())
    return (n_valid * shape.H_kv * shape.d * 2 * 2 + 2 * shape.B * shape.H_q * shape.d * 2
            + 4 * shape.B)


class GraphChain:
    """`calls` back-to-back calls fn(i, stream) (i = 0, 1, ...) captured in one
    CUDA graph on `stream`, so nothing on the host sits between the kernels;
    the inputs are rotated by the callers over enough copies that a call's
    operands are not in the L2 when they come round again."""

    def __init__(self, torch, fn, calls, stream):
        self.calls = calls
        self.graph = None
        if calls > 0:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=stream):
                for i in range(calls):
                    fn(i, stream)

    def replay(self):
        if self.graph is not None:
            self.graph.replay()


def copies_for(bytes_per_call, cap_bytes=1 << 30):
    """Copies of a call's inputs to rotate over: three L2 sizes' worth, at
    least two, and no more than cap_bytes in all (then at least two)."""
    n = max(2, math.ceil(3 * L2_BYTES / max(1, bytes_per_call)))
    return max(2, min(n, cap_bytes // max(1, bytes_per_call)))


def time_calls(torch, fn, copies, stream, reps=21, min_chain_us=300.0, est_us=None):
    """Median device time of one call, in ms, over `reps` repetitions of a
    graph of back-to-back calls over the rotating copies (CUDA events on the
    launching stream around each replay: a graph captured on `stream` is
    replayed on the current stream). Returns (ms_per_call, calls_per_rep)."""
    launch = torch.cuda.current_stream()
    if est_us is None:
        g = GraphChain(torch, fn, copies, stream)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(launch)
        g.replay()
        e1.record(launch)
        torch.cuda.synchronize()
        est_us = max(1e-3, e0.elapsed_time(e1) * 1e3 / copies)
    chain = copies * max(1, math.ceil(min_chain_us / est_us / copies))
    g = GraphChain(torch, fn, chain, stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record(launch)
        g.replay()
        b.record(launch)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev) / chain, chain


def roofline_obj(bound, achieved, peak, unit, peak_src, kernel, traffic=None):
    return {"bound": bound, "kernel": kernel, "achieved": round(achieved, 3), "peak": peak,
            "unit": unit, "frac": round(achieved / peak, 4), "peak_source": peak_src,
            "traffic": traffic}


def prefill_cluster_size(torch, ops, shape):
    """CTAs per cluster the dense prefill uses for `shape` (for naming the
    kernel instantiation): g / 2 for two-tile units of a 4- or 8-head group
    from four units per SM up, else 1."""
    units = ops.gqa_attn_prefill_plan(shape.B, shape.H_q, shape.H_kv, shape.N_q, shape.N_kv,
                                      shape.causal)
    g = shape.H_q // shape.H_kv
    pairs = any(u[3][2] > 0 for u in units)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if pairs and g in (4, 8) and shape.d <= 128 and len(units) >= 4 * sms:
        return g // 2
    return 1


def config_blocks(torch, ops, inputs, dev, stream, tc_peak, hbm_peak, peak_src, only=None):
    """Per-workload throughput beside the headline step: the MHA/GQA/MQA sweep
    (six variants), the long-sequence case and decode at B = 1, 8, 64. Each
    is the median over 21 repetitions of a graph of back-to-back calls over
    rotating input copies. ``only``: the groups to run (sweep, long, backward,
    decode, decode_fp8, decode_int8), all when None."""
    out = {}
    want = lambda group: only is None or group in only

    def prefill_block(shape):
        cluster = prefill_cluster_size(torch, ops, shape)
        q, k, v = inputs.prefill_inputs_for(shape)
        nbytes = (q.numel() + k.numel() + v.numel()) * 2
        copies = copies_for(nbytes)
        bufs = [(q.to(dev), k.to(dev), v.to(dev)) for _ in range(copies)]
        o = torch.empty_like(bufs[0][0])

        def call(i, s):
            a, b, c = bufs[i % copies]
            ops.gqa_attn_fwd(a, b, c, o, causal=shape.causal, scale=shape.scale, stream=s)

        for i in range(copies):
            call(i, stream)
        ms, chain = time_calls(torch, call, copies, stream)
        assert ops.gqa_attn_get_device_error(stream=stream) == 0
        del bufs, o
        torch.cuda.empty_cache()
        ach = shape.flops / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 6), "value": round(ach, 3), "unit": "TFLOP/s",
                "shape": {"B": shape.B, "H_q": shape.H_q, "H_kv": shape.H_kv, "N": shape.N_q,
                          "d": shape.d, "causal": shape.causal},
                "calls_per_rep": chain, "reps": 21, "l2": f"{copies} rotating copies",
                "roofline": roofline_obj("tensor", ach, tc_peak, "TFLOP/s",
                                         f"{peak_src} bf16_tflops (burst)",
                                         f"prefill_tc_kernel<{shape.d}, 0, {cluster}>",
                                         recorded_traffic("gqa_flash_attention_02_gb300/csrc/prefill_tc.cu",
                                                          f"prefill_tc_kernel<{shape.d}, 0, {cluster}> {shape.name}"))}

    for shape in inputs.sweep_shapes() if want("sweep") else []:
        out[shape.name] = prefill_block(shape)
    if want("long"):
        out[inputs.LONG_SEQ.name] = prefill_block(inputs.LONG_SEQ)
    if want("backward"):
        backward_block(torch, ops, inputs, dev, stream, tc_peak, peak_src, out)
    if want("decode"):
        decode_blocks(torch, ops, inputs, dev, stream, hbm_peak, peak_src, out)
    if want("decode_fp8"):
        decode_byte_block(torch, ops, inputs, dev, stream, hbm_peak, peak_src, out, "fp8")
    if want("decode_int8"):
        decode_byte_block(torch, ops, inputs, dev, stream, hbm_peak, peak_src, out, "int8")
    return out


def backward_block(torch, ops, inputs, dev, stream, tc_peak, peak_src, out):
    # attention backward on the prefill layer: algorithmic FLOPs are the five
    # products of the standard backward (S, dP, dV, dK, dQ: 2.5 x the
    # forward's), halved for causal; the kernel's recomputed S and dP in the
    # dQ units are not counted
    shape = inputs.LLAMA3_8B_LAYER
    q, k, v = inputs.prefill_inputs_for(shape)
    dout = inputs.prefill_inputs(shape.B, shape.H_q, shape.H_kv, shape.N_q, shape.N_kv, shape.d,
                                 torch.bfloat16, shape.seed + 1)[0]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=shape.causal, scale=shape.scale, stream=stream)
    torch.cuda.synchronize()
    nbytes = (q.numel() * 3 + k.numel() * 2) * 2 + lse.numel() * 4
    copies = copies_for(nbytes)
    bufs = [(qd.clone(), kd.clone(), vd.clone(), o.clone(), dout.to(dev), lse.clone())
            for _ in range(copies)]
    grads = (torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd))

    def call_bwd(i, s):
        a, b_, c, d_, e, f = bufs[i % copies]
        ops.gqa_attn_bwd(a, b_, c, d_, e, f, *grads, causal=shape.causal, scale=shape.scale,
                         stream=s)

    for i in range(copies):
        call_bwd(i, stream)
    ms, chain = time_calls(torch, call_bwd, copies, stream)
    assert ops.gqa_attn_get_device_error(stream=stream) == 0
    ach = 2.5 * shape.flops / (ms * 1e-3) / 1e12
    out["backward_" + shape.name] = {
        "ms": round(ms, 6), "value": round(ach, 3), "unit": "TFLOP/s",
        "shape": {"B": shape.B, "H_q": shape.H_q, "H_kv": shape.H_kv, "N": shape.N_q,
                  "d": shape.d, "causal": shape.causal},
        "flops": "2.5 x the forward's algorithmic FLOPs", "launches_per_call": 2,
        "calls_per_rep": chain, "reps": 21, "l2": f"{copies} rotating copies",
        "roofline": dict(roofline_obj("tensor", ach, tc_peak, "TFLOP/s",
                                      f"{peak_src} bf16_tflops (burst)",
                                      f"bwd_prep_kernel<{shape.d}, {shape.d}> + bwd_kernel<{shape.d}, {shape.d}>",
                                      recorded_traffic("gqa_flash_attention_02_gb300/csrc/attn_bwd.cu",
                                                       f"bwd_kernel<{shape.d}, {shape.d}>")),
                         traffic_kernel=f"bwd_kernel<{shape.d}, {shape.d}> (the main launch)")}
    del bufs, grads, qd, kd, vd, o, lse
    torch.cuda.empty_cache()


def decode_blocks(torch, ops, inputs, dev, stream, hbm_peak, peak_src, out):
    for shape in inputs.decode_shapes():
        sl, q, kc, vc = inputs.decode_inputs_for(shape)
        in_bytes = (q.numel() + kc.numel() + vc.numel()) * 2
        copies = copies_for(in_bytes)
        bufs = [(sl.to(dev), q.to(dev), kc.to(dev), vc.to(dev)) for _ in range(copies)]
        o = torch.empty_like(bufs[0][1])

        def call(i, s):
            a, b, c, d = bufs[i % copies]
            ops.gqa_attn_decode(b, c, d, a, o, scale=shape.scale, stream=s)

        for i in range(copies):
            call(i, stream)
        ms, chain = time_calls(torch, call, copies, stream)
        assert ops.gqa_attn_get_device_error(stream=stream) == 0
        nbytes = decode_bytes(sl, shape)
        ach = nbytes / (ms * 1e-3) / 1e9
        out[shape.name] = {
            "ms": round(ms, 6), "value": round(ach, 2), "unit": "GB/s",
            "shape": {"B": shape.B, "H_q": shape.H_q, "H_kv": shape.H_kv,
                      "max_len": shape.max_len, "d": shape.d, "sum_seqlens": int(sl.sum())},
            "bytes_per_call": nbytes, "calls_per_rep": chain, "reps": 21,
            "l2": f"{copies} rotating copies",
            "roofline": roofline_obj("hbm", ach, hbm_peak, "GB/s", f"{peak_src} hbm_gbs",
                                     "decode_kernel<128,5,0,128,0>",
                                     # the capture is of the B=64 workload; the
                                     # smaller batches have none of their own
                                     recorded_traffic("gqa_flash_attention_02_gb300/csrc/decode_splitkv.cu",
                                                      "decode_kernel<128,5,0,128,0>")
                                     if shape.name == "decode_b64" else None)}
        del bufs, o
        torch.cuda.empty_cache()


def decode_byte_block(torch, ops, inputs, dev, stream, hbm_peak, peak_src, out, kind):
    # decode against a one-byte cache (kind "fp8": e4m3 codes, "int8": int8
    # codes; per-K/V-head scales): bytes actually read (one byte per cached
    # value, K and V once per K/V head, plus q, o and seqlens)
    shape = inputs.decode_shapes()[-1]
    make = inputs.decode_inputs_fp8 if kind == "fp8" else inputs.decode_inputs_int8
    entry = ops.gqa_attn_decode_fp8 if kind == "fp8" else ops.gqa_attn_decode_int8
    sl, q, k8, v8, ks, vs = make(shape.B, shape.H_q, shape.H_kv, shape.max_len, shape.d,
                                 seed=shape.seed)
    in_bytes = q.numel() * 2 + k8.numel() + v8.numel()
    copies = copies_for(in_bytes)
    bufs = [(sl.to(dev), q.to(dev), k8.to(dev), v8.to(dev)) for _ in range(copies)]
    ksd, vsd = ks.to(dev), vs.to(dev)
    o = torch.empty_like(bufs[0][1])

    def call8(i, s):
        a, b_, c, d_ = bufs[i % copies]
        entry(b_, c, d_, ksd, vsd, a, o, scale=shape.scale, stream=s)

    for i in range(copies):
        call8(i, stream)
    ms, chain = time_calls(torch, call8, copies, stream)
    assert ops.gqa_attn_get_device_error(stream=stream) == 0
    nbytes = int(sl.sum()) * shape.H_kv * shape.d * 2 + 2 * shape.B * shape.H_q * shape.d * 2 + 4 * shape.B
    ach = nbytes / (ms * 1e-3) / 1e9
    kernel = f"decode_kernel<128,5,1,128,{1 if kind == 'int8' else 0}>"
    out[f"decode_{kind}_b64"] = {
        "ms": round(ms, 6), "value": round(ach, 2), "unit": "GB/s",
        "shape": {"B": shape.B, "H_q": shape.H_q, "H_kv": shape.H_kv, "max_len": shape.max_len,
                  "d": shape.d, "sum_seqlens": int(sl.sum()),
                  "cache": ("e4m3" if kind == "fp8" else "int8") + ", per-head scales"},
        "bytes_per_call": nbytes, "calls_per_rep": chain, "reps": 21,
        "l2": f"{copies} rotating copies",
        "roofline": roofline_obj("hbm", ach, hbm_peak, "GB/s", f"{peak_src} hbm_gbs",
                                 f"{kernel} ({kind} cache)",
                                 recorded_traffic("gqa_flash_attention_02_gb300/csrc/decode_splitkv.cu",
                                                  kernel))}
    del bufs, o
    torch.cuda.empty_cache()


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
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))

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
    dec_bytes = decode_bytes(sl0, ds)

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

    # A chain graph holds `chain` back-to-back calls of one kernel over the
    # rotating copies (a multiple of `copies`, so replays continue the
    # rotation); one repetition of the step is K prefill calls then K decode
    # calls: reps * chain + rest calls per kernel, the rest as one more graph.
    K = args.steps
    chain = copies * max(1, 24 // copies)
    n_chain, rest = divmod(K, chain)
    chain_pre, chain_dec = GraphChain(torch, call_pre, chain, cap), GraphChain(torch, call_dec, chain, cap)
    rest_pre, rest_dec = GraphChain(torch, call_pre, rest, cap), GraphChain(torch, call_dec, rest, cap)
    torch.cuda.synchronize()

    def run_kernel(chain_g, rest_g):
        for _ in range(n_chain):
            chain_g.replay()
        rest_g.replay()

    for _ in range(max(1, math.ceil(args.warmup / chain))):  # at least W calls of each
        chain_pre.replay()
        chain_dec.replay()
    torch.cuda.synchronize()
    # Repetitions of the K-step region: at least 21, and enough to last about
    # a second, so the median is robust and the clock sampler sees the load.
    t0 = time.perf_counter()
    run_kernel(chain_pre, rest_pre)
    run_kernel(chain_dec, rest_dec)
    torch.cuda.synchronize()
    rep_s = max(1e-6, time.perf_counter() - t0)
    reps = int(min(max(21, math.ceil(1.0 / rep_s)), 5001))
    if args.reps:
        reps = args.reps  # profiling runs: a fixed, small count
    reps += 1 - reps % 2  # odd: the median is one repetition's time

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

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                      else local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for e in ev:
            e[0].record(stream)
            run_kernel(chain_pre, rest_pre)     # K prefill launches
            e[1].record(stream)
            run_kernel(chain_dec, rest_dec)     # K decode launches
            e[2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        var_ms, var_chain = time_calls(torch, call_var, var_copies, cap, min_chain_us=2000.0)
        only = set(args.configs.split(",")) if args.configs else None
        blocks = None if args.no_configs else config_blocks(
            torch, ops, inputs, dev, cap, tc_peak, hbm_peak, peak_src, only)
    tot_pre = statistics.median(e[0].elapsed_time(e[1]) for e in ev)   # ms for K calls
    tot_dec = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
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
    e2e_pre = statistics.median(e[0].elapsed_time(e[1]) for e in eev)
    e2e_dec = statistics.median(e[1].elapsed_time(e[2]) for e in eev)

    # The same calls pipelined as a serving loop would run them: step i's
    # inputs go up (one stream per input tensor, so several copy engines
    # work at once) while step i-1 computes and step i-2's result comes down
    # on another stream (two device buffers); every step still copies its
    # inputs from pinned host memory and reads its result back.
    s_ins = [torch.cuda.Stream() for _ in range(4)]
    s_out = torch.cuda.Stream()

    def pipelined(host_in, host_out_like, run, n):
        nbuf = 2
        dins = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(nbuf)]
        douts = [torch.empty(host_out_like.shape, dtype=host_out_like.dtype, device=dev)
                 for _ in range(nbuf)]
        houts = [torch.empty(host_out_like.shape, dtype=host_out_like.dtype).pin_memory()
                 for _ in range(nbuf)]
        ev = lambda: torch.cuda.Event(enable_timing=False)
        in_done = [[ev() for _ in host_in] for _ in range(n)]
        comp_done = [ev() for _ in range(n)]
        out_done = [ev() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for si in s_ins:
            si.wait_event(t0)
        s_out.wait_event(t0)
        for i in range(n):
            b = i % nbuf
            for j, (d, h) in enumerate(zip(dins[b], host_in)):
                si = s_ins[j % len(s_ins)]
                with torch.cuda.stream(si):
                    if i >= nbuf:
                        si.wait_event(comp_done[i - nbuf])   # buffer b's last reader
                    d.copy_(h, non_blocking=True)
                    in_done[i][j].record(si)
            for e in in_done[i]:
                stream.wait_event(e)
            if i >= nbuf:
                stream.wait_event(out_done[i - nbuf])      # buffer b's result is down
            run(dins[b], douts[b])
            comp_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                houts[b].copy_(douts[b], non_blocking=True)
                out_done[i].record(s_out)
        stream.wait_event(out_done[n - 1])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    def run_pre(din, dout):
        ops.gqa_attn_fwd(din[0], din[1], din[2], dout, causal=True, scale=ps.scale, stream=stream)

    def run_dec(din, dout):
        ops.gqa_attn_decode(din[1], din[2], din[3], din[0], dout, scale=ds.scale, stream=stream)

    pipe_steps = max(8, min(args.steps, 64))
    pipelined((hq, hk, hv), o_pre, run_pre, 4)  # warm-up
    pipe_pre = min(pipelined((hq, hk, hv), o_pre, run_pre, pipe_steps) for _ in range(3))
    pipelined((hsl, hdq, hkc, hvc), o_dec, run_dec, 4)
    pipe_dec = min(pipelined((hsl, hdq, hkc, hvc), o_dec, run_dec, pipe_steps) for _ in range(3))

    # ---- max over ranks
    tot_pre, tot_dec, wall, e2e_pre, e2e_dec, pipe_pre, pipe_dec, var_ms = max_over_ranks(
        [tot_pre, tot_dec, wall, e2e_pre, e2e_dec, pipe_pre, pipe_dec, var_ms], dev, world)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    pre_ms = tot_pre / K
    dec_ms = tot_dec / K
    value = job_throughput(world, K, pre_flops, tot_pre, 1e12)
    dec_gbs = job_throughput(world, K, dec_bytes, tot_dec, 1e9)
    pre_ach = pre_flops / (pre_ms * 1e-3) / 1e12
    dec_ach = dec_bytes / (dec_ms * 1e-3) / 1e9
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
            "timing": f"median over {reps} repetitions of the K-step region "
                      "(CUDA events around the K prefill and the K decode calls of each)",
            "parallelism": f"replicas x{world}",
        },
        "repetitions": reps,
        "roofline": roofline_obj(
            "tensor", pre_ach, tc_peak, "TFLOP/s", f"{peak_src} bf16_tflops (burst)",
            "prefill_tc_kernel<128, 0, 1> (no lse output, no clusters)",
            recorded_traffic("gqa_flash_attention_02_gb300/csrc/prefill_tc.cu",
                             "prefill_tc_kernel<128, 0, 1>")),
        "decode": {
            "value": round(dec_gbs, 2),
            "unit": "GB/s",
            "ms": round(dec_ms, 6),
            "roofline": roofline_obj(
                "hbm", dec_ach, hbm_peak, "GB/s", f"{peak_src} hbm_gbs",
                "decode_kernel<128,5,0,128,0> (persistent split-KV + in-kernel merge)",
                recorded_traffic("gqa_flash_attention_02_gb300/csrc/decode_splitkv.cu",
                                 "decode_kernel<128,5,0,128,0>")),
            "e2e": {"value": round(dec_bytes / (pipe_dec * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d_dec, "d2h_bytes_per_step": d2h_dec,
                    "mode": E2E_MODE,
                    "serial_value": round(dec_bytes / (e2e_dec * 1e-3) / 1e9, 2)},
        },
        "varlen": {
            "value": round(job_throughput(world, 1, vs.flops, var_ms, 1e12), 3),
            "unit": "TFLOP/s",
            "ms": round(var_ms, 6),
            "calls_per_rep": var_chain,
            "reps": 21,
            "gpu_launches_per_call": 2,  # the plan kernel + the prefill kernel
            "config": {"workload": vs.name, "lens": list(vs.lens_q), "H_q": vs.H_q,
                       "H_kv": vs.H_kv, "d": vs.d, "causal": vs.causal,
                       "layout": "token-major [total][H][d], cu_seqlens on the device",
                       "l2": f"inputs rotated over {var_copies} copies "
                             f"({var_copies * var_bytes / 2**20:.0f} MiB)"},
            "roofline": roofline_obj(
                "tensor", vs.flops / (var_ms * 1e-3) / 1e12, tc_peak, "TFLOP/s",
                f"{peak_src} bf16_tflops (burst)",
                "varlen_plan_kernel + prefill_varlen_kernel<128, 0> (per call)",
                recorded_traffic("gqa_flash_attention_02_gb300/csrc/prefill_tc.cu",
                                 "prefill_varlen_kernel<128, 0>")),
        },
        "configs": blocks,
        "e2e": {"value": round(pre_flops / (pipe_pre * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_pre, "d2h_bytes_per_step": d2h_pre,
                "mode": E2E_MODE,
                "serial_value": round(pre_flops / (e2e_pre * 1e-3) / 1e12, 3)},
        "gpu_launches": 2 * K * reps,  # one prefill + one decode launch per step, per repetition
        "wall_ms_per_step": round(wall * 1e3 / (K * reps), 6),
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


def cpu_baseline(ps, min_seconds=10.0, max_passes=64, single_seconds=5.0):
    """The oracle as it stands, timed on the host cores: whole passes over
    the prefill layer (every head, every row) with OpenMP over heads until at
    least `min_seconds` of work; beside it, one thread on the first two heads
    until at least `single_seconds` (the rate per FLOP of the whole layer,
    since every head of the layer costs the same)."""
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
    one_heads, one_passes, one_dt = 2, 0, 0.0
    while one_passes == 0 or one_dt < single_seconds:
        t0 = time.perf_counter()
        oracle.prefill(q, k, v, ps.causal, ps.scale, heads=(0, one_heads), n_threads=1)
        one_dt += time.perf_counter() - t0
        one_passes += 1
    one_flops = one_passes * ps.flops * one_heads / heads
    return {"value": round(passes * ps.flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} passes over the whole prefill layer ({heads} heads x "
                      f"{ps.N_q} rows), float64, OpenMP over heads, {dt:.1f} s",
            "single_thread": {
                "value": round(one_flops / one_dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                "sample": f"{one_passes} passes over heads 0-{one_heads - 1} of the prefill "
                          f"layer, one thread, {one_dt:.1f} s"}}


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
    ap.add_argument("--reps", type=int, default=0,
                    help="repetitions of the K-step region (default: at least 21, about 1 s)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload blocks after the step (profiling runs)")
    ap.add_argument("--configs", default="",
                    help="comma-separated groups of per-workload blocks to run (sweep, long, "
                         "backward, decode, decode_fp8, decode_int8; profiling runs); default all")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
