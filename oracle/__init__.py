"""Float64 CPU oracle for grouped-query scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline / reference legs may import this package. The product
library (``gqa_flash_attention_02_gb300``) never imports it, and this package
imports nothing from the product.

The arithmetic lives in ``gqa_oracle.c`` (plain C, float64, the definition of
attention written out loop by loop). This module compiles that file with gcc
and exposes it through ctypes, taking and returning numpy float64 arrays.
Inputs in bf16 or fp32 are widened exactly to float64 by the caller (every
bf16/fp32 value is representable in float64), so the oracle sees the very
values the GPU path sees.

What each function follows (page title and section):
  * head mapping h_kv = h_q / (H_q / H_kv) -- BootstrapAI evolution log,
    collab-014 "Kernel 9 GQA";
  * softmax as max / exp / sum / weighted average, which the online form of
    the tiled kernels equals -- BootstrapAI evolution log, collab-005
    "Kernel 2 tiling";
  * causal GQA without replicating K/V heads -- microLLM-rocm optimisation
    log, Experiment 044;
  * log-sum-exp merge of key-range partials -- microLLM-rocm optimisation
    log, Experiments 282-284 (split-sequence cached attention);
  * a ragged batch as the list of its sequences, each attended on its own
    -- microLLM-rocm optimisation log, Experiment 101;
  * attention backward with the GQA head reduction of dK and dV (numpy,
    float64) -- microLLM-rocm optimisation log, Experiments 051-057;
  * decode against an fp8 (e4m3) cache with per-K/V-head scales, the codes
    decoded from the format's definition -- microLLM-rocm optimisation log,
    Experiment 065;
  * decode against an int8 cache (one-byte two's-complement codes with an
    explicit per-K/V-head scale) -- microLLM-rocm optimisation log,
    Experiments 352 and 354 (the one-byte tensor with an explicit scale, read
    and widened inside the decode kernel).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgqa_oracle.so")

_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attend_row.argtypes = [_dp, _dp, _dp, ctypes.c_long,
                                              ctypes.c_long, ctypes.c_double,
                                              _dp, _dp]
            lib.oracle_attend_row.restype = None
            lib.oracle_prefill.argtypes = [_dp, _dp, _dp, _dp, _dp] + [ctypes.c_long] * 6 + [
                ctypes.c_int, ctypes.c_double, ctypes.c_long, ctypes.c_long, ctypes.c_int]
            lib.oracle_prefill.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [_dp, _dp, _dp, _ip, _dp, _dp] + [ctypes.c_long] * 5 + [
                ctypes.c_double]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_lse_merge.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_long, _dp, _dp]
            lib.oracle_lse_merge.restype = None
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening to a contiguous float64 numpy array (torch or numpy input)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch  # local: torch is only needed when a tensor is passed
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def attend_row(q_row, k_rows, v_rows, scale: float):
    """Attention of one query row q[d] over all rows of k[n][d], v[n][d].

    Returns (o[d], lse)."""
    q_row, k_rows, v_rows = _f64(q_row), _f64(k_rows), _f64(v_rows)
    n, d = k_rows.shape if k_rows.ndim == 2 else (0, q_row.shape[-1])
    o = np.empty(d, dtype=np.float64)
    lse = ctypes.c_double()
    _load().oracle_attend_row(_ptr(q_row), _ptr(k_rows), _ptr(v_rows), n, d,
                              float(scale), _ptr(o), ctypes.byref(lse))
    return o, lse.value


def prefill(q, k, v, causal: bool, scale: float, heads=None, n_threads: int = 1):
    """Prefill attention. q:[B,H_q,N_q,d], k,v:[B,H_kv,N_kv,d] -> (o, lse).

    ``heads`` optionally restricts the work to a contiguous range
    (begin, end) of flattened b*H_q + h_q heads; the other heads of the
    returned arrays are NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:3], np.nan)
    begin, end = (0, B * H_q) if heads is None else heads
    rc = _load().oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                B, H_q, H_kv, N_q, N_kv, d, int(bool(causal)),
                                float(scale), begin, end, int(n_threads))
    if rc != 0:
        raise ValueError("oracle_prefill: H_q must be a positive multiple of H_kv")
    return o, lse


def prefill_rows(q, k, v, causal: bool, scale: float, rows):
    """Prefill output for selected rows only.

    ``rows`` is an iterable of (b, h_q, i). Returns (o[len(rows), d], lse[len(rows)])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    group = H_q // H_kv
    rows = list(rows)
    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    for r, (b, h_q, i) in enumerate(rows):
        n = N_kv if not causal else max(0, min(N_kv, i + (N_kv - N_q) + 1))
        h_kv = h_q // group
        o[r], lse[r] = attend_row(q[b, h_q, i], k[b, h_kv, :n], v[b, h_kv, :n], scale)
    return o, lse


def _offsets(cu) -> np.ndarray:
    if hasattr(cu, "detach"):
        cu = cu.detach().cpu().numpy()
    return np.asarray(cu, dtype=np.int64).reshape(-1)


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float,
                   n_threads: int = 1):
    """Ragged-batch prefill. q:[total_q,H_q,d], k,v:[total_k,H_kv,d] (token-major).

    Sequence b owns query rows [cu_q[b], cu_q[b+1]) and key rows
    [cu_k[b], cu_k[b+1]) and is attended on its own, exactly as a batch of
    one by ``prefill`` (bottom-right causal inside the sequence): the ragged
    batch is the list of its sequences (microLLM-rocm optimisation log,
    Experiment 101, prompts batched into one prefill).
    Returns (o [total_q,H_q,d], lse [H_q,total_q]); rows no sequence owns are NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _offsets(cu_seqlens_q), _offsets(cu_seqlens_k)
    if cq.shape != ck.shape or cq.size < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be [B + 1]")
    o = np.full(q.shape, np.nan)
    lse = np.full((q.shape[1], q.shape[0]), np.nan)
    for b in range(cq.size - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        # [len, H, d] -> [1, H, len, d]
        qb = np.ascontiguousarray(q[q0:q1].transpose(1, 0, 2))[None]
        kb = np.ascontiguousarray(k[k0:k1].transpose(1, 0, 2))[None]
        vb = np.ascontiguousarray(v[k0:k1].transpose(1, 0, 2))[None]
        ob, lb = prefill(qb, kb, vb, causal, scale, n_threads=n_threads)
        o[q0:q1] = ob[0].transpose(1, 0, 2)
        lse[:, q0:q1] = lb[0]
    return o, lse


def prefill_varlen_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float, rows):
    """Ragged-batch prefill output for selected (token t, head h_q) rows only.

    Returns (o[len(rows), d], lse[len(rows)])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cq, ck = _offsets(cu_seqlens_q), _offsets(cu_seqlens_k)
    H_q, H_kv = q.shape[1], k.shape[1]
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    group = H_q // H_kv
    rows = list(rows)
    o = np.empty((len(rows), q.shape[2]))
    lse = np.empty(len(rows))
    for r, (t, h_q) in enumerate(rows):
        b = int(np.searchsorted(cq, t, side="right")) - 1
        i = t - int(cq[b])
        len_q, k0, len_k = int(cq[b + 1] - cq[b]), int(ck[b]), int(ck[b + 1] - ck[b])
        n = len_k if not causal else max(0, min(len_k, i + (len_k - len_q) + 1))
        h_kv = h_q // group
        o[r], lse[r] = attend_row(q[t, h_q], k[k0:k0 + n, h_kv], v[k0:k0 + n, h_kv], scale)
    return o, lse


def prefill_backward(q, k, v, do, causal: bool, scale: float):
    """Gradients of prefill attention. q:[B,H_q,N_q,d], k,v:[B,H_kv,N_kv,d],
    do = dL/dO:[B,H_q,N_q,d] -> (dq, dk, dv) in float64.

    Row recompute, then the softmax backward, then the GQA head reduction
    of dK and dV over the query heads of a group (microLLM-rocm optimisation
    log, Experiments 051-057: causal GQA attention backward). Per (b, h_q),
    with h_kv = h_q / (H_q / H_kv) and the bottom-right causal mask:
        S = scale Q K^T (masked to -inf),  P = softmax(S),  O = P V
        dV[h_kv] += P^T dO                dP = dO V^T
        Delta_i = sum_d dO_i O_i          dS = P * (dP - Delta)
        dQ = scale dS K                   dK[h_kv] += scale dS^T Q
    A matrix product serves as a step; nothing else is fused or reordered.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    if H_kv <= 0 or H_q % H_kv:
        raise ValueError("H_q must be a positive multiple of H_kv")
    group = H_q // H_kv
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    rows = np.arange(N_q)[:, None]
    keys = np.arange(N_kv)[None, :]
    visible = keys <= rows + (N_kv - N_q) if causal else np.ones((N_q, N_kv), dtype=bool)
    for b in range(B):
        for h in range(H_q):
            hk = h // group
            s = scale * (q[b, h] @ k[b, hk].T)
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)  # a row with no visible key
            e = np.where(visible, np.exp(s - m), 0.0)
            z = e.sum(axis=1, keepdims=True)
            p = np.divide(e, z, out=np.zeros_like(e), where=z > 0)
            o = p @ v[b, hk]
            dv[b, hk] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, hk].T
            delta = (do[b, h] * o).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def decode(q, k_cache, v_cache, seqlens, scale: float):
    """Decode attention. q:[B,H_q,d], caches [B,H_kv,max_len,d], seqlens[B] -> (o, lse)."""
    q, k_cache, v_cache = _f64(q), _f64(k_cache), _f64(v_cache)
    if hasattr(seqlens, "detach"):
        seqlens = seqlens.detach().cpu().numpy()
    seqlens = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    B, H_q, d = q.shape
    _, H_kv, max_len, _ = k_cache.shape
    o = np.empty(q.shape)
    lse = np.empty(q.shape[:2])
    rc = _load().oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                               seqlens.ctypes.data_as(_ip), _ptr(o), _ptr(lse),
                               B, H_q, H_kv, max_len, d, float(scale))
    if rc == -1:
        raise ValueError("oracle_decode: H_q must be a positive multiple of H_kv")
    if rc == -2:
        raise ValueError("oracle_decode: seqlens outside [0, max_len]")
    return o, lse


def e4m3_value(codes):
    """Values of OCP FP8 E4M3 codes (bytes) as float64, from the format's
    definition: bit 7 sign, bits 6-3 exponent with bias 7, bits 2-0 mantissa;
    exponent field 0 is subnormal, (m / 8) 2^-6; otherwise (1 + m / 8)
    2^(e - 7); the codes S.1111.111 (0x7F, 0xFF) are NaN and there are no
    infinities (largest finite value 448)."""
    if hasattr(codes, "detach"):
        import torch
        t = codes.detach().cpu()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        codes = t.numpy()
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return np.where((c & 0x7F) == 0x7F, np.nan, sign * mag)


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, seqlens, scale: float):
    """Decode against an fp8 cache: the cache value of a byte is its e4m3
    value times the scale of its K/V head (microLLM-rocm optimisation log,
    Experiment 065: a narrower cache, attention in full precision); the
    widened caches then go through ``decode``. Returns (o, lse)."""
    ks, vs = _f64(k_scale), _f64(v_scale)
    k = e4m3_value(k_codes) * ks[None, :, None, None]
    v = e4m3_value(v_codes) * vs[None, :, None, None]
    return decode(q, k, v, seqlens, scale)


def int8_value(codes):
    """Values of int8 codes (bytes, two's complement) as float64: bit 7
    weighs -128, bits 6-0 weigh 64, 32, ..., 1."""
    if hasattr(codes, "detach"):
        import torch
        t = codes.detach().cpu()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        codes = t.numpy()
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return ((c & 0x7F) - (c & 0x80)).astype(np.float64)


def decode_int8(q, k_codes, v_codes, k_scale, v_scale, seqlens, scale: float):
    """Decode against an int8 cache: the cache value of a byte is its int8
    value times the scale of its K/V head (microLLM-rocm optimisation log,
    Experiments 352 and 354: a one-byte tensor with an explicit scale); the
    widened caches then go through ``decode``. Returns (o, lse)."""
    ks, vs = _f64(k_scale), _f64(v_scale)
    k = int8_value(k_codes) * ks[None, :, None, None]
    v = int8_value(v_codes) * vs[None, :, None, None]
    return decode(q, k, v, seqlens, scale)


def lse_merge(o_parts, lse_parts):
    """Merge partial results o_parts[S,d], lse_parts[S] -> (o[d], lse)."""
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    S, d = o_parts.shape
    o = np.empty(d)
    lse = ctypes.c_double()
    _load().oracle_lse_merge(_ptr(o_parts), _ptr(lse_parts), S, d, _ptr(o),
                             ctypes.byref(lse))
    return o, lse.value
