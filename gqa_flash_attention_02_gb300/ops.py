"""ctypes binding of libgqa_attn.so with the C ABI's names.

Argument marshalling only: shapes and dtypes are checked, pointers and the
current CUDA stream are passed through, and every step of the computation
runs in the library's kernels. If the library cannot be loaded the call
raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GQA_OK = 0
STATUS_NAMES = {
    0: "GQA_OK",
    1: "GQA_ERR_INVALID_ARG",
    2: "GQA_ERR_UNSUPPORTED",
    3: "GQA_ERR_CUDA",
    4: "GQA_ERR_DEVICE_TIMEOUT",
    5: "GQA_ERR_OOM",
    6: "GQA_ERR_BAD_SEQLEN",
}

EXPORTED = [
    "gqa_attn_fwd", "gqa_attn_fwd_f32", "gqa_attn_decode", "gqa_attn_decode_chunked",
    "gqa_attn_decode_f32", "gqa_attn_status_string", "gqa_attn_get_device_error",
    "gqa_attn_prefill_plan", "gqa_attn_selftest_wait_timeout", "gqa_attn_shutdown",
    "gqa_attn_decode_noalloc", "gqa_attn_fwd_lse", "gqa_attn_decode_lse",
    "gqa_attn_fwd_varlen", "gqa_attn_fwd_varlen_lse", "gqa_attn_fwd_bshd", "gqa_attn_bwd",
    "gqa_attn_decode_fp8", "gqa_attn_fwd_strided", "gqa_attn_decode_int8",
    "gqa_attn_selftest_decode_early_lengths",
]


class GqaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgqa_attn.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"libgqa_attn.so not found at {path}")
            lib = ctypes.CDLL(path)
            fwd = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp]
            for name in ("gqa_attn_fwd", "gqa_attn_fwd_f32"):
                getattr(lib, name).argtypes = fwd
                getattr(lib, name).restype = _i
            dec = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
            for name in ("gqa_attn_decode", "gqa_attn_decode_f32"):
                getattr(lib, name).argtypes = dec
                getattr(lib, name).restype = _i
            lib.gqa_attn_decode_chunked.argtypes = dec[:-1] + [_i, _vp]
            lib.gqa_attn_decode_chunked.restype = _i
            lib.gqa_attn_decode_noalloc.argtypes = dec
            lib.gqa_attn_decode_noalloc.restype = _i
            lib.gqa_attn_fwd_lse.argtypes = fwd[:4] + [_vp] + fwd[4:]
            lib.gqa_attn_fwd_lse.restype = _i
            lib.gqa_attn_decode_lse.argtypes = dec[:5] + [_vp] + dec[5:]
            lib.gqa_attn_decode_lse.restype = _i
            # q, k, v, o, cu_q, cu_k, B, H_q, H_kv, total_q, total_k, d, causal, scale, stream
            var = [_vp] * 6 + [_i] * 7 + [_f, _vp]
            lib.gqa_attn_fwd_varlen.argtypes = var
            lib.gqa_attn_fwd_varlen.restype = _i
            lib.gqa_attn_fwd_varlen_lse.argtypes = var[:4] + [_vp] + var[4:]
            lib.gqa_attn_fwd_varlen_lse.restype = _i
            lib.gqa_attn_fwd_bshd.argtypes = fwd
            lib.gqa_attn_fwd_bshd.restype = _i
            lib.gqa_attn_bwd.argtypes = [_vp] * 9 + [_i] * 7 + [_f, _vp]
            lib.gqa_attn_bwd.restype = _i
            lib.gqa_attn_decode_fp8.argtypes = [_vp] * 8 + [_i] * 5 + [_f, _vp]
            lib.gqa_attn_decode_fp8.restype = _i
            lib.gqa_attn_decode_int8.argtypes = [_vp] * 8 + [_i] * 5 + [_f, _vp]
            lib.gqa_attn_decode_int8.restype = _i
            _ll = ctypes.c_longlong
            lib.gqa_attn_fwd_strided.argtypes = ([_vp, _ll, _ll, _ll] * 4 + [_i] * 7 + [_f, _vp])
            lib.gqa_attn_fwd_strided.restype = _i
            lib.gqa_attn_status_string.argtypes = [_i]
            lib.gqa_attn_status_string.restype = ctypes.c_char_p
            lib.gqa_attn_get_device_error.argtypes = [_vp]
            lib.gqa_attn_get_device_error.restype = _i
            lib.gqa_attn_prefill_plan.argtypes = [_i] * 7 + [ctypes.POINTER(_i)]
            lib.gqa_attn_prefill_plan.restype = _i
            lib.gqa_attn_selftest_wait_timeout.argtypes = [_i, _vp]
            lib.gqa_attn_selftest_wait_timeout.restype = _i
            lib.gqa_attn_selftest_decode_early_lengths.argtypes = [_vp] * 7 + [_i] * 5 + [_f, _vp]
            lib.gqa_attn_selftest_decode_early_lengths.restype = _i
            lib.gqa_attn_shutdown.argtypes = []
            lib.gqa_attn_shutdown.restype = None
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gqa_attn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != GQA_OK:
        raise GqaError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, name: str, ndim: int):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------- prefill

def gqa_attn_fwd(q, k, v, o=None, causal=False, scale=None, stream=None):
    """bf16 prefill. q [B,H_q,N_q,d], k/v [B,H_kv,N_kv,d] -> o [B,H_q,N_q,d] (bf16)."""
    return _fwd("gqa_attn_fwd", torch.bfloat16, q, k, v, o, causal, scale, stream)


def gqa_attn_fwd_lse(q, k, v, o=None, lse=None, causal=False, scale=None, stream=None):
    """bf16 prefill that also returns each row's log-sum-exp (fp32 [B,H_q,N_q]).
    Returns (o, lse)."""
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("lse must be [B, H_q, N_q]")
    o = _fwd("gqa_attn_fwd_lse", torch.bfloat16, q, k, v, o, causal, scale, stream,
             lse=_dev(lse, torch.float32, "lse", 3))
    return o, lse


def gqa_attn_fwd_f32(q, k, v, o=None, causal=False, scale=None, stream=None):
    """fp32 prefill with the same layouts."""
    return _fwd("gqa_attn_fwd_f32", torch.float32, q, k, v, o, causal, scale, stream)


def _fwd(name, dtype, q, k, v, o, causal, scale, stream, lse=None):
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    args = (_dev(q, dtype, "q", 4), _dev(k, dtype, "k", 4), _dev(v, dtype, "v", 4),
            _dev(o, dtype, "o", 4))
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d or \
            tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, k, v, o")
    if lse is not None:
        args = args + (lse,)
    rc = getattr(load(), name)(*args, B, H_q, H_kv, N_q, N_kv, d, int(bool(causal)),
                               float(scale), _stream(stream))
    _check(rc, name)
    return o


def gqa_attn_fwd_strided(q, k, v, o=None, causal=False, scale=None, stream=None):
    """bf16 prefill on strided views: q, o [B,H_q,N_q,d] and k, v [B,H_kv,N_kv,d]
    as torch views with any batch / head / row strides (the last dim contiguous),
    e.g. slices of a fused QKV buffer. ``o`` defaults to a packed tensor."""
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    if o is None:
        o = torch.empty((B, H_q, N_q, d), dtype=q.dtype, device=q.device)
    if scale is None:
        scale = d ** -0.5
    args = []
    for name, t, shape in (("q", q, (B, H_q, N_q, d)), ("k", k, (B, H_kv, N_kv, d)),
                           ("v", v, (B, H_kv, N_kv, d)), ("o", o, (B, H_q, N_q, d))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a bf16 CUDA tensor")
        if tuple(t.shape) != shape or t.stride(3) != 1:
            raise ValueError(f"{name} must be {shape} with a contiguous last dim")
        args += [ctypes.c_void_p(t.data_ptr()), t.stride(0), t.stride(1), t.stride(2)]
    rc = load().gqa_attn_fwd_strided(*args, B, H_q, H_kv, N_q, N_kv, d, int(bool(causal)),
                                     float(scale), _stream(stream))
    _check(rc, "gqa_attn_fwd_strided")
    return o


# ---------------------------------------------------------------- backward

def gqa_attn_bwd(q, k, v, o, dout, lse, dq=None, dk=None, dv=None, causal=False, scale=None,
                 stream=None):
    """Gradients of bf16 prefill attention. q, o, dout [B,H_q,N_q,d], k, v [B,H_kv,N_kv,d]
    (bf16), lse fp32 [B,H_q,N_q] from gqa_attn_fwd_lse -> (dq, dk, dv), bf16."""
    B, H_q, N_q, d = q.shape
    _, H_kv, N_kv, _ = k.shape
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d or \
            tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) or \
            tuple(dq.shape) != tuple(q.shape) or tuple(dk.shape) != tuple(k.shape) or \
            tuple(dv.shape) != tuple(k.shape) or tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("shape mismatch between q, k, v, o, dout, lse and the gradients")
    bf = torch.bfloat16
    rc = load().gqa_attn_bwd(_dev(q, bf, "q", 4), _dev(k, bf, "k", 4), _dev(v, bf, "v", 4),
                             _dev(o, bf, "o", 4), _dev(dout, bf, "dout", 4),
                             _dev(lse, torch.float32, "lse", 3), _dev(dq, bf, "dq", 4),
                             _dev(dk, bf, "dk", 4), _dev(dv, bf, "dv", 4), B, H_q, H_kv, N_q,
                             N_kv, d, int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "gqa_attn_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------- ragged batches

def gqa_attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, o=None, causal=False, scale=None,
                        stream=None):
    """bf16 prefill over a ragged batch packed token-major.

    q [total_q,H_q,d], k/v [total_k,H_kv,d], cu_seqlens_q/k int32 [B+1] on the
    device (sequence b owns rows [cu[b], cu[b+1])) -> o [total_q,H_q,d] (bf16)."""
    return _fwd_varlen("gqa_attn_fwd_varlen", q, k, v, cu_seqlens_q, cu_seqlens_k, o, causal,
                       scale, stream)


def gqa_attn_fwd_varlen_lse(q, k, v, cu_seqlens_q, cu_seqlens_k, o=None, lse=None, causal=False,
                            scale=None, stream=None):
    """gqa_attn_fwd_varlen that also returns each row's log-sum-exp, fp32
    [H_q, total_q]. Returns (o, lse)."""
    if lse is None:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    if tuple(lse.shape) != (q.shape[1], q.shape[0]):
        raise ValueError("lse must be [H_q, total_q]")
    o = _fwd_varlen("gqa_attn_fwd_varlen_lse", q, k, v, cu_seqlens_q, cu_seqlens_k, o, causal,
                    scale, stream, lse=_dev(lse, torch.float32, "lse", 2))
    return o, lse


def gqa_attn_fwd_bshd(q, k, v, o=None, causal=False, scale=None, stream=None):
    """bf16 prefill, token-major batch: q [B,N_q,H_q,d], k/v [B,N_kv,H_kv,d] -> o [B,N_q,H_q,d]."""
    B, N_q, H_q, d = q.shape
    _, N_kv, H_kv, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != d or \
            tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, k, v, o")
    rc = load().gqa_attn_fwd_bshd(_dev(q, torch.bfloat16, "q", 4), _dev(k, torch.bfloat16, "k", 4),
                                  _dev(v, torch.bfloat16, "v", 4), _dev(o, torch.bfloat16, "o", 4),
                                  B, H_q, H_kv, N_q, N_kv, d, int(bool(causal)), float(scale),
                                  _stream(stream))
    _check(rc, "gqa_attn_fwd_bshd")
    return o


def _fwd_varlen(name, q, k, v, cu_q, cu_k, o, causal, scale, stream, lse=None):
    total_q, H_q, d = q.shape
    total_k, H_kv, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    if tuple(v.shape) != tuple(k.shape) or k.shape[2] != d or tuple(o.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q, k, v, o")
    if cu_q.dim() != 1 or tuple(cu_k.shape) != tuple(cu_q.shape) or cu_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be [B + 1] with B >= 1")
    args = [_dev(q, torch.bfloat16, "q", 3), _dev(k, torch.bfloat16, "k", 3),
            _dev(v, torch.bfloat16, "v", 3), _dev(o, torch.bfloat16, "o", 3)]
    if lse is not None:
        args.append(lse)
    args += [_dev(cu_q, torch.int32, "cu_seqlens_q", 1), _dev(cu_k, torch.int32, "cu_seqlens_k", 1)]
    rc = getattr(load(), name)(*args, cu_q.numel() - 1, H_q, H_kv, total_q, total_k, d,
                               int(bool(causal)), float(scale), _stream(stream))
    _check(rc, name)
    return o


# ---------------------------------------------------------------- decode

def gqa_attn_decode(q, k_cache, v_cache, seqlens, o=None, scale=None, chunk_tokens=0,
                    stream=None):
    """bf16 decode. q [B,H_q,d], caches [B,H_kv,max_len,d], seqlens int32 [B] -> o [B,H_q,d]."""
    return _decode("gqa_attn_decode_chunked", torch.bfloat16, q, k_cache, v_cache, seqlens, o,
                   scale, chunk_tokens, stream)


def gqa_attn_decode_lse(q, k_cache, v_cache, seqlens, o=None, lse=None, scale=None, stream=None):
    """bf16 decode that also returns each head's log-sum-exp (fp32 [B,H_q],
    -inf for an empty sequence). Returns (o, lse)."""
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if tuple(lse.shape) != tuple(q.shape[:2]):
        raise ValueError("lse must be [B, H_q]")
    o = _decode("gqa_attn_decode_lse", torch.bfloat16, q, k_cache, v_cache, seqlens, o, scale,
                None, stream, lse=_dev(lse, torch.float32, "lse", 2))
    return o, lse


def gqa_attn_decode_noalloc(q, k_cache, v_cache, seqlens, o, scale=None, stream=None):
    """bf16 decode that allocates nothing (the library's fixed scratch array);
    ``o`` must be given. See gqa_attn_decode_noalloc in include/gqa_attn.h."""
    return _decode("gqa_attn_decode_noalloc", torch.bfloat16, q, k_cache, v_cache, seqlens, o,
                   scale, None, stream)


def _decode_byte_cache(entry, dtypes, q, k_cache, v_cache, k_scale, v_scale, seqlens, o, lse,
                       scale, stream):
    B, H_q, d = q.shape
    _, H_kv, max_len, _ = k_cache.shape
    if o is None:
        o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not t.is_cuda or t.dtype not in dtypes or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-d CUDA tensor of "
                             f"{' / '.join(str(x) for x in dtypes)}")
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != d or tuple(o.shape) != tuple(q.shape) or \
            tuple(seqlens.shape) != (B,) or tuple(k_scale.shape) != (H_kv,) or \
            tuple(v_scale.shape) != (H_kv,):
        raise ValueError("shape mismatch between q, caches, scales, seqlens, o")
    lse_p = None
    if lse is not None:
        if tuple(lse.shape) != (B, H_q):
            raise ValueError("lse must be [B, H_q]")
        lse_p = _dev(lse, torch.float32, "lse", 2)
    rc = getattr(load(), entry)(
        _dev(q, torch.bfloat16, "q", 3), ctypes.c_void_p(k_cache.data_ptr()),
        ctypes.c_void_p(v_cache.data_ptr()), _dev(k_scale, torch.float32, "k_scale", 1),
        _dev(v_scale, torch.float32, "v_scale", 1), _dev(seqlens, torch.int32, "seqlens", 1),
        _dev(o, torch.bfloat16, "o", 3), lse_p, B, H_q, H_kv, max_len, d, float(scale),
        _stream(stream))
    _check(rc, entry)
    return o


def gqa_attn_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, seqlens, o=None, lse=None,
                        scale=None, stream=None):
    """Decode against an fp8 (e4m3) cache. q [B,H_q,d] bf16; caches [B,H_kv,max_len,d] of
    torch.float8_e4m3fn (or uint8 bytes); k_scale, v_scale fp32 [H_kv]; seqlens int32 [B].
    Returns o [B,H_q,d] bf16 (and fills lse [B,H_q] fp32 when given)."""
    dtypes = tuple(t for t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if t is not None)
    return _decode_byte_cache("gqa_attn_decode_fp8", dtypes, q, k_cache, v_cache, k_scale,
                              v_scale, seqlens, o, lse, scale, stream)


def gqa_attn_decode_int8(q, k_cache, v_cache, k_scale, v_scale, seqlens, o=None, lse=None,
                         scale=None, stream=None):
    """Decode against an int8 cache. q [B,H_q,d] bf16; caches [B,H_kv,max_len,d] torch.int8
    (two's-complement codes); k_scale, v_scale fp32 [H_kv]; seqlens int32 [B].
    Returns o [B,H_q,d] bf16 (and fills lse [B,H_q] fp32 when given)."""
    return _decode_byte_cache("gqa_attn_decode_int8", (torch.int8,), q, k_cache, v_cache,
                              k_scale, v_scale, seqlens, o, lse, scale, stream)


def gqa_attn_decode_f32(q, k_cache, v_cache, seqlens, o=None, scale=None, stream=None):
    return _decode("gqa_attn_decode_f32", torch.float32, q, k_cache, v_cache, seqlens, o, scale,
                   None, stream)


def _decode(name, dtype, q, kc, vc, seqlens, o, scale, chunk, stream, lse=None):
    B, H_q, d = q.shape
    _, H_kv, max_len, _ = kc.shape
    if o is None:
        o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    if tuple(vc.shape) != tuple(kc.shape) or kc.shape[0] != B or kc.shape[3] != d or \
            tuple(o.shape) != tuple(q.shape) or tuple(seqlens.shape) != (B,):
        raise ValueError("shape mismatch between q, caches, seqlens, o")
    args = [_dev(q, dtype, "q", 3), _dev(kc, dtype, "k_cache", 4), _dev(vc, dtype, "v_cache", 4),
            _dev(seqlens, torch.int32, "seqlens", 1), _dev(o, dtype, "o", 3)]
    if lse is not None:
        args.append(lse)
    args += [B, H_q, H_kv, max_len, d, float(scale)]
    if chunk is not None:
        args.append(int(chunk))
    rc = getattr(load(), name)(*args, _stream(stream))
    _check(rc, name)
    return o


# ---------------------------------------------------------------- misc

def gqa_attn_get_device_error(stream=None) -> int:
    return load().gqa_attn_get_device_error(_stream(stream))


def gqa_attn_prefill_plan(B, H_q, H_kv, N_q, N_kv, causal):
    """Return the scheduler's unit list: [(b, h_kv, (h_q0, qt0, nb0), (h_q1, qt1, nb1)), ...]."""
    lib = load()
    n = lib.gqa_attn_prefill_plan(B, H_q, H_kv, N_q, N_kv, int(bool(causal)), -1, None)
    if n < 0:
        raise ValueError("invalid sizes")
    out = (ctypes.c_int * 8)()
    units = []
    for u in range(n):
        lib.gqa_attn_prefill_plan(B, H_q, H_kv, N_q, N_kv, int(bool(causal)), u, out)
        units.append((out[0], out[1], (out[2], out[3], out[4]), (out[5], out[6], out[7])))
    return units


def gqa_attn_selftest_wait_timeout(timeout_us: int = 1000, stream=None) -> int:
    return load().gqa_attn_selftest_wait_timeout(int(timeout_us), _stream(stream))


def gqa_attn_selftest_decode_early_lengths(q, k_cache, v_cache, seqlens, seqlens_early,
                                           scale=None, stream=None):
    """gqa_attn_decode_lse with the kernel's pre-wait read of the lengths taken
    from ``seqlens_early`` (int32 [B] on the device). Returns (o, lse)."""
    B, H_q, d = q.shape
    if tuple(seqlens_early.shape) != (B,):
        raise ValueError("seqlens_early must be [B]")
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    early = _dev(seqlens_early, torch.int32, "seqlens_early", 1)
    _, H_kv, max_len, _ = k_cache.shape
    o = torch.empty_like(q)
    if scale is None:
        scale = d ** -0.5
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != d or tuple(seqlens.shape) != (B,):
        raise ValueError("shape mismatch between q, caches, seqlens")
    rc = load().gqa_attn_selftest_decode_early_lengths(
        _dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
        _dev(v_cache, torch.bfloat16, "v_cache", 4), _dev(seqlens, torch.int32, "seqlens", 1),
        early, _dev(o, torch.bfloat16, "o", 3), _dev(lse, torch.float32, "lse", 2), B, H_q, H_kv,
        max_len, d, float(scale), _stream(stream))
    _check(rc, "gqa_attn_selftest_decode_early_lengths")
    return o, lse


def gqa_attn_shutdown():
    load().gqa_attn_shutdown()
