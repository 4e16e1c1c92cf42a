"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws random tensors and
names the workload shapes, so that the CUDA path and the CPU oracle can be fed
identical values. Recipe:

* ``torch.Generator('cpu').manual_seed(seed)``; ``randn`` in fp32, iid N(0,1);
* bf16 inputs are the fp32 draws rounded to nearest-even by ``.to(bfloat16)``;
* draw order: q, k, v; for decode: seqlens (uniform on [1, max_len] via
  ``randint(1, max_len + 1)``), then q, k_cache, v_cache;
* cache rows at or beyond ``seqlens[b]`` are set to NaN, so a kernel that
  reads them produces NaN and fails parity;
* workload ``c`` uses seed ``1000 + c``; sweep variants add ``10 * sub``;
* ragged batches: lengths uniform on [lo, hi] via ``randint`` (their own
  seed), offsets ``cu[0] = 0, cu[b+1] = cu[b] + len[b]``, then q, k, v
  token-major ([total, H, d]) in that order.

The shapes follow the synthetic stand-ins for the pages' workloads: a tiny
fp32 GQA case, an MHA/GQA/MQA sweep, a LLaMA-3-8B-shaped prefill layer
(BootstrapAI evolution log, collab-014 "Kernel 9 GQA": seq 2048, H_q=32,
H_kv=8, d=128), a long-sequence case sized like the persistent-kernel entry's
"seq=4096, h=16, b=4" example, and a decode step against a bf16 K/V cache
(microLLM-rocm optimisation log, Experiments 064-065), and a ragged batch of
prompts prefilled in one call (microLLM-rocm optimisation log, Experiment
101) with the LLaMA-3-8B layer's heads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillShape:
    name: str
    B: int
    H_q: int
    H_kv: int
    N_q: int
    N_kv: int
    d: int
    causal: bool
    dtype: torch.dtype
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H_q*N_q*N_kv*d, halved when causal."""
        f = 4.0 * self.B * self.H_q * self.N_q * self.N_kv * self.d
        return f / 2 if self.causal else f


@dataclass(frozen=True)
class DecodeShape:
    name: str
    B: int
    H_q: int
    H_kv: int
    max_len: int
    d: int
    dtype: torch.dtype
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def sweep_shapes() -> list[PrefillShape]:
    """MHA/GQA/MQA sweep: B=2, H_q=8, H_kv in {8,4,1}, N=1024, d=64, bf16."""
    out = []
    for sub, h_kv in enumerate((8, 4, 1)):
        for causal in (False, True):
            out.append(PrefillShape(f"sweep_hkv{h_kv}_{'causal' if causal else 'full'}",
                                    2, 8, h_kv, 1024, 1024, 64, causal,
                                    torch.bfloat16, 1001 + 10 * sub + int(causal)))
    return out


TINY = PrefillShape("tiny_gqa_fp32", 1, 4, 2, 128, 128, 64, False, torch.float32, 1000)
LLAMA3_8B_LAYER = PrefillShape("llama3_8b_prefill_layer", 1, 32, 8, 2048, 2048, 128, True,
                               torch.bfloat16, 1002)
LONG_SEQ = PrefillShape("long_seq_persistent", 4, 16, 4, 4096, 4096, 64, True,
                        torch.bfloat16, 1003)


@dataclass(frozen=True)
class VarlenShape:
    name: str
    lens_q: tuple
    lens_k: tuple
    H_q: int
    H_kv: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: sum over sequences of 4*H_q*len_q*len_k*d, halved when
        causal (the dense layer's convention)."""
        f = sum(4.0 * self.H_q * lq * lk * self.d for lq, lk in zip(self.lens_q, self.lens_k))
        return f / 2 if self.causal else f


def varlen_batch_shape() -> VarlenShape:
    """Eight prompts of 256-4096 tokens (seeded), LLaMA-3-8B heads (32 / 8, d = 128),
    causal self-attention (len_k = len_q)."""
    lens = tuple(varlen_lengths(8, 256, 4096, seed=1005))
    return VarlenShape("llama3_8b_varlen_batch8", lens, lens, 32, 8, 128, True, 1006)


def varlen_inputs_for(shape: VarlenShape):
    return varlen_inputs(list(shape.lens_q), list(shape.lens_k), shape.H_q, shape.H_kv, shape.d,
                         torch.bfloat16, shape.seed)


def decode_shapes() -> list[DecodeShape]:
    """Decode against a bf16 cache: B in {1,8,64}, H_q=12, H_kv=2, d=128, max_len=2048."""
    return [DecodeShape(f"decode_b{b}", b, 12, 2, 2048, 128, torch.bfloat16, 1004 + 10 * i)
            for i, b in enumerate((1, 8, 64))]


def prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, dtype=torch.bfloat16, seed=0):
    """Return CPU tensors (q, k, v) in ``dtype``: q [B,H_q,N_q,d], k/v [B,H_kv,N_kv,d]."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, H_q, N_q, d, generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn(B, H_kv, N_kv, d, generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn(B, H_kv, N_kv, d, generator=g, dtype=torch.float32).to(dtype)
    return q, k, v


def prefill_inputs_for(shape: PrefillShape):
    return prefill_inputs(shape.B, shape.H_q, shape.H_kv, shape.N_q, shape.N_kv, shape.d,
                          shape.dtype, shape.seed)


def varlen_inputs(lens_q, lens_k, H_q, H_kv, d, dtype=torch.bfloat16, seed=0):
    """Return CPU tensors (q [total_q,H_q,d], k, v [total_k,H_kv,d], cu_q, cu_k int32 [B+1])
    for a ragged batch packed token-major; values N(0, 1) like prefill_inputs."""
    g = torch.Generator("cpu").manual_seed(seed)
    cu_q = torch.zeros(len(lens_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(lens_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.cumsum(torch.tensor(lens_q, dtype=torch.int64), 0).to(torch.int32)
    cu_k[1:] = torch.cumsum(torch.tensor(lens_k, dtype=torch.int64), 0).to(torch.int32)
    total_q, total_k = int(cu_q[-1]), int(cu_k[-1])
    q = torch.randn(total_q, H_q, d, generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn(total_k, H_kv, d, generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn(total_k, H_kv, d, generator=g, dtype=torch.float32).to(dtype)
    return q, k, v, cu_q, cu_k


def varlen_lengths(B, lo, hi, seed):
    """B sequence lengths drawn uniformly from [lo, hi] (seeded)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).tolist()


def decode_inputs(B, H_q, H_kv, max_len, d, dtype=torch.bfloat16, seed=0, seqlens=None):
    """Return CPU tensors (seqlens int32 [B], q [B,H_q,d], k_cache, v_cache [B,H_kv,max_len,d]).

    Rows at or beyond seqlens[b] of both caches are NaN."""
    g = torch.Generator("cpu").manual_seed(seed)
    drawn = torch.randint(1, max_len + 1, (B,), generator=g, dtype=torch.int64)
    if seqlens is None:
        seqlens = drawn
    seqlens = torch.as_tensor(seqlens, dtype=torch.int64).clone()
    q = torch.randn(B, H_q, d, generator=g, dtype=torch.float32).to(dtype)
    kc = torch.randn(B, H_kv, max_len, d, generator=g, dtype=torch.float32).to(dtype)
    vc = torch.randn(B, H_kv, max_len, d, generator=g, dtype=torch.float32).to(dtype)
    pos = torch.arange(max_len).view(1, 1, max_len, 1)
    dead = pos >= seqlens.view(B, 1, 1, 1)
    kc = kc.masked_fill(dead, float("nan"))
    vc = vc.masked_fill(dead, float("nan"))
    return seqlens.to(torch.int32), q, kc, vc


def decode_inputs_for(shape: DecodeShape):
    return decode_inputs(shape.B, shape.H_q, shape.H_kv, shape.max_len, shape.d, shape.dtype,
                         shape.seed)


# ---------------------------------------------------------------------------
# Structured variants for parity at wide logit spreads. Each starts from the
# iid draws above and overwrites column 0 of q and k, so the score of key j,
# q . k_j, gets one large, known component; the values stay bf16-exact
# (they are rounded like every other input). They exercise the running-max
# update of the online softmax, which iid N(0,1) inputs at scale 1/sqrt(d)
# hardly ever reach after the first key block.

def with_rising_logits(q, k, key_pos, step, q_level=8.0):
    """Copies of q, k with q[..., 0] = q_level and k[..., 0] = step * key_pos,
    so the score of every query row grows by q_level * step per key position.
    ``key_pos`` holds each key row's position inside its sequence and
    broadcasts against k[..., :1] (e.g. [1, 1, N, 1] for [B, H, N, d], or
    [total, 1, 1] for token-major rows)."""
    q = q.float().clone()
    k = k.float().clone()
    q[..., 0] = q_level
    k[..., :1] = step * key_pos.to(torch.float32).expand_as(k[..., :1])
    return q.to(torch.bfloat16), k.to(torch.bfloat16)


def with_dominant_keys(q, k, key_mask, level=64.0):
    """Copies of q, k with q[..., 0] = 2 + |q[..., 0]| (positive for every
    query row) and k[..., 0] = level on the key rows where ``key_mask`` (a
    bool tensor broadcasting against k[..., :1]) is set: each such key's score
    exceeds the others' by about 2 * level."""
    q = q.float().clone()
    k = k.float().clone()
    q[..., 0] = 2.0 + q[..., 0].abs()
    col = k[..., :1]
    k[..., :1] = torch.where(key_mask.expand_as(col), torch.full_like(col, level), col)
    return q.to(torch.bfloat16), k.to(torch.bfloat16)


def token_positions(cu_seqlens, total):
    """Position of each packed token inside its own sequence: int64 [total]."""
    cu = [int(x) for x in cu_seqlens]
    pos = torch.zeros(total, dtype=torch.int64)
    for b in range(len(cu) - 1):
        pos[cu[b]:cu[b + 1]] = torch.arange(cu[b + 1] - cu[b])
    return pos


def decode_inputs_fp8(B, H_q, H_kv, max_len, d, seed=0, seqlens=None):
    """decode_inputs with an fp8 cache: the same draws (q rounded to bf16),
    with each K/V head of the caches quantised to OCP FP8 E4M3: its scale is
    the largest |value| over the valid rows / 448 (fp32), its bytes
    torch.float8_e4m3fn(value / scale) (round to nearest even); rows at or
    beyond seqlens[b] hold the NaN code. Returns (seqlens, q, k8, v8,
    k_scale, v_scale): k8, v8 float8_e4m3fn [B,H_kv,max_len,d], the scales
    fp32 [H_kv]."""
    seqlens, q, kc, vc = decode_inputs(B, H_q, H_kv, max_len, d, torch.float32, seed, seqlens)
    pos = torch.arange(max_len).view(1, 1, max_len, 1)
    dead = pos >= seqlens.long().view(B, 1, 1, 1)
    out = []
    for x in (kc, vc):
        amax = torch.where(dead, torch.zeros_like(x), x).abs().amax(dim=(0, 2, 3))
        sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
        out.append(((x / sc.view(1, H_kv, 1, 1)).to(torch.float8_e4m3fn), sc))
    (k8, ks), (v8, vs) = out
    return seqlens, q.to(torch.bfloat16), k8, v8, ks, vs


def decode_inputs_int8(B, H_q, H_kv, max_len, d, seed=0, seqlens=None):
    """decode_inputs with an int8 cache: the same draws (q rounded to bf16),
    with each K/V head of the caches quantised symmetrically to int8: its
    scale is the largest |value| over the valid rows / 127 (fp32), its codes
    round(value / scale) (to nearest even) in [-127, 127]; rows at or beyond
    seqlens[b] hold -128, a code the quantiser never writes. Returns
    (seqlens, q, k8, v8, k_scale, v_scale): k8, v8 int8 [B,H_kv,max_len,d],
    the scales fp32 [H_kv]."""
    seqlens, q, kc, vc = decode_inputs(B, H_q, H_kv, max_len, d, torch.float32, seed, seqlens)
    pos = torch.arange(max_len).view(1, 1, max_len, 1)
    dead = pos >= seqlens.long().view(B, 1, 1, 1)
    out = []
    for x in (kc, vc):
        x = torch.where(dead, torch.zeros_like(x), x)
        amax = x.abs().amax(dim=(0, 2, 3))
        sc = torch.where(amax > 0, amax / 127.0, torch.ones_like(amax)).to(torch.float32)
        codes = torch.round(x / sc.view(1, H_kv, 1, 1)).clamp(-127, 127).to(torch.int8)
        out.append((torch.where(dead, torch.full_like(codes, -128), codes), sc))
    (k8, ks), (v8, vs) = out
    return seqlens, q.to(torch.bfloat16), k8, v8, ks, vs
