"""GPU parity of the attention backward (dQ, dK, dV with the GQA head
reduction) against the float64 oracle's prefill_backward (microLLM-rocm
optimisation log, Experiments 051-057).

The kernel takes o and the per-row lse from this library's own forward
(gqa_attn_fwd_lse), as a caller would, and dO; the oracle recomputes
everything from q, k, v and dO in float64.

Tolerance (the pages fix none for the backward; derived from the
arithmetic): per gradient tensor G, max |G - G_ref| <= 2e-2 * max |G_ref|
and mean |G - G_ref| <= 1e-2 * mean |G_ref|. The kernel rounds P and dS to
bf16 before the products (relative error 2^-9 each), accumulates in fp32
and rounds the gradients to bf16; an emulation of exactly that arithmetic
in numpy reaches at most 6.7e-3 * max |G_ref| and 2.3e-3 * mean |G_ref|
on the shapes below. Gradients grow with the number of rows that attend a
key (dV of key 0 under the causal mask sums over every row), hence bounds
relative to the tensor's own magnitude.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

REL_MAX = 2e-2
REL_MEAN = 1e-2


def _check(got, ref, what):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    err = np.abs(got - ref)
    mx, mean = err.max(), err.mean()
    assert mx <= REL_MAX * np.abs(ref).max(), f"{what}: max {mx:.3e} vs |ref| max {np.abs(ref).max():.3e}"
    assert mean <= REL_MEAN * np.abs(ref).mean(), f"{what}: mean {mean:.3e} vs |ref| mean {np.abs(ref).mean():.3e}"


def _run(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=causal, scale=scale)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ops.gqa_attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    return dq, dk, dv


SHAPES = [
    # B, H_q, H_kv, N_q, N_kv, d, causal
    (1, 4, 2, 128, 128, 64, False),
    (1, 4, 2, 300, 300, 64, True),     # ragged tail, several tiles
    (2, 6, 2, 200, 520, 128, True),    # N_q < N_kv bottom-right, group of 3
    (1, 8, 8, 384, 384, 128, True),    # MHA
    (1, 8, 1, 256, 700, 64, False),    # MQA, ragged K/V
    (2, 2, 1, 1, 129, 128, False),     # a single query row
    (1, 16, 2, 257, 257, 128, True),   # group of 8
    (1, 4, 1, 640, 640, 128, False),   # 5 key blocks through the K/V ring
    (1, 4, 2, 300, 300, 32, True),     # d = 32 and 96: zero-padded tiles of the
    (2, 6, 2, 200, 520, 96, True),     #   64- and 128-column kernels
    (1, 8, 1, 256, 700, 96, False),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_backward_matches_oracle(shape):
    B, H_q, H_kv, N_q, N_kv, d, causal = shape
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=400 + N_q)
    do = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=401 + N_q)[0]
    dq, dk, dv = _run(q, k, v, do, causal, d ** -0.5)
    rq, rk, rv = oracle.prefill_backward(q, k, v, do, causal, d ** -0.5)
    _check(dq, rq, f"dq {shape}")
    _check(dk, rk, f"dk {shape}")
    _check(dv, rv, f"dv {shape}")


def test_backward_deterministic():
    q, k, v = inputs.prefill_inputs(1, 8, 2, 512, 512, 128, torch.bfloat16, seed=410)
    do = inputs.prefill_inputs(1, 8, 2, 512, 512, 128, torch.bfloat16, seed=411)[0]
    a = _run(q, k, v, do, True, 128 ** -0.5)
    b = _run(q, k, v, do, True, 128 ** -0.5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_llama3_8b_heads(d):
    """The LLaMA-3-8B layer's heads (32 query, 8 K/V) at N = 1024 (the full
    2048-row layer is measured in the bench; the float64 backward oracle
    takes minutes there)."""
    q, k, v = inputs.prefill_inputs(1, 32, 8, 1024, 1024, d, torch.bfloat16, seed=420 + d)
    do = inputs.prefill_inputs(1, 32, 8, 1024, 1024, d, torch.bfloat16, seed=421 + d)[0]
    dq, dk, dv = _run(q, k, v, do, True, d ** -0.5)
    rq, rk, rv = oracle.prefill_backward(q, k, v, do, True, d ** -0.5)
    _check(dq, rq, "dq")
    _check(dk, rk, "dk")
    _check(dv, rv, "dv")


def test_backward_wide_logits():
    """q scaled by 8: peaked rows, where P = exp(s - lse) must use the
    forward's lse exactly."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 512, 512, 128, torch.bfloat16, seed=430)
    q = (q.float() * 8).to(torch.bfloat16)
    do = inputs.prefill_inputs(1, 4, 2, 512, 512, 128, torch.bfloat16, seed=431)[0]
    dq, dk, dv = _run(q, k, v, do, True, 128 ** -0.5)
    rq, rk, rv = oracle.prefill_backward(q, k, v, do, True, 128 ** -0.5)
    _check(dq, rq, "dq")
    _check(dk, rk, "dk")
    _check(dv, rv, "dv")
