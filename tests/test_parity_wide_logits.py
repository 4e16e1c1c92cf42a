"""GPU parity at wide logit spreads: the running-maximum update of the
online softmax (BootstrapAI evolution log, collab-005 "Kernel 2 tiling").

The tensor-core prefill keeps a reference maximum per row and raises it
(rescaling O in tensor memory) only when a later key block's maximum exceeds
it by more than a threshold of 2^8 (log2 units). On iid N(0,1) inputs at
scale 1/sqrt(d) that almost never happens after the first block, so these
cases build inputs where it must:

  * rising logits: q[..., 0] = 8 and k[..., j, 0] = 0.1 j, so every row's
    score grows by 0.8 per key; times scale * log2(e) that is more than 10
    log2 units per 128-key block at d = 128 (more than 14 at d = 64), so
    every row raises its maximum at every block after the first;
  * one dominant key in the last key block of a long row (k[..., 0] = 256
    or 64 against q[..., 0] >= 2, so its score leads the others' by tens of
    natural-log units): the rows that see it raise their maximum at that
    block;
  * q scaled by 4, 8 and 16: wide score spreads, where the bf16 rounding of
    the weights and the lag of the reference maximum weigh most;
  * a zero scale (uniform weights) and a negative one.

Everything is compared element by element with the float64 oracle at the
bf16 bounds (max abs <= 2e-2, mean abs <= 2e-3; lse max abs <= 5e-3).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

BF16_MAX = 2e-2
BF16_MEAN = 2e-3
LSE_MAX = 5e-3
THREADS = max(1, min(16, os.cpu_count() or 1))
STEP = 0.1


def _check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got - ref)
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, \
        f"{what}: max {d.max():.3e} mean {d.mean():.3e}"


def _check_lse(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf pattern"
    m = np.isfinite(ref)
    err = np.abs(got[m] - ref[m]).max() if m.any() else 0.0
    assert err <= LSE_MAX, f"{what}: lse max err {err:.3e}"


def _fwd_lse(q, k, v, causal, scale):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.full_like(qd, float("nan"))
    o, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, o, causal=causal, scale=scale)
    o_plain = ops.gqa_attn_fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy(), o_plain.float().cpu().numpy()


def _varlen_lse(q, k, v, cu_q, cu_k, causal, scale):
    qd, kd, vd, cqd, ckd = (t.cuda() for t in (q, k, v, cu_q, cu_k))
    o = torch.full_like(qd, float("nan"))
    o, lse = ops.gqa_attn_fwd_varlen_lse(qd, kd, vd, cqd, ckd, o, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


# ------------------------------------------------------------------ rising logits

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_rising_logits_prefill(d, causal):
    """Every row's maximum jumps at every key block (5 blocks)."""
    N = 640
    q, k, v = inputs.prefill_inputs(1, 4, 2, N, N, d, torch.bfloat16, seed=200 + d)
    q, k = inputs.with_rising_logits(q, k, torch.arange(N).view(1, 1, N, 1), STEP)
    got, lse, plain = _fwd_lse(q, k, v, causal, d ** -0.5)
    ref, ref_lse = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check(got, ref, f"rising logits d {d} causal {causal}")
    _check(plain, ref, f"rising logits d {d} causal {causal}, plain entry point")
    _check_lse(lse, ref_lse, f"rising logits d {d} causal {causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_rising_logits_varlen(d):
    """The same through the ragged-batch path: positions restart at every
    sequence, one sequence follows a cached prefix (more keys than queries)."""
    lens_q, lens_k = [600, 130, 1, 300], [600, 130, 1, 450]
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, 8, 2, d, torch.bfloat16,
                                               seed=210 + d)
    pos = inputs.token_positions(cu_k, k.shape[0]).view(-1, 1, 1)
    q, k = inputs.with_rising_logits(q, k, pos, STEP)
    got, lse = _varlen_lse(q, k, v, cu_q, cu_k, True, d ** -0.5)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, d ** -0.5,
                                         n_threads=THREADS)
    _check(got, ref, f"rising logits, ragged batch, d {d}")
    _check_lse(lse, ref_lse, f"rising logits, ragged batch, d {d}")


# ------------------------------------------------------------------ a dominant late key

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_dominant_late_key_prefill(d, causal):
    """Key 990 of 1000 (the last of 8 blocks) dominates every row that sees it."""
    N, key = 1000, 990
    q, k, v = inputs.prefill_inputs(1, 6, 2, N, N, d, torch.bfloat16, seed=220 + d)
    mask = torch.zeros(1, 1, N, 1, dtype=torch.bool)
    mask[:, :, key] = True
    q, k = inputs.with_dominant_keys(q, k, mask, level=256.0)
    got, lse, plain = _fwd_lse(q, k, v, causal, d ** -0.5)
    ref, ref_lse = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check(got, ref, f"dominant key d {d} causal {causal}")
    _check(plain, ref, f"dominant key d {d} causal {causal}, plain entry point")
    _check_lse(lse, ref_lse, f"dominant key d {d} causal {causal}")
    # the rows that see the key return (almost exactly) its V row
    rows = slice(key, N) if causal else slice(0, N)
    vk = v[0, :, key].float().numpy()  # [H_kv, d]
    assert np.abs(got[0, :, rows] - np.repeat(vk, 3, axis=0)[:, None, :]).max() <= BF16_MAX


@pytest.mark.parametrize("d", [64, 128])
def test_dominant_late_key_varlen(d):
    lens = [900, 300, 129]
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens, lens, 8, 4, d, torch.bfloat16, seed=230 + d)
    mask = torch.zeros(k.shape[0], 1, 1, dtype=torch.bool)
    for b in range(len(lens)):
        mask[int(cu_k[b + 1]) - 3] = True  # third-last key of every sequence
    q, k = inputs.with_dominant_keys(q, k, mask)
    got, lse = _varlen_lse(q, k, v, cu_q, cu_k, True, d ** -0.5)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, d ** -0.5,
                                         n_threads=THREADS)
    _check(got, ref, f"dominant key, ragged batch, d {d}")
    _check_lse(lse, ref_lse, f"dominant key, ragged batch, d {d}")


@pytest.mark.parametrize("d", [64, 128])
def test_dominant_late_key_decode(d):
    """Decode with the last valid cache row of every sequence dominant: in a
    split plane it sits in the last part, whose maximum then wins the merge."""
    seqlens, q, kc, vc = inputs.decode_inputs(8, 12, 2, 2048, d, torch.bfloat16, seed=240 + d,
                                              seqlens=[2048, 1, 700, 64, 65, 1999, 1024, 130])
    pos = torch.arange(2048).view(1, 1, 2048, 1)
    mask = pos == (seqlens.view(8, 1, 1, 1).long() - 1)
    q, kc = inputs.with_dominant_keys(q, kc, mask)
    qd, kd, vd, sd = (t.cuda() for t in (q, kc, vc, seqlens))
    o = torch.full_like(qd, float("nan"))
    o, lse = ops.gqa_attn_decode_lse(qd, kd, vd, sd, o, scale=d ** -0.5)
    o64 = ops.gqa_attn_decode(qd, kd, vd, sd, scale=d ** -0.5, chunk_tokens=64)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, ref_lse = oracle.decode(q, kc, vc, seqlens, d ** -0.5)
    _check(o.float().cpu().numpy(), ref, f"decode, dominant last key, d {d}")
    _check(o64.float().cpu().numpy(), ref, f"decode, dominant last key, 64-row splits, d {d}")
    _check_lse(lse.cpu().numpy(), ref_lse, f"decode, dominant last key, d {d}")


# ------------------------------------------------------------------ scaled queries

@pytest.mark.parametrize("mul", [4, 8, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_scaled_queries_prefill(d, mul):
    """q times 4, 8, 16 (exact in bf16): score spreads of tens of log2 units."""
    q, k, v = inputs.prefill_inputs(1, 8, 2, 1024, 1024, d, torch.bfloat16, seed=250 + d + mul)
    q = (q.float() * mul).to(torch.bfloat16)
    got, lse, plain = _fwd_lse(q, k, v, True, d ** -0.5)
    ref, ref_lse = oracle.prefill(q, k, v, True, d ** -0.5, n_threads=THREADS)
    _check(got, ref, f"q x{mul} d {d}")
    _check(plain, ref, f"q x{mul} d {d}, plain entry point")
    _check_lse(lse, ref_lse, f"q x{mul} d {d}")


@pytest.mark.parametrize("mul", [4, 16])
def test_scaled_queries_varlen(mul):
    lens_q, lens_k = [700, 200, 5], [700, 333, 5]
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, 8, 2, 128, torch.bfloat16,
                                               seed=260 + mul)
    q = (q.float() * mul).to(torch.bfloat16)
    got, lse = _varlen_lse(q, k, v, cu_q, cu_k, True, 128 ** -0.5)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, 128 ** -0.5,
                                         n_threads=THREADS)
    _check(got, ref, f"ragged batch, q x{mul}")
    _check_lse(lse, ref_lse, f"ragged batch, q x{mul}")


# ------------------------------------------------------------------ zero and negative scales

@pytest.mark.parametrize("scale", [0.0, -0.09])
@pytest.mark.parametrize("d", [64, 128])
def test_zero_and_negative_scale(d, scale):
    """scale = 0 gives the mean of the visible V rows; a negative scale
    reverses the order of the scores. Causal with a ragged tail, so masked
    keys meet the scale in both cases."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 300, 300, d, torch.bfloat16, seed=270 + d)
    got, lse, plain = _fwd_lse(q, k, v, True, scale)
    ref, ref_lse = oracle.prefill(q, k, v, True, scale)
    _check(got, ref, f"prefill scale {scale} d {d}")
    _check(plain, ref, f"prefill scale {scale} d {d}, plain entry point")
    _check_lse(lse, ref_lse, f"prefill scale {scale} d {d}")
    lens = [300, 77]
    q2, k2, v2, cu_q, cu_k = inputs.varlen_inputs(lens, lens, 4, 2, d, torch.bfloat16,
                                                  seed=271 + d)
    got, _ = _varlen_lse(q2, k2, v2, cu_q, cu_k, True, scale)
    ref, _ = oracle.prefill_varlen(q2, k2, v2, cu_q, cu_k, True, scale)
    _check(got, ref, f"ragged batch scale {scale} d {d}")
    seqlens, dq, kc, vc = inputs.decode_inputs(4, 8, 2, 300, d, torch.bfloat16, seed=272 + d,
                                               seqlens=[300, 1, 0, 129])
    qd, kd, vd, sd = (t.cuda() for t in (dq, kc, vc, seqlens))
    o = ops.gqa_attn_decode(qd, kd, vd, sd, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.decode(dq, kc, vc, seqlens, scale)
    _check(o.float().cpu().numpy(), ref, f"decode scale {scale} d {d}")
