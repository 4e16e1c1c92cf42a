"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (fixed by the method's statement of the target):
  * fp32 path: max abs error <= 2e-5;
  * bf16 path (bf16 inputs, fp32 accumulation, bf16 output): max abs error
    <= 2e-2 and mean abs error <= 2e-3.
The oracle reads the very same bf16/fp32 values, widened exactly to float64.
Small shapes are compared element by element; the full-size prefill layers
are compared on every row of two heads plus 64 random rows of every head.
Every output buffer starts as NaN, so a tile the scheduler never visited
shows up as a non-finite value.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

F32_MAX = 2e-5
BF16_MAX = 2e-2
BF16_MEAN = 2e-3
THREADS = max(1, min(16, os.cpu_count() or 1))


def _dev(*ts):
    return [t.cuda() for t in ts]


def _err(got, ref):
    d = np.abs(got.astype(np.float64) - ref)
    return float(d.max()), float(d.mean())


def _check_bf16(got, ref, what):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx, mean = _err(got, ref)
    assert mx <= BF16_MAX and mean <= BF16_MEAN, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def _prefill_bf16(q, k, v, causal, scale):
    qd, kd, vd = _dev(q, k, v)
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd(qd, kd, vd, o, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    return o.float().cpu().numpy()


# ------------------------------------------------------------------ fp32 path

def test_tiny_gqa_fp32_matches_oracle():
    s = inputs.TINY
    q, k, v = inputs.prefill_inputs_for(s)
    qd, kd, vd = _dev(q, k, v)
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd_f32(qd, kd, vd, o, causal=s.causal, scale=s.scale)
    ref, _ = oracle.prefill(q, k, v, s.causal, s.scale)
    mx, _ = _err(o.cpu().numpy(), ref)
    assert mx <= F32_MAX, mx


@pytest.mark.parametrize("shape", [
    (2, 8, 2, 77, 77, 32, True), (1, 4, 1, 200, 333, 96, False), (1, 6, 6, 130, 130, 128, True),
    (2, 4, 2, 1, 45, 64, False), (1, 2, 1, 64, 300, 64, True)])
def test_fp32_prefill_shapes(shape):
    B, H_q, H_kv, N_q, N_kv, d, causal = shape
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.float32, seed=31 + d)
    qd, kd, vd = _dev(q, k, v)
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd_f32(qd, kd, vd, o, causal=causal, scale=d ** -0.5)
    ref, _ = oracle.prefill(q, k, v, causal, d ** -0.5)
    mx, _ = _err(o.cpu().numpy(), ref)
    assert mx <= F32_MAX, mx


def test_fp32_decode_matches_oracle():
    seqlens, q, kc, vc = inputs.decode_inputs(8, 12, 2, 300, 128, torch.float32, seed=41,
                                              seqlens=[0, 300, 1, 17, 128, 129, 250, 299])
    qd, kd, vd, sd = _dev(q, kc, vc, seqlens)
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_decode_f32(qd, kd, vd, sd, o, scale=128 ** -0.5)
    ref, _ = oracle.decode(q, kc, vc, seqlens, 128 ** -0.5)
    mx, _ = _err(o.cpu().numpy(), ref)
    assert mx <= F32_MAX, mx


# ------------------------------------------------------------------ bf16 prefill

SMALL_BF16 = [
    # B, H_q, H_kv, N_q, N_kv, d, causal
    (1, 4, 2, 128, 128, 64, False),
    (1, 4, 2, 300, 300, 64, True),      # ragged tail, several tiles
    (2, 6, 2, 200, 520, 128, True),     # N_q < N_kv bottom-right, odd group 3
    (1, 8, 8, 384, 384, 128, True),     # MHA
    (1, 8, 1, 256, 700, 64, False),     # MQA, ragged K/V
    (2, 2, 1, 1, 129, 128, False),      # single query row
    (1, 3, 3, 129, 129, 64, True),      # odd tile count: half-empty last unit
    (1, 2, 2, 640, 640, 128, False),    # 5 K/V blocks through a 4-stage ring
]


@pytest.mark.parametrize("shape", SMALL_BF16)
def test_bf16_prefill_small_shapes(shape):
    B, H_q, H_kv, N_q, N_kv, d, causal = shape
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=51 + N_q)
    got = _prefill_bf16(q, k, v, causal, d ** -0.5)
    ref, _ = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check_bf16(got, ref, str(shape))


@pytest.mark.parametrize("shape", inputs.sweep_shapes(), ids=lambda s: s.name)
def test_bf16_sweep_mha_gqa_mqa(shape):
    q, k, v = inputs.prefill_inputs_for(shape)
    got = _prefill_bf16(q, k, v, shape.causal, shape.scale)
    ref, _ = oracle.prefill(q, k, v, shape.causal, shape.scale, n_threads=THREADS)
    _check_bf16(got, ref, shape.name)


def _sampled_rows_check(shape):
    q, k, v = inputs.prefill_inputs_for(shape)
    got = _prefill_bf16(q, k, v, shape.causal, shape.scale)
    assert np.isfinite(got).all(), "a tile was never written"
    B, H_q, N = shape.B, shape.H_q, shape.N_q
    # every row of two heads: the first and the last (b, h_q)
    for bh in (0, B * H_q - 1):
        ref, _ = oracle.prefill(q, k, v, shape.causal, shape.scale, heads=(bh, bh + 1),
                                n_threads=THREADS)
        b, h = divmod(bh, H_q)
        _check_bf16(got[b, h], ref[b, h], f"{shape.name} head {bh}")
    # 64 random rows of every head
    rng = np.random.default_rng(shape.seed)
    rows = [(b, h, int(i)) for b in range(B) for h in range(H_q)
            for i in rng.choice(N, 64, replace=False)]
    ref, _ = oracle.prefill_rows(q, k, v, shape.causal, shape.scale, rows)
    sel = np.stack([got[b, h, i] for (b, h, i) in rows])
    _check_bf16(sel, ref, f"{shape.name} sampled rows")


def test_bf16_llama3_8b_layer_sampled():
    _sampled_rows_check(inputs.LLAMA3_8B_LAYER)


def test_bf16_long_sequence_sampled():
    _sampled_rows_check(inputs.LONG_SEQ)


def test_bf16_prefill_deterministic():
    s = inputs.LLAMA3_8B_LAYER
    q, k, v = _dev(*inputs.prefill_inputs_for(s))
    o1 = ops.gqa_attn_fwd(q, k, v, causal=True, scale=s.scale)
    o2 = ops.gqa_attn_fwd(q, k, v, causal=True, scale=s.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_prefill_output_only_16_byte_aligned(d):
    """O at a 16- but not 32-byte aligned address takes the 16-byte store
    path and gives the same bits as an aligned O."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 320, 320, d, torch.bfloat16, seed=77 + d)
    qd, kd, vd = _dev(q, k, v)
    o_al = ops.gqa_attn_fwd(qd, kd, vd, causal=True, scale=d ** -0.5)
    flat = torch.full((qd.numel() + 8,), float("nan"), dtype=torch.bfloat16, device=qd.device)
    o_off = flat[8:].view(qd.shape)  # 16 bytes past a 256-byte aligned allocation
    assert o_off.data_ptr() % 32 == 16
    ops.gqa_attn_fwd(qd, kd, vd, o_off, causal=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    assert torch.equal(o_al, o_off)
    ref, _ = oracle.prefill(q, k, v, True, d ** -0.5)
    _check_bf16(o_off.float().cpu().numpy(), ref, f"16-byte aligned O, d {d}")


def test_bf16_prefill_repeated_launches_rearm_scheduler():
    """The work counter re-arms itself: many back-to-back launches stay correct."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 300, 300, 64, torch.bfloat16, seed=61)
    qd, kd, vd = _dev(q, k, v)
    ref, _ = oracle.prefill(q, k, v, True, 0.125)
    outs = [ops.gqa_attn_fwd(qd, kd, vd, causal=True, scale=0.125) for _ in range(20)]
    torch.cuda.synchronize()
    for o in outs:
        _check_bf16(o.float().cpu().numpy(), ref, "repeat")


# ------------------------------------------------------------------ bf16 decode

def _decode_run(seqlens, q, kc, vc, scale, chunk=0):
    qd, kd, vd, sd = _dev(q, kc, vc, seqlens)
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_decode(qd, kd, vd, sd, o, scale=scale, chunk_tokens=chunk)
    torch.cuda.synchronize()
    return o.float().cpu().numpy()


@pytest.mark.parametrize("shape", inputs.decode_shapes(), ids=lambda s: s.name)
def test_bf16_decode_matches_oracle(shape):
    seqlens, q, kc, vc = inputs.decode_inputs_for(shape)
    got = _decode_run(seqlens, q, kc, vc, shape.scale)
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.decode(q, kc, vc, seqlens, shape.scale)
    _check_bf16(got, ref, shape.name)


@pytest.mark.parametrize("chunk", [64, 128, 256, 512])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_decode_split_invariance(chunk, d):
    """Every split size gives the same operation (microLLM-rocm Exp 282-284)."""
    seqlens, q, kc, vc = inputs.decode_inputs(5, 8, 2, 700, d, torch.bfloat16, seed=71 + d,
                                              seqlens=[1, 700, 255, 256, 513])
    ref, _ = oracle.decode(q, kc, vc, seqlens, d ** -0.5)
    got = _decode_run(seqlens, q, kc, vc, d ** -0.5, chunk)
    _check_bf16(got, ref, f"chunk {chunk} d {d}")


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_decode_plane_split_over_many_ctas(d):
    """One long sequence cut into 64-row splits: each (K/V head, head group)
    spreads over ~150 CTAs, so the log-sum-exp merge takes its parts in
    several chunks. Also a 40-part case next to short sequences."""
    seqlens, q, kc, vc = inputs.decode_inputs(1, 8, 1, 40000, d, torch.bfloat16, seed=95 + d,
                                              seqlens=[40000])
    ref, _ = oracle.decode(q, kc, vc, seqlens, d ** -0.5)
    got = _decode_run(seqlens, q, kc, vc, d ** -0.5, 64)
    assert ops.gqa_attn_get_device_error() == 0
    _check_bf16(got, ref, f"one long sequence d {d}")
    seqlens, q, kc, vc = inputs.decode_inputs(3, 20, 2, 10240, d, torch.bfloat16, seed=97 + d,
                                              seqlens=[10240, 3, 9000])
    ref, _ = oracle.decode(q, kc, vc, seqlens, d ** -0.5)
    got = _decode_run(seqlens, q, kc, vc, d ** -0.5, 64)
    _check_bf16(got, ref, f"long and short sequences d {d}")


@pytest.mark.parametrize("B", [200, 1100])
def test_bf16_decode_large_batch(B):
    """More sequences than one warp pass of the start search (128) and than
    the lengths kept in shared memory (1024); some sequences are empty."""
    seqlens, q, kc, vc = inputs.decode_inputs(B, 4, 1, 96, 64, torch.bfloat16, seed=99 + B)
    seqlens[::7] = 0
    got = _decode_run(seqlens, q, kc, vc, 0.125)
    assert ops.gqa_attn_get_device_error() == 0
    assert np.all(got[::7] == 0)
    ref, _ = oracle.decode(q, kc, vc, seqlens, 0.125)
    _check_bf16(got, ref, f"B={B}")


def test_bf16_decode_edge_lengths():
    seqlens, q, kc, vc = inputs.decode_inputs(4, 16, 1, 512, 128, torch.bfloat16, seed=81,
                                              seqlens=[0, 512, 1, 2])
    got = _decode_run(seqlens, q, kc, vc, 0.1)
    assert np.all(got[0] == 0), "an empty sequence must give O = 0"
    ref, _ = oracle.decode(q, kc, vc, seqlens, 0.1)
    _check_bf16(got, ref, "edge lengths")
    assert ops.gqa_attn_get_device_error() == 0


def test_bf16_decode_bad_seqlen_is_reported():
    seqlens, q, kc, vc = inputs.decode_inputs(2, 4, 2, 64, 64, torch.bfloat16, seed=82,
                                              seqlens=[10, 64])
    bad = torch.tensor([10, 65], dtype=torch.int32)  # 65 > max_len
    got = _decode_run(bad, q, kc, vc, 0.125)
    assert ops.gqa_attn_get_device_error() == 6      # GQA_ERR_BAD_SEQLEN
    assert ops.gqa_attn_get_device_error() == 0      # reading clears it
    # the valid sequence is still right, the invalid one is zero
    assert np.all(got[1] == 0)
    ref, _ = oracle.decode(q[:1], kc[:1], vc[:1], seqlens[:1], 0.125)
    _check_bf16(got[:1], ref, "valid sequence next to an invalid one")


def test_decode_equals_last_row_of_causal_prefill():
    """Decode at length L == last row of causal prefill with N_q = N_kv = L."""
    L, d = 333, 128
    q, k, v = inputs.prefill_inputs(1, 12, 2, L, L, d, torch.bfloat16, seed=91)
    pre = _prefill_bf16(q, k, v, True, d ** -0.5)
    seqlens = torch.tensor([L], dtype=torch.int32)
    dec = _decode_run(seqlens, q[:, :, L - 1].contiguous(), k, v, d ** -0.5)
    mx, _ = _err(dec[0], pre[0, :, L - 1].astype(np.float64))
    assert mx <= 2 * BF16_MAX


def test_bf16_decode_deterministic():
    s = inputs.decode_shapes()[-1]
    seqlens, q, kc, vc = inputs.decode_inputs_for(s)
    a = _decode_run(seqlens, q, kc, vc, s.scale)
    b = _decode_run(seqlens, q, kc, vc, s.scale)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ log-sum-exp output

# The lse kernels sum fp32 exponentials of fp32 scores, so the lse error is
# fp32 rounding of the scores and the sum; the bound 5e-3 (natural-log
# units) also covers a sum of bf16-rounded weights (up to 2^-8 relative
# error each).
LSE_MAX = 5e-3


def _plain_o_matches(o, o_plain, d, ref, what):
    """The plain entry point's O: the same bits as the lse kernel's (the same
    arithmetic; the lse instantiation only adds the lse store), and within
    the bf16 bounds of the oracle."""
    assert torch.equal(o, o_plain), what
    _check_bf16(o_plain.float().cpu().numpy(), ref, what)


@pytest.mark.parametrize("d,causal,N", [(128, True, 640), (64, False, 384), (64, True, 1000)])
def test_bf16_prefill_lse_matches_oracle(d, causal, N):
    q, k, v = inputs.prefill_inputs(2, 8, 2, N, N, d, torch.bfloat16, seed=120 + d + N)
    qd, kd, vd = _dev(q, k, v)
    o, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref_o, ref_lse = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check_bf16(o.float().cpu().numpy(), ref_o, "o with lse")
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max()
    assert err <= LSE_MAX, f"lse max err {err:.3e}"
    _plain_o_matches(o, ops.gqa_attn_fwd(qd, kd, vd, causal=causal, scale=d ** -0.5), d, ref_o,
                     "the plain entry point")


@pytest.mark.parametrize("case", ["mixed", "one_long"])
def test_bf16_decode_lse_matches_oracle(case):
    """Whole-plane runs, planes split over several CTAs (merged in-kernel)
    and an empty sequence (lse = -inf)."""
    if case == "mixed":
        seqlens, q, kc, vc = inputs.decode_inputs(6, 24, 2, 1500, 128, torch.bfloat16, seed=130,
                                                  seqlens=[1500, 0, 7, 900, 64, 1201])
    else:
        seqlens, q, kc, vc = inputs.decode_inputs(1, 8, 1, 20000, 64, torch.bfloat16, seed=131,
                                                  seqlens=[20000])
    qd, kd, vd, sd = _dev(q, kc, vc, seqlens)
    o, lse = ops.gqa_attn_decode_lse(qd, kd, vd, sd, scale=0.09)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref_o, ref_lse = oracle.decode(q, kc, vc, seqlens, 0.09)
    _check_bf16(o.float().cpu().numpy(), ref_o, f"decode with lse ({case})")
    got = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref_lse))
    mask = np.isfinite(ref_lse)
    assert np.abs(got[mask] - ref_lse[mask]).max() <= LSE_MAX
    # the plain entry point gives the same O
    assert torch.equal(o, ops.gqa_attn_decode(qd, kd, vd, sd, scale=0.09))


# ------------------------------------------------------------------ launch order

def test_dependent_launches_back_to_back():
    """Kernels may start while the previous grid of the stream finishes
    (programmatic launch); one that reads the previous kernel's output, queued
    right behind it with no synchronisation, must still see all of it."""
    q, k, v = _dev(*inputs.prefill_inputs(1, 8, 2, 640, 640, 128, torch.bfloat16, seed=111))
    o1 = ops.gqa_attn_fwd(q, k, v, causal=True, scale=0.09)
    o2 = ops.gqa_attn_fwd(o1, k, v, causal=True, scale=0.09)   # reads o1 at once
    torch.cuda.synchronize()
    r1 = ops.gqa_attn_fwd(q, k, v, causal=True, scale=0.09)
    torch.cuda.synchronize()
    r2 = ops.gqa_attn_fwd(r1, k, v, causal=True, scale=0.09)
    torch.cuda.synchronize()
    assert torch.equal(o2, r2)

    seqlens, dq, kc, vc = _dev(*inputs.decode_inputs(16, 12, 2, 1024, 128, torch.bfloat16, seed=112))
    a = dq * 1.0                                                  # a PyTorch kernel writes the query
    d1 = ops.gqa_attn_decode(a, kc, vc, seqlens, scale=0.09)
    d2 = ops.gqa_attn_decode(d1, kc, vc, seqlens, scale=0.09)     # reads d1 at once
    torch.cuda.synchronize()
    e1 = ops.gqa_attn_decode(dq, kc, vc, seqlens, scale=0.09)
    torch.cuda.synchronize()
    e2 = ops.gqa_attn_decode(e1, kc, vc, seqlens, scale=0.09)
    torch.cuda.synchronize()
    assert torch.equal(d1, e1) and torch.equal(d2, e2)
    assert ops.gqa_attn_get_device_error() == 0


# ------------------------------------------------------------------ failure detection

# ------------------------------------------------------------------ ragged batches

VARLEN_SMALL = [
    # lens_q, lens_k (None: = lens_q), H_q, H_kv, d, causal
    ([300, 1, 128, 129, 77], None, 8, 2, 128, True),   # ragged tails, a one-row sequence
    ([64, 200, 1], [164, 500, 128], 12, 4, 64, True),  # prefill after a cached prefix, g = 3
    ([500, 37], [20, 700], 4, 1, 128, False),          # MQA, fewer / more keys than queries
    ([0, 130, 0, 5], [0, 130, 10, 5], 8, 8, 64, True), # MHA, empty sequences
    ([1000, 257], None, 16, 2, 128, True),             # g = 8, several K/V blocks
]


def _varlen_run(q, k, v, cu_q, cu_k, causal, scale, o=None):
    qd, kd, vd, cqd, ckd = _dev(q, k, v, cu_q, cu_k)
    if o is None:
        o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, o, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy()


@pytest.mark.parametrize("case", VARLEN_SMALL, ids=lambda c: "-".join(map(str, c[0])))
def test_bf16_varlen_matches_oracle(case):
    lens_q, lens_k, H_q, H_kv, d, causal = case
    lens_k = lens_k or lens_q
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, H_q, H_kv, d, torch.bfloat16,
                                               seed=140 + sum(lens_q))
    got = _varlen_run(q, k, v, cu_q, cu_k, causal, d ** -0.5)
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill_varlen(q, k, v, cu_q, cu_k, causal, d ** -0.5, n_threads=THREADS)
    _check_bf16(got, ref, f"varlen {case}")


def test_bf16_varlen_batch_sampled():
    """The eight-prompt LLaMA-3-8B-headed batch: one whole sequence, the first
    and last token of every sequence in every head, and 256 random rows."""
    s = inputs.varlen_batch_shape()
    q, k, v, cu_q, cu_k = inputs.varlen_inputs_for(s)
    got = _varlen_run(q, k, v, cu_q, cu_k, s.causal, s.scale)
    assert ops.gqa_attn_get_device_error() == 0
    assert np.isfinite(got).all(), "a tile was never written"
    b = int(np.argmin(s.lens_q))  # the shortest sequence, every row of every head
    q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
    ref, _ = oracle.prefill_varlen(q[q0:q1], k[k0:k1], v[k0:k1], [0, q1 - q0], [0, k1 - k0],
                                   s.causal, s.scale, n_threads=THREADS)
    _check_bf16(got[q0:q1], ref, "varlen batch, whole sequence")
    rng = np.random.default_rng(s.seed)
    ends = [int(t) for t in cu_q[:-1]] + [int(t) - 1 for t in cu_q[1:]]
    rows = [(t, h) for t in ends for h in range(s.H_q)]
    rows += [(int(t), int(h)) for t, h in zip(rng.integers(0, int(cu_q[-1]), 256),
                                              rng.integers(0, s.H_q, 256))]
    ref, _ = oracle.prefill_varlen_rows(q, k, v, cu_q, cu_k, s.causal, s.scale, rows)
    _check_bf16(np.stack([got[t, h] for t, h in rows]), ref, "varlen batch, sampled rows")


def test_bf16_varlen_many_short_sequences():
    """300 prompts of 0-200 tokens after cached prefixes of 0-64 keys: many
    one-tile sequences in one unit list."""
    lens_q = inputs.varlen_lengths(300, 0, 200, seed=152)
    extra = inputs.varlen_lengths(300, 0, 64, seed=153)
    lens_k = [lq + e if lq + e > 0 else 1 for lq, e in zip(lens_q, extra)]
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, 8, 2, 64, torch.bfloat16, seed=154)
    got = _varlen_run(q, k, v, cu_q, cu_k, True, 0.125)
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, 0.125)
    _check_bf16(got, ref, "300 short sequences")


def test_bf16_varlen_most_sequences():
    """4096 sequences (the per-call limit): one-token prompts over 1-3 keys,
    plus a 300-token prompt in the middle."""
    lens_q = [1] * 4096
    lens_q[2000] = 300
    lens_k = [1 + (b % 3) for b in range(4096)]
    lens_k[2000] = 300
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, 4, 1, 64, torch.bfloat16, seed=155)
    got = _varlen_run(q, k, v, cu_q, cu_k, True, 0.125)
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, 0.125)
    _check_bf16(got, ref, "4096 sequences")


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_varlen_lse_and_determinism(d):
    q, k, v, cu_q, cu_k = inputs.varlen_inputs([300, 1, 129], [400, 1, 129], 8, 2, d,
                                               torch.bfloat16, seed=150 + d)
    qd, kd, vd, cqd, ckd = _dev(q, k, v, cu_q, cu_k)
    o, lse = ops.gqa_attn_fwd_varlen_lse(qd, kd, vd, cqd, ckd, causal=True, scale=0.09)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref_o, ref_lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, 0.09)
    _check_bf16(o.float().cpu().numpy(), ref_o, "varlen with lse")
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max()
    assert err <= LSE_MAX, f"lse max err {err:.3e}"
    o2 = ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, causal=True, scale=0.09)
    o3 = ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, causal=True, scale=0.09)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3)
    _plain_o_matches(o, o2, d, ref_o, "the plain ragged-batch entry point")


def test_bf16_varlen_bad_offsets_reported_and_skipped():
    """Sequence 2 has fewer keys than queries under the causal mask: the device
    records GQA_ERR_BAD_SEQLEN and leaves its rows alone; the others are right."""
    q, k, v, cu_q, cu_k = inputs.varlen_inputs([130, 50, 60], [130, 50, 40], 4, 2, 64,
                                               torch.bfloat16, seed=151)
    got = _varlen_run(q, k, v, cu_q, cu_k, True, 0.125)
    assert ops.gqa_attn_get_device_error() == 6  # GQA_ERR_BAD_SEQLEN
    assert np.isnan(got[180:]).all()
    ref, _ = oracle.prefill_varlen(q[:180], k[:180], v[:180], cu_q[:3], cu_k[:3], True, 0.125)
    _check_bf16(got[:180], ref, "valid sequences next to a bad one")
    # the context is still usable
    got = _varlen_run(q[:180], k[:180], v[:180], cu_q[:3], cu_k[:3], True, 0.125)
    assert ops.gqa_attn_get_device_error() == 0
    _check_bf16(got, ref, "after a bad call")


@pytest.mark.parametrize("shape", [(2, 8, 2, 300, 300, 128, True), (3, 4, 1, 77, 500, 64, False),
                                   (1, 6, 3, 129, 256, 128, True)])
def test_bf16_bshd_matches_oracle_and_bhsd(shape):
    """[B][N][H][d] batches: against the oracle, and bit for bit against the
    [B][H][N][d] path on the same values (each row's arithmetic is the same)."""
    B, H_q, H_kv, N_q, N_kv, d, causal = shape
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=160 + N_q)
    qd, kd, vd = _dev(q, k, v)
    tok = lambda t: t.transpose(1, 2).contiguous()  # [B][H][N][d] -> [B][N][H][d]
    o = torch.full_like(tok(qd), float("nan"))
    ops.gqa_attn_fwd_bshd(tok(qd), tok(kd), tok(vd), o, causal=causal, scale=d ** -0.5)
    o_bhsd = ops.gqa_attn_fwd(qd, kd, vd, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check_bf16(o.transpose(1, 2).float().cpu().numpy(), ref, f"bshd {shape}")
    assert torch.equal(o.transpose(1, 2), o_bhsd)


def test_bounded_wait_reports_timeout_and_context_survives():
    assert ops.gqa_attn_selftest_wait_timeout(2000) == 4  # GQA_ERR_DEVICE_TIMEOUT
    assert ops.gqa_attn_get_device_error() == 0           # the word was cleared
    # the context is still usable
    q, k, v = inputs.prefill_inputs(1, 2, 1, 128, 128, 64, torch.bfloat16, seed=99)
    got = _prefill_bf16(q, k, v, False, 0.125)
    ref, _ = oracle.prefill(q, k, v, False, 0.125)
    _check_bf16(got, ref, "after timeout")
