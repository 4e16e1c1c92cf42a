"""GPU parity for layouts and head dims beyond the packed d = 64 / 128 cases
(microLLM-rocm optimisation log, Experiments 202-206: attention on the
token-major layout without strided copies).

* gqa_attn_fwd_strided on views: q, k, v sliced out of one fused QKV
  buffer [B][N][H_q + 2 H_kv][d], O written into a token-major view, and
  padded row strides; against the oracle and, bit for bit, against
  gqa_attn_fwd on packed copies (the same units, the same arithmetic).
* Head dims 32 and 96 (zero-padded tiles of the 64- and 128-column kernels)
  through the dense, lse, ragged-batch and token-major entry points.
* Head dim 256 (one query tile per CTA: its S and O fill the tensor memory)
  through the dense, lse, strided, ragged-batch and token-major entry
  points, with ragged tile tails, more keys than queries, empty sequences,
  and MHA / GQA / MQA groupings.
* Decode at head dims 32 and 96 (the 64- and 128-column decode kernels on
  zero-padded boxes) and 256 (two MMA warps per row group, a column half
  each), through the plain, lse, chunked and allocation-free entry points,
  with NaN past every sequence and planes split over CTAs.
Bounds: the bf16 ones of the other tests (max abs 2e-2, mean abs 2e-3; lse
max abs 5e-3).
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


def _check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    d = np.abs(got - ref)
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, f"{what}: max {d.max():.3e} mean {d.mean():.3e}"


@pytest.mark.parametrize("shape", [(2, 8, 2, 300, 300, 128, True), (1, 12, 4, 200, 520, 64, True),
                                   (2, 4, 1, 129, 129, 96, False), (1, 8, 8, 256, 256, 32, True)],
                         ids=lambda s: "-".join(map(str, s)))
def test_strided_fused_qkv(shape):
    B, H_q, H_kv, N_q, N_kv, d, causal = shape
    Ht = H_q + 2 * H_kv
    N = max(N_q, N_kv)
    g = torch.Generator("cpu").manual_seed(600 + N_q)
    buf = torch.randn(B, N, Ht, d, generator=g).to(torch.bfloat16).cuda()
    q = buf[:, :N_q, :H_q].transpose(1, 2)                       # [B, H_q, N_q, d] view
    k = buf[:, :N_kv, H_q:H_q + H_kv].transpose(1, 2)
    v = buf[:, :N_kv, H_q + H_kv:].transpose(1, 2)
    o_tok = torch.full((B, N_q, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.gqa_attn_fwd_strided(q, k, v, o_tok.transpose(1, 2), causal=causal, scale=d ** -0.5)
    packed = ops.gqa_attn_fwd(q.contiguous(), k.contiguous(), v.contiguous(), causal=causal,
                              scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    got = o_tok.transpose(1, 2)
    assert torch.equal(got, packed), "strided and packed calls differ"
    ref, _ = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), causal, d ** -0.5, n_threads=THREADS)
    _check(got.float().cpu().numpy(), ref, f"fused QKV {shape}")


def test_strided_padded_rows_and_heads():
    """Row strides above d and gaps between heads and batches; O padded too."""
    B, H_q, H_kv, N, d = 2, 6, 3, 333, 128
    q0, k0, v0 = inputs.prefill_inputs(B, H_q, H_kv, N, N, d, torch.bfloat16, seed=610)

    def padded(t, row_pad, head_gap, batch_gap):
        b, h, n, dd = t.shape
        big = torch.full((b, h, n + head_gap, dd + row_pad), float("nan"), dtype=t.dtype)
        big = torch.cat([big, torch.full((b, 1, n + head_gap, dd + row_pad), float("nan"),
                                         dtype=t.dtype)], 1) if batch_gap else big
        big = big.cuda()
        view = big[:, :h, :n, :dd]
        view.copy_(t.cuda())
        return view

    q = padded(q0, 8, 3, True)
    k = padded(k0, 64, 0, False)
    v = padded(v0, 16, 5, True)
    o_big = torch.full((B, H_q, N, d + 24), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = o_big[..., :d]
    ops.gqa_attn_fwd_strided(q, k, v, o, causal=True, scale=0.09)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    assert torch.isnan(o_big[..., d:].float()).all(), "columns past d were written"
    ref, _ = oracle.prefill(q0, k0, v0, True, 0.09, n_threads=THREADS)
    _check(o.float().cpu().numpy(), ref, "padded strides")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [32, 96])
def test_head_dims_32_96_dense_and_lse(d, causal):
    q, k, v = inputs.prefill_inputs(2, 8, 2, 300, 300, d, torch.bfloat16, seed=620 + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd(qd, kd, vd, o, causal=causal, scale=d ** -0.5)
    o2, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, ref_lse = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check(o.float().cpu().numpy(), ref, f"d {d}")
    _check(o2.float().cpu().numpy(), ref, f"d {d} lse kernel")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_MAX


@pytest.mark.parametrize("d", [32, 96])
def test_head_dims_32_96_ragged_and_token_major(d):
    lens_q, lens_k = [300, 1, 129], [400, 1, 129]
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, 8, 2, d, torch.bfloat16, seed=630 + d)
    qd, kd, vd, cqd, ckd = (t.cuda() for t in (q, k, v, cu_q, cu_k))
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, o, causal=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill_varlen(q, k, v, cu_q, cu_k, True, d ** -0.5)
    _check(o.float().cpu().numpy(), ref, f"ragged batch d {d}")
    q, k, v = inputs.prefill_inputs(2, 8, 4, 200, 200, d, torch.bfloat16, seed=640 + d)
    tok = lambda t: t.transpose(1, 2).contiguous()
    ob = ops.gqa_attn_fwd_bshd(tok(q).cuda(), tok(k).cuda(), tok(v).cuda(), causal=False,
                               scale=d ** -0.5)
    torch.cuda.synchronize()
    ref, _ = oracle.prefill(q, k, v, False, d ** -0.5, n_threads=THREADS)
    _check(ob.transpose(1, 2).float().cpu().numpy(), ref, f"token-major d {d}")


@pytest.mark.parametrize("shape", [(2, 8, 2, 300, 300, True), (1, 4, 4, 200, 520, True),
                                   (2, 6, 1, 129, 129, False), (1, 16, 4, 640, 640, True)],
                         ids=lambda s: "-".join(map(str, s)))
def test_head_dim_256_dense_and_lse(shape):
    B, H_q, H_kv, N_q, N_kv, causal = shape
    d = 256
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=650 + N_q)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd(qd, kd, vd, o, causal=causal, scale=d ** -0.5)
    o2, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, ref_lse = oracle.prefill(q, k, v, causal, d ** -0.5, n_threads=THREADS)
    _check(o.float().cpu().numpy(), ref, f"d 256 {shape}")
    _check(o2.float().cpu().numpy(), ref, f"d 256 {shape} lse kernel")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_MAX


def test_head_dim_256_strided_fused_qkv():
    B, H_q, H_kv, N, d = 2, 4, 2, 200, 256
    Ht = H_q + 2 * H_kv
    g = torch.Generator("cpu").manual_seed(660)
    buf = torch.randn(B, N, Ht, d, generator=g).to(torch.bfloat16).cuda()
    q = buf[:, :, :H_q].transpose(1, 2)
    k = buf[:, :, H_q:H_q + H_kv].transpose(1, 2)
    v = buf[:, :, H_q + H_kv:].transpose(1, 2)
    o_tok = torch.full((B, N, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.gqa_attn_fwd_strided(q, k, v, o_tok.transpose(1, 2), causal=True, scale=d ** -0.5)
    packed = ops.gqa_attn_fwd(q.contiguous(), k.contiguous(), v.contiguous(), causal=True,
                              scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    assert torch.equal(o_tok.transpose(1, 2), packed), "strided and packed calls differ"
    ref, _ = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), True, d ** -0.5, n_threads=THREADS)
    _check(packed.float().cpu().numpy(), ref, "d 256 fused QKV")


@pytest.mark.parametrize("case", [([300, 1, 129, 77], [400, 1, 129, 200], 8, 2, True),
                                  ([500, 37], [20, 700], 4, 1, False),
                                  ([0, 130, 0, 5], [0, 130, 10, 5], 4, 4, True)],
                         ids=lambda c: "-".join(map(str, c[0])))
def test_head_dim_256_ragged(case):
    """Ragged batches at d = 256: one query tile per listed unit; the lse
    and plain kernels give the same O bits, repeated calls too."""
    lens_q, lens_k, H_q, H_kv, causal = case
    d = 256
    q, k, v, cu_q, cu_k = inputs.varlen_inputs(lens_q, lens_k, H_q, H_kv, d, torch.bfloat16,
                                               seed=670 + sum(lens_q))
    qd, kd, vd, cqd, ckd = (t.cuda() for t in (q, k, v, cu_q, cu_k))
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, o, causal=causal, scale=d ** -0.5)
    o2, lse = ops.gqa_attn_fwd_varlen_lse(qd, kd, vd, cqd, ckd, causal=causal, scale=d ** -0.5)
    o3 = ops.gqa_attn_fwd_varlen(qd, kd, vd, cqd, ckd, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, causal, d ** -0.5, n_threads=THREADS)
    _check(o.float().cpu().numpy(), ref, f"ragged d 256 {case}")
    assert torch.equal(o, o2) and torch.equal(o, o3)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_MAX


def test_head_dim_256_token_major():
    B, H_q, H_kv, N_q, N_kv, d = 2, 8, 2, 200, 330, 256
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=680)
    tok = lambda t: t.transpose(1, 2).contiguous()
    ob = ops.gqa_attn_fwd_bshd(tok(q).cuda(), tok(k).cuda(), tok(v).cuda(), causal=True,
                               scale=d ** -0.5)
    od = ops.gqa_attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.prefill(q, k, v, True, d ** -0.5, n_threads=THREADS)
    _check(ob.transpose(1, 2).float().cpu().numpy(), ref, "token-major d 256")
    # the same tiles in the same order of key blocks: the same bits as the dense path
    assert torch.equal(ob.transpose(1, 2), od)


@pytest.mark.parametrize("shape", [(8, 12, 2, 700), (3, 16, 16, 300), (64, 8, 1, 520),
                                   (1, 32, 8, 2048), (2, 16, 2, 4000)],
                         ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("d", [32, 96, 256])
def test_decode_head_dims(d, shape):
    """Decode at head dims 32 and 96 (the 64- and 128-column kernels on
    zero-padded boxes) and 256 (two MMA warps per 16-row group, 128 columns
    each); the last two shapes spread a plane over many CTAs."""
    B, H_q, H_kv, L = shape
    sl, q, kc, vc = inputs.decode_inputs(B, H_q, H_kv, L, d, torch.bfloat16, seed=670 + d + B)
    sld, qd, kcd, vcd = sl.cuda(), q.cuda(), kc.cuda(), vc.cuda()
    scale = d ** -0.5
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_decode(qd, kcd, vcd, sld, o, scale=scale)
    o2, lse = ops.gqa_attn_decode_lse(qd, kcd, vcd, sld, scale=scale)
    o3 = ops.gqa_attn_decode(qd, kcd, vcd, sld, scale=scale, chunk_tokens=128)
    o4 = torch.full_like(qd, float("nan"))
    ops.gqa_attn_decode_noalloc(qd, kcd, vcd, sld, o4, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    assert torch.equal(o, o2), "the lse kernel's O differs from the plain kernel's"
    ref, ref_lse = oracle.decode(q, kc, vc, sl, scale)
    for got, what in ((o, "plain"), (o2, "lse"), (o3, "chunked"), (o4, "no-alloc")):
        _check(got.float().cpu().numpy(), ref, f"decode d {d} {shape} {what}")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_MAX
