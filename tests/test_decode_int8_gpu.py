"""GPU parity of the decode against an int8 K/V cache.

The caches hold one-byte two's-complement codes with a per-K/V-head scale
(microLLM-rocm optimisation log, Experiments 352 and 354: a one-byte tensor
with an explicit scale, widened inside the decode kernel). The oracle
widens every code from its definition, times its head's scale, in float64,
and attends exactly; the kernel widens the codes exactly too (K to bf16, V
to f16), so the comparison carries the bf16 cache's bounds: max abs <= 2e-2,
mean abs <= 2e-3 (lse max abs <= 5e-3). Rows past each sequence hold -128,
a code the quantiser never writes.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

BF16_MAX = 2e-2
BF16_MEAN = 2e-3
LSE_MAX = 5e-3


def _run(sl, q, k8, v8, ks, vs, scale, with_lse=True):
    sd, qd, kd, vd, ksd, vsd = (t.cuda() for t in (sl, q, k8, v8, ks, vs))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    ops.gqa_attn_decode_int8(qd, kd, vd, ksd, vsd, sd, o, lse, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    return o.float().cpu().numpy(), None if lse is None else lse.cpu().numpy()


def _check(got, ref, lse, ref_lse, what):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = np.abs(got.astype(np.float64) - ref)
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, f"{what}: max {d.max():.3e} mean {d.mean():.3e}"
    if lse is not None:
        lse = lse.astype(np.float64)
        assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), what
        m = np.isfinite(ref_lse)
        assert np.abs(lse[m] - ref_lse[m]).max() <= LSE_MAX, what


@pytest.mark.parametrize("shape", inputs.decode_shapes(), ids=lambda s: s.name)
def test_int8_decode_matches_oracle(shape):
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(shape.B, shape.H_q, shape.H_kv, shape.max_len,
                                                      shape.d, seed=shape.seed)
    got, lse = _run(sl, q, k8, v8, ks, vs, shape.scale)
    ref, ref_lse = oracle.decode_int8(q, k8, v8, ks, vs, sl, shape.scale)
    _check(got, ref, lse, ref_lse, shape.name)


@pytest.mark.parametrize("d", [32, 64, 96, 128])
def test_int8_decode_edge_lengths(d):
    """Empty sequences, one row, unit boundaries (128 rows) and a full cache."""
    lens = [0, 1, 127, 128, 129, 255, 256, 700]
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(8, 16, 2, 700, d, seed=600 + d, seqlens=lens)
    got, lse = _run(sl, q, k8, v8, ks, vs, d ** -0.5)
    assert np.all(got[0] == 0) and np.all(np.isneginf(lse[0]))
    ref, ref_lse = oracle.decode_int8(q, k8, v8, ks, vs, sl, d ** -0.5)
    _check(got, ref, lse, ref_lse, f"edge lengths d {d}")


@pytest.mark.parametrize("d", [32, 64, 96, 128])
def test_int8_decode_one_long_sequence_split_over_many_ctas(d):
    """One 20000-row sequence: its plane is cut over many CTAs and merged."""
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(1, 8, 1, 20000, d, seed=610 + d, seqlens=[20000])
    got, lse = _run(sl, q, k8, v8, ks, vs, d ** -0.5)
    ref, ref_lse = oracle.decode_int8(q, k8, v8, ks, vs, sl, d ** -0.5)
    _check(got, ref, lse, ref_lse, f"one long sequence d {d}")


@pytest.mark.parametrize("shape", [(8, 12, 2, 700), (64, 8, 1, 520), (2, 16, 2, 4000)],
                         ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("d", [32, 96])
def test_int8_decode_padded_head_dims(d, shape):
    """Head dims 32 and 96 on the 64- and 128-column kernels; O rows are d
    wide and the guard after the last one stays NaN."""
    B, H_q, H_kv, L = shape
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(B, H_q, H_kv, L, d, seed=620 + d + B)
    sd, qd, kd, vd, ksd, vsd = (t.cuda() for t in (sl, q, k8, v8, ks, vs))
    buf = torch.full((B * H_q * d + 256,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[: B * H_q * d].view(B, H_q, d)
    lse = torch.full((B, H_q), float("nan"), dtype=torch.float32, device="cuda")
    ops.gqa_attn_decode_int8(qd, kd, vd, ksd, vsd, sd, o, lse, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    assert torch.isnan(buf[B * H_q * d:]).all(), "store past the last row"
    ref, ref_lse = oracle.decode_int8(q, k8, v8, ks, vs, sl, d ** -0.5)
    _check(o.float().cpu().numpy(), ref, lse.cpu().numpy(), ref_lse, f"int8 d {d} {shape}")


def test_int8_decode_scales_groups_and_extreme_codes():
    """Different scales per K/V head, a group of 24 query heads (two head
    groups of 16 per K/V head), codes at both ends of the range (-128 and
    127 inside the sequences), no lse output, deterministic."""
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(5, 48, 2, 1500, 128, seed=630,
                                                      seqlens=[1500, 3, 900, 64, 1201])
    g = torch.Generator().manual_seed(631)
    pick = torch.rand(k8.shape, generator=g) < 0.02
    k8 = torch.where(pick, torch.where(torch.rand(k8.shape, generator=g) < 0.5,
                                       torch.tensor(-128, dtype=torch.int8),
                                       torch.tensor(127, dtype=torch.int8)), k8)
    v8 = torch.where(pick.flip(-1), torch.tensor(-128, dtype=torch.int8), v8)
    # (V scales kept at most 1x: the extreme codes pull O to a few units,
    # where bf16's own rounding of O stays within the bounds)
    ks = ks * torch.tensor([0.5, 2.0])
    vs = vs * torch.tensor([1.0, 0.25])
    a, _ = _run(sl, q, k8, v8, ks, vs, 0.09, with_lse=False)
    b, _ = _run(sl, q, k8, v8, ks, vs, 0.09, with_lse=False)
    assert np.array_equal(a, b)
    ref, _ = oracle.decode_int8(q, k8, v8, ks, vs, sl, 0.09)
    _check(a, ref, None, None, "scales, groups and extreme codes")


def test_int8_decode_ignores_rows_past_each_sequence():
    """Other codes in the rows past each sequence give the same bits."""
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(16, 12, 2, 600, 128, seed=640)
    a, la = _run(sl, q, k8, v8, ks, vs, 0.088)
    dead = torch.arange(600).view(1, 1, 600, 1) >= sl.long().view(16, 1, 1, 1)
    k2 = torch.where(dead, torch.full_like(k8, 127), k8)
    v2 = torch.where(dead, torch.full_like(v8, 99), v8)
    b, lb = _run(sl, q, k2, v2, ks, vs, 0.088)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_int8_decode_close_to_bf16_decode_of_the_same_values():
    """The int8 path and the bf16 path on the widened values give the same
    operation: with scales 2^-7 the widened values are exact in bf16."""
    shape = inputs.decode_shapes()[1]
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(shape.B, shape.H_q, shape.H_kv, shape.max_len,
                                                      shape.d, seed=650)
    sc = torch.full((shape.H_kv,), 2.0 ** -7)
    got, _ = _run(sl, q, k8, v8, sc, sc, shape.scale, with_lse=False)
    kb = (k8.to(torch.float32) * 2.0 ** -7).to(torch.bfloat16).cuda()
    vb = (v8.to(torch.float32) * 2.0 ** -7).to(torch.bfloat16).cuda()
    o = ops.gqa_attn_decode(q.cuda(), kb, vb, sl.cuda(), scale=shape.scale)
    torch.cuda.synchronize()
    d = np.abs(got - o.float().cpu().numpy())
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN
