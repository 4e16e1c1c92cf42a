"""The decode entry point that allocates nothing (GPU).

Some callers cannot let a library call cudaMalloc: a serving loop held to a
pre-reserved memory budget, a latency-critical path where an allocation may
synchronise the device, a process whose device memory another allocator
owns. gqa_attn_decode_noalloc serves them from a fixed scratch array in the
library's device memory. Through the C ABI, this file checks two calls in a
row against the float64 oracle (within the bf16 bounds the other tests use)
and against the regular gqa_attn_decode, including a batch whose partials
only fit the fixed scratch after the grid is trimmed. It is collected last,
so a run that stops at the first failure has run every other test; it also
passes when run on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

BF16_MAX = 2e-2
BF16_MEAN = 2e-3


def _err(got, ref):
    d = np.abs(got.float().cpu().numpy().astype(np.float64) - ref)
    return float(d.max()), float(d.mean())


def _two_calls_against_oracle_and_regular(seqlens, q, kc, vc, scale):
    ref, _ = oracle.decode(q, kc, vc, seqlens, scale)
    sd, qd, kd, vd = (t.cuda() for t in (seqlens, q, kc, vc))
    o1 = torch.full_like(qd, float("nan"))
    o2 = torch.full_like(qd, float("nan"))
    # two calls in a row share the scratch; each must be right on its own
    ops.gqa_attn_decode_noalloc(qd, kd, vd, sd, o1, scale=scale)
    ops.gqa_attn_decode_noalloc(qd, kd, vd, sd, o2, scale=scale)
    regular = ops.gqa_attn_decode(qd, kd, vd, sd, scale=scale)
    torch.cuda.synchronize()
    for o in (o1, o2):
        assert torch.isfinite(o.float()).all()
        mx, mean = _err(o, ref)
        assert mx <= BF16_MAX and mean <= BF16_MEAN, ("against the oracle", mx, mean)
        mx, mean = _err(o, regular.float().cpu().numpy().astype(np.float64))
        assert mx <= BF16_MAX and mean <= BF16_MEAN, ("against gqa_attn_decode", mx, mean)


@pytest.mark.parametrize("shape", [inputs.decode_shapes()[1], inputs.decode_shapes()[2]],
                         ids=lambda s: s.name)
def test_noalloc_decode_matches_oracle_and_regular_entry_point_twice(shape):
    _two_calls_against_oracle_and_regular(*inputs.decode_inputs_for(shape), shape.scale)


def test_noalloc_decode_with_the_grid_trimmed_to_fit_the_scratch():
    """450 sequences x 2 K/V heads at d = 64 are 900 planes; a partial slot is
    16 * (64 + 2) * 4 bytes, so 4 MiB hold 992 slots and the grid is cut to
    92 CTAs (one slot per CTA plus one per plane)."""
    seqlens, q, kc, vc = inputs.decode_inputs(450, 2, 2, 128, 64, torch.bfloat16, seed=301)
    _two_calls_against_oracle_and_regular(seqlens, q, kc, vc, 0.125)


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    q = torch.zeros(4096, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4096, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(4096, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(ops.GqaError) as err:
        ops.gqa_attn_decode_noalloc(q, kc, kc, sl, o, scale=0.1)
    assert err.value.status == 2  # GQA_ERR_UNSUPPORTED
