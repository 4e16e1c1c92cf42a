"""The decode entry point that allocates nothing (GPU).

Some callers cannot let a library call cudaMalloc: a serving loop held to a
pre-reserved memory budget, a latency-critical path where an allocation may
synchronise the device, a process whose device memory another allocator
owns. gqa_attn_decode_noalloc serves them from a fixed scratch array in the
library's device memory. This file checks, through the C ABI, that two calls
in a row give the same result as the regular gqa_attn_decode within the bf16
tolerance the other tests use, and that it runs without any workspace
existing first (it is also collected last, after every other test).
"""
import numpy as np
import pytest
import torch

from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

BF16_MAX = 2e-2
BF16_MEAN = 2e-3


def _close(a, b):
    d = np.abs(a.float().cpu().numpy().astype(np.float64) - b.float().cpu().numpy())
    return float(d.max()), float(d.mean())


@pytest.mark.parametrize("shape", [inputs.decode_shapes()[1], inputs.decode_shapes()[2]],
                         ids=lambda s: s.name)
def test_noalloc_decode_matches_regular_entry_point_twice(shape):
    seqlens, q, kc, vc = (t.cuda() for t in inputs.decode_inputs_for(shape))
    o1 = torch.full_like(q, float("nan"))
    o2 = torch.full_like(q, float("nan"))
    # two calls in a row share the scratch; each must be right on its own
    ops.gqa_attn_decode_noalloc(q, kc, vc, seqlens, o1, scale=shape.scale)
    ops.gqa_attn_decode_noalloc(q, kc, vc, seqlens, o2, scale=shape.scale)
    ref = ops.gqa_attn_decode(q, kc, vc, seqlens, scale=shape.scale)
    torch.cuda.synchronize()
    for o in (o1, o2):
        assert torch.isfinite(o.float()).all()
        mx, mean = _close(o, ref)
        assert mx <= BF16_MAX and mean <= BF16_MEAN, (mx, mean)


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    q = torch.zeros(4096, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4096, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
    sl = torch.ones(4096, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(ops.GqaError) as err:
        ops.gqa_attn_decode_noalloc(q, kc, kc, sl, o, scale=0.1)
    assert err.value.status == 2  # GQA_ERR_UNSUPPORTED
