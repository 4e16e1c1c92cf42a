"""GPU test of the decode's early start.

The split-KV decode kernel locates each CTA's first unit from a read of the
sequence lengths made before its grid-dependency wait (the previous grid may
still be writing them) and prefetches that unit into L2; after the wait it
reads the lengths again and works the start out afresh if any changed. The
self-test entry feeds the first read from a decoy array, so these cases take
the second path (up to 128 sequences; a larger batch reads its lengths only
after the wait, and the decoy must then have no effect at all): the outputs
must be bit for bit those of the plain call (whose first read sees the real
lengths) and close to the oracle, with no device error from the decoy's
out-of-range values. Split-sequence cached
attention: microLLM-rocm optimisation log, Experiments 282-284.
"""
import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs, ops

pytestmark = pytest.mark.gpu

BF16_MAX = 2e-2
BF16_MEAN = 2e-3


def _decoys(sl, max_len, seed):
    g = torch.Generator().manual_seed(seed)
    B = sl.numel()
    other = torch.randint(1, max_len + 1, (B,), generator=g, dtype=torch.int32)
    one = sl.clone()
    one[B // 2] = max(1, int(one[B // 2]) - 1)
    bad = sl.clone()
    bad[0] = max_len + 7
    bad[-1] = -3
    return {"same": sl.clone(), "other": other, "one_changed": one,
            "zeros": torch.zeros(B, dtype=torch.int32), "out_of_range": bad}


@pytest.mark.parametrize("shape", [(64, 12, 2, 2048, 128), (8, 16, 2, 1500, 64),
                                   (5, 12, 2, 900, 256), (3, 8, 8, 700, 96),
                                   (200, 8, 2, 300, 128)],
                         ids=lambda s: "-".join(map(str, s)))
def test_decode_early_start_decoy_lengths(shape):
    B, H_q, H_kv, L, d = shape
    sl, q, kc, vc = inputs.decode_inputs(B, H_q, H_kv, L, d, torch.bfloat16, seed=700 + B + d)
    sld, qd, kcd, vcd = sl.cuda(), q.cuda(), kc.cuda(), vc.cuda()
    scale = d ** -0.5
    o_ref, lse_ref = ops.gqa_attn_decode_lse(qd, kcd, vcd, sld, scale=scale)
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    ref, _ = oracle.decode(q, kc, vc, sl, scale)
    d_ = np.abs(o_ref.float().cpu().numpy().astype(np.float64) - ref)
    assert d_.max() <= BF16_MAX and d_.mean() <= BF16_MEAN
    for name, early in _decoys(sl, L, 710 + B).items():
        o, lse = ops.gqa_attn_selftest_decode_early_lengths(qd, kcd, vcd, sld, early.cuda(),
                                                            scale=scale)
        torch.cuda.synchronize()
        assert ops.gqa_attn_get_device_error() == 0, name
        assert torch.equal(o, o_ref), f"{name}: O differs from the plain call"
        assert torch.equal(lse, lse_ref), f"{name}: lse differs from the plain call"
