"""GPU parity for the clustered dense prefill: units that pair the tiles of
a group of 4 or 8 query heads run in clusters of g / 2 CTAs, and each K/V
block is loaded once for the whole group and multicast to the cluster
(one K/V tile load per query-head group, the GQA saving of the
BootstrapAI evolution log, collab-014 "Kernel 9 GQA").

Shapes have at least four two-tile units per SM (the clustered schedule
is used from there up), with g = 4 (clusters of 2) and g = 8 (clusters of
4), head dims 64 (one 64-column panel per block, loaded by the cluster's
first CTA) and 128 (two panels, one per CTA), causal and not, a ragged
last tile and more keys than queries. Bounds: the bf16 ones of the
other tests (max abs 2e-2, mean abs 2e-3; lse max abs 5e-3), on every row
of a few heads (the oracle's cost), and repeated launches must agree bit
for bit (the work counter and the hand-out between the CTAs re-arm).
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

CASES = [
    (4, 32, 8, 1280, 1280, 128, True),    # g = 4: clusters of 2, two panels; 640 pairs
    (4, 32, 8, 1200, 1200, 64, False),    # g = 4, one panel, ragged last tile
    (2, 64, 8, 1280, 1280, 128, True),    # g = 8: clusters of 4; 640 pairs
    (2, 64, 8, 1300, 1500, 64, True),     # g = 8, more keys than queries; 704 pairs
]


def _heads(H_q, g):
    # one whole group and a head of the last group
    return list(range(g)) + [H_q - 1]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_clustered_prefill_matches_oracle(case):
    B, H_q, H_kv, N_q, N_kv, d, causal = case
    g = H_q // H_kv
    q, k, v = inputs.prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.bfloat16, seed=700 + N_q + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    ops.gqa_attn_fwd(qd, kd, vd, o, causal=causal, scale=d ** -0.5)
    o2, lse = ops.gqa_attn_fwd_lse(qd, kd, vd, causal=causal, scale=d ** -0.5)
    runs = [o.clone()]
    for _ in range(3):
        ops.gqa_attn_fwd(qd, kd, vd, o, causal=causal, scale=d ** -0.5)
        runs.append(o.clone())
    torch.cuda.synchronize()
    assert ops.gqa_attn_get_device_error() == 0
    for r in runs[1:]:
        assert torch.equal(r, runs[0]), "repeated launches differ"
    assert not torch.isnan(o.float()).any(), "rows left unwritten"
    heads = _heads(H_q, g)
    bsel = B - 1
    qs = q[bsel:bsel + 1, heads]
    kv_heads = sorted({h // g for h in heads})
    ks, vs = k[bsel:bsel + 1, kv_heads], v[bsel:bsel + 1, kv_heads]
    # the oracle on the selected heads: map each selected query head to its K/V head
    for i, h in enumerate(heads):
        j = kv_heads.index(h // g)
        ref, ref_lse = oracle.prefill(qs[:, i:i + 1], ks[:, j:j + 1], vs[:, j:j + 1], causal,
                                      d ** -0.5, n_threads=THREADS)
        for got, what in ((o, "plain"), (o2, "lse kernel")):
            x = got[bsel, h].float().cpu().numpy().astype(np.float64)
            diff = np.abs(x - ref[0, 0])
            assert diff.max() <= BF16_MAX and diff.mean() <= BF16_MEAN, \
                f"{case} head {h} {what}: max {diff.max():.3e} mean {diff.mean():.3e}"
        assert np.abs(lse[bsel, h].cpu().numpy().astype(np.float64) - ref_lse[0, 0]).max() <= LSE_MAX
