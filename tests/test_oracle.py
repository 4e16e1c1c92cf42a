"""Pins for the float64 CPU oracle (no GPU).

The oracle is the definition of attention written out; these tests tie it to
things other than itself: hand-derived closed forms (tests/golden), invariants
the mathematics fixes, special cases that reduce to a textbook formula, and a
library routine (torch's scaled_dot_product_attention in float64 on the CPU).

The second half plants plausible mistakes -- a wrong head mapping, a dropped
term, a missing normalisation, a flipped sign, an off-by-one mask -- into a
plain numpy restatement and checks that the pin suite rejects every one of
them, so the pins are shown to have teeth.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_02_gb300 import inputs
from gqa_flash_attention_02_gb300.inputs import decode_inputs, prefill_inputs, varlen_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _arr(x):
    return np.array(x, dtype=np.float64)


def _rand(B, H_q, H_kv, N_q, N_kv, d, seed):
    q, k, v = prefill_inputs(B, H_q, H_kv, N_q, N_kv, d, torch.float64, seed)
    return q.numpy(), k.numpy(), v.numpy()


# --------------------------------------------------------------------------
# Pin checks. Each takes a prefill implementation
#     impl(q, k, v, causal, scale) -> (o, lse)
# and raises AssertionError when the implementation violates the pin.
# --------------------------------------------------------------------------

def pin_golden_closed_forms(impl):
    """Hand-derived fixtures: weights such as [1/4, 3/4] and [1/8, 2/8, 5/8]."""
    for name in ("two_keys_quarter_threequarter.json", "three_keys_scaled.json",
                 "gqa_head_mapping.json", "bottom_right_causal.json"):
        fx = _load(name)
        for mode, exp in fx["expect"].items():
            o, lse = impl(_arr(fx["q"]), _arr(fx["k"]), _arr(fx["v"]), mode == "causal",
                          fx["scale"])
            np.testing.assert_allclose(o, _arr(exp["o"]), rtol=0, atol=1e-12,
                                       err_msg=f"{name}:{mode}")
            np.testing.assert_allclose(lse, _arr(exp["lse"]), rtol=0, atol=1e-12,
                                       err_msg=f"{name}:{mode} lse")


def pin_gqa_equals_replicated_mha(impl):
    """GQA == MHA on K/V with each head repeated group times (collab-014 mapping)."""
    for (H_q, H_kv) in ((6, 2), (8, 1), (4, 4)):
        q, k, v = _rand(2, H_q, H_kv, 9, 13, 8, seed=7 + H_q + H_kv)
        g = H_q // H_kv
        k_rep, v_rep = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
        for causal in (False, True):
            o_gqa, _ = impl(q, k, v, causal, 0.3)
            o_mha, _ = impl(q, k_rep, v_rep, causal, 0.3)
            np.testing.assert_allclose(o_gqa, o_mha, rtol=0, atol=1e-14)


def pin_identical_keys_give_mean(impl):
    """All K rows equal -> uniform weights -> O = mean of the visible V rows."""
    q, k, v = _rand(1, 2, 1, 6, 6, 4, seed=3)
    k[:] = k[:, :, :1, :]
    o, _ = impl(q, k, v, False, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    o, _ = impl(q, k, v, True, 0.7)
    csum = np.cumsum(v, axis=2) / np.arange(1, 7).reshape(1, 1, 6, 1)
    np.testing.assert_allclose(o, np.broadcast_to(csum, o.shape), rtol=0, atol=1e-13)


def pin_scale_zero_gives_mean(impl):
    q, k, v = _rand(1, 2, 2, 5, 7, 4, seed=4)
    o, lse = impl(q, k, v, False, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(7), rtol=0, atol=1e-13)


def pin_dominant_logit_selects_row(impl):
    """One key aligned with q at a huge logit -> O equals that key's V row."""
    q, k0, v = _rand(1, 1, 1, 3, 8, 4, seed=5)
    for i, jstar in enumerate((2, 5, 7)):
        # key j* scores 60 against row i; every other key scores below 1 in size
        k = 0.05 * k0.copy()
        q_hat = q[0, 0, i] / np.linalg.norm(q[0, 0, i])
        k[0, 0, jstar] = 60.0 * q_hat
        o, _ = impl(q_hat.reshape(1, 1, 1, 4), k, v, False, 1.0)
        np.testing.assert_allclose(o[0, 0, 0], v[0, 0, jstar], rtol=0, atol=1e-12)


def pin_single_key_returns_it(impl):
    q, k, v = _rand(2, 4, 2, 3, 1, 8, seed=6)
    o, lse = impl(q, k, v, False, 0.5)
    want = np.repeat(v, 2, axis=1)  # every query row of head h_q sees K/V head h_q // 2
    np.testing.assert_allclose(o, np.broadcast_to(want, o.shape), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.5 * np.einsum("bhid,bhd->bhi", q, np.repeat(k[:, :, 0], 2, axis=1)),
                               rtol=0, atol=1e-13)


def pin_causal_row_is_truncated_full(impl):
    """Causal row i (N_q = N_kv) equals unmasked attention over keys [0, i]."""
    q, k, v = _rand(1, 2, 1, 7, 7, 4, seed=8)
    o_c, lse_c = impl(q, k, v, True, 0.4)
    for i in range(7):
        o_t, lse_t = impl(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], False, 0.4)
        np.testing.assert_allclose(o_c[:, :, i:i + 1], o_t, rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse_c[:, :, i:i + 1], lse_t, rtol=0, atol=1e-14)
    np.testing.assert_allclose(o_c[:, :, 0], np.repeat(v[:, :, 0], 2, axis=1), rtol=0, atol=1e-15)


def pin_permutation_invariance(impl):
    """Permuting K and V rows together leaves unmasked attention unchanged."""
    q, k, v = _rand(1, 2, 2, 4, 9, 4, seed=9)
    perm = np.random.default_rng(0).permutation(9)
    o1, l1 = impl(q, k, v, False, 0.6)
    o2, l2 = impl(q, k[:, :, perm], v[:, :, perm], False, 0.6)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_convex_hull(impl):
    """Each output coordinate lies between the min and max of the visible V column."""
    q, k, v = _rand(2, 4, 2, 6, 6, 4, seed=10)
    for causal in (False, True):
        o, _ = impl(q, k, v, causal, 2.0)
        vr = np.repeat(v, 2, axis=1)
        for i in range(6):
            n = i + 1 if causal else 6
            lo = vr[:, :, :n].min(axis=2)
            hi = vr[:, :, :n].max(axis=2)
            assert np.all(o[:, :, i] >= lo - 1e-12) and np.all(o[:, :, i] <= hi + 1e-12)


def pin_library_sdpa(impl):
    """Special case that reduces to torch's float64 CPU scaled_dot_product_attention."""
    F = torch.nn.functional
    for (H_q, H_kv, N_q, N_kv, causal) in ((4, 2, 11, 11, False), (4, 2, 11, 11, True),
                                           (6, 1, 5, 12, False), (3, 3, 16, 16, True)):
        q, k, v = _rand(2, H_q, H_kv, N_q, N_kv, 8, seed=11 + H_q + N_kv)
        o, _ = impl(q, k, v, causal, 0.35)
        ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                             torch.from_numpy(v), is_causal=causal,
                                             scale=0.35, enable_gqa=True).numpy()
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


PINS = [pin_golden_closed_forms, pin_gqa_equals_replicated_mha, pin_identical_keys_give_mean,
        pin_scale_zero_gives_mean, pin_dominant_logit_selects_row, pin_single_key_returns_it,
        pin_causal_row_is_truncated_full, pin_permutation_invariance, pin_convex_hull,
        pin_library_sdpa]


def _oracle_impl(q, k, v, causal, scale):
    return oracle.prefill(q, k, v, causal, scale)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_prefill_pins(pin):
    pin(_oracle_impl)


# --------------------------------------------------------------------------
# Decode, split merge and row-sampling pins (oracle only).
# --------------------------------------------------------------------------

def test_oracle_decode_golden():
    fx = _load("decode_two_sequences.json")
    kc = _arr([[[[float(x) for x in r] for r in h] for h in b] for b in fx["k_cache"]])
    vc = _arr([[[[float(x) for x in r] for r in h] for h in b] for b in fx["v_cache"]])
    o, lse = oracle.decode(_arr(fx["q"]), kc, vc, fx["seqlens"], fx["scale"])
    np.testing.assert_allclose(o, _arr(fx["expect"]["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, _arr(fx["expect"]["lse"]), rtol=0, atol=1e-12)


def test_oracle_decode_is_last_causal_prefill_row():
    """Decode at length L equals the last row of causal prefill with N_q = N_kv = L."""
    seqlens, q, kc, vc = decode_inputs(3, 6, 2, 40, 8, torch.float64, seed=12)
    o, lse = oracle.decode(q, kc, vc, seqlens, 0.25)
    assert np.isfinite(o).all()
    for b in range(3):
        L = int(seqlens[b])
        qp = np.zeros((1, 6, L, 8))
        qp[0, :, L - 1] = q[b].numpy()
        op, lp = oracle.prefill(qp, kc[b:b + 1, :, :L].numpy(), vc[b:b + 1, :, :L].numpy(),
                                True, 0.25)
        np.testing.assert_allclose(o[b], op[0, :, L - 1], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[b], lp[0, :, L - 1], rtol=0, atol=1e-14)


def test_oracle_decode_rejects_bad_seqlen():
    seqlens, q, kc, vc = decode_inputs(2, 2, 1, 8, 4, torch.float64, seed=13)
    with pytest.raises(ValueError):
        oracle.decode(q, kc, vc, [3, 9], 1.0)


def test_oracle_lse_merge_equals_unsplit():
    """Merging key-range partials by log-sum-exp reproduces the unsplit result
    (split-sequence cached attention, microLLM-rocm Experiments 282-284)."""
    q, k, v = _rand(1, 1, 1, 3, 37, 8, seed=14)
    o_full, lse_full = oracle.prefill(q, k, v, False, 0.5)
    cuts = [0, 5, 6, 20, 37]
    for i in range(3):
        parts_o, parts_l = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o_p, l_p = oracle.attend_row(q[0, 0, i], k[0, 0, a:b], v[0, 0, a:b], 0.5)
            parts_o.append(o_p)
            parts_l.append(l_p)
        parts_o.append(np.zeros(8))  # an empty part carries no weight
        parts_l.append(-np.inf)
        o_m, l_m = oracle.lse_merge(np.stack(parts_o), np.array(parts_l))
        np.testing.assert_allclose(o_m, o_full[0, 0, i], rtol=0, atol=1e-14)
        assert abs(l_m - lse_full[0, 0, i]) < 1e-13


def test_oracle_empty_row_and_empty_merge():
    o, lse = oracle.attend_row(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.all(o == 0) and lse == -np.inf
    o, lse = oracle.lse_merge(np.ones((2, 4)), np.array([-np.inf, -np.inf]))
    assert np.all(o == 0) and lse == -np.inf


def test_oracle_prefill_rows_match_full():
    q, k, v = _rand(2, 4, 2, 10, 14, 8, seed=15)
    o, lse = oracle.prefill(q, k, v, True, 0.3)
    rows = [(0, 0, 0), (1, 3, 9), (0, 2, 5), (1, 1, 3)]
    o_r, l_r = oracle.prefill_rows(q, k, v, True, 0.3, rows)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o_r[r], o[b, h, i])
        assert l_r[r] == lse[b, h, i]


def test_oracle_head_subset_and_threads():
    q, k, v = _rand(2, 4, 2, 10, 10, 8, seed=16)
    o_all, _ = oracle.prefill(q, k, v, True, 0.3)
    o_sub, _ = oracle.prefill(q, k, v, True, 0.3, heads=(2, 5), n_threads=2)
    flat_all, flat_sub = o_all.reshape(8, 10, 8), o_sub.reshape(8, 10, 8)
    np.testing.assert_array_equal(flat_sub[2:5], flat_all[2:5])
    assert np.isnan(flat_sub[:2]).all() and np.isnan(flat_sub[5:]).all()


# ------------------------------------------------------------------ ragged batches

def _varlen_brute(q, k, v, cu_q, cu_k, causal, scale):
    """Attention of every owned (token, head) row by the definition, written
    out with Python loops over the sequence's visible keys."""
    total_q, H_q, d = q.shape
    H_kv = k.shape[1]
    o = np.full(q.shape, np.nan)
    lse = np.full((H_q, total_q), np.nan)
    for b in range(len(cu_q) - 1):
        len_q, len_k = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        for i in range(len_q):
            t = cu_q[b] + i
            n = min(len_k, i + (len_k - len_q) + 1) if causal else len_k
            for h in range(H_q):
                hk = h // (H_q // H_kv)
                logits = [scale * sum(q[t, h, c] * k[cu_k[b] + j, hk, c] for c in range(d))
                          for j in range(n)]
                m = max(logits)
                w = [math.exp(x - m) for x in logits]
                z = sum(w)
                for c in range(d):
                    o[t, h, c] = sum(w[j] * v[cu_k[b] + j, hk, c] for j in range(n)) / z
                lse[h, t] = m + math.log(z)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_varlen_brute_force(causal):
    """A ragged batch -- lengths 1, 3, 0, 5 with 2, 3, 4, 7 keys (bottom-right
    offsets 1, 0, -, 2) -- against the definition evaluated row by row."""
    lens_q, lens_k = [1, 3, 0, 5], [2, 3, 4, 7]
    q, k, v = (np.random.default_rng(21).standard_normal(s) for s in
               ((9, 4, 3), (16, 2, 3), (16, 2, 3)))
    cu_q, cu_k = np.cumsum([0] + lens_q), np.cumsum([0] + lens_k)
    o, lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, causal, 0.7)
    o_b, lse_b = _varlen_brute(q, k, v, cu_q, cu_k, causal, 0.7)
    np.testing.assert_allclose(o, o_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_b, rtol=0, atol=1e-13)


def test_oracle_varlen_equal_lengths_is_dense_batch():
    """Equal lengths packed token-major give the dense batch, transposed."""
    q, k, v = _rand(3, 4, 2, 6, 9, 8, seed=22)
    o, lse = oracle.prefill(q, k, v, True, 0.4)
    pack = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(-1, x.shape[1], 8))
    cu_q, cu_k = np.arange(4) * 6, np.arange(4) * 9
    o_v, lse_v = oracle.prefill_varlen(pack(q), pack(k), pack(v), cu_q, cu_k, True, 0.4)
    np.testing.assert_array_equal(o_v, pack(o))
    np.testing.assert_array_equal(lse_v, lse.transpose(1, 0, 2).reshape(4, -1))


def test_oracle_varlen_rows_and_unowned_rows():
    """Selected rows equal the full result; rows past cu_q[B] stay NaN."""
    q, k, v, cu_q, cu_k = (x.numpy() for x in
                           varlen_inputs([4, 1, 7], [6, 1, 9], 6, 2, 8, torch.float64, seed=23))
    q_pad = np.concatenate([q, np.ones((2, 6, 8))])  # two tokens no sequence owns
    o, lse = oracle.prefill_varlen(q_pad, k, v, cu_q, cu_k, True, 0.3)
    assert np.isnan(o[12:]).all() and np.isnan(lse[:, 12:]).all()
    assert np.isfinite(o[:12]).all()
    rows = [(0, 0), (4, 5), (11, 3), (7, 1)]
    o_r, l_r = oracle.prefill_varlen_rows(q, k, v, cu_q, cu_k, True, 0.3, rows)
    for r, (t, h) in enumerate(rows):
        np.testing.assert_array_equal(o_r[r], o[t, h])
        assert l_r[r] == lse[h, t]


# ------------------------------------------------------------------ backward

def _sdpa_grads(q, k, v, do, causal, scale):
    """Gradients from torch autograd through scaled_dot_product_attention in
    float64 on the CPU (a library routine, with the bottom-right mask given
    explicitly)."""
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    n_q, n_kv = q.shape[2], k.shape[2]
    mask = torch.ones(n_q, n_kv, dtype=torch.bool).tril(n_kv - n_q) if causal else None
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale,
                                                         enable_gqa=True)
    o.backward(torch.tensor(do))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def pin_backward_autograd(bwd):
    """bwd(q, k, v, do, causal, scale) -> (dq, dk, dv) agrees with autograd."""
    for (H_q, H_kv, N_q, N_kv), causal in [((4, 2, 5, 7), True), ((6, 1, 4, 4), False),
                                           ((2, 2, 3, 9), True)]:
        q, k, v = _rand(2, H_q, H_kv, N_q, N_kv, 6, seed=30 + N_kv)
        do = np.random.default_rng(31 + N_q).standard_normal(q.shape)
        got = bwd(q, k, v, do, causal, 0.6)
        ref = _sdpa_grads(q, k, v, do, causal, 0.6)
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            np.testing.assert_allclose(g, r, rtol=0, atol=1e-12, err_msg=f"{name} causal={causal}")


def test_oracle_backward_matches_autograd():
    pin_backward_autograd(oracle.prefill_backward)


def test_oracle_backward_finite_differences():
    """Central differences of L = sum(O * dO), O from the forward oracle,
    against the backward oracle: independent of the backward formula."""
    q, k, v = _rand(1, 4, 2, 3, 5, 3, seed=32)
    do = np.random.default_rng(33).standard_normal(q.shape)
    dq, dk, dv = oracle.prefill_backward(q, k, v, do, True, 0.8)

    def loss(q_, k_, v_):
        return float((oracle.prefill(q_, k_, v_, True, 0.8)[0] * do).sum())

    eps = 1e-6
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args_p, args_m = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def test_oracle_backward_gqa_is_sum_over_replicated_heads():
    """dK, dV of a K/V head are the sums over its query heads of the MHA
    gradients with that head replicated; dQ is unchanged."""
    q, k, v = _rand(1, 6, 2, 5, 5, 4, seed=34)
    do = np.random.default_rng(35).standard_normal(q.shape)
    dq, dk, dv = oracle.prefill_backward(q, k, v, do, True, 0.5)
    k_r, v_r = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    dq_m, dk_m, dv_m = oracle.prefill_backward(q, k_r, v_r, do, True, 0.5)
    np.testing.assert_allclose(dq, dq_m, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, dk_m.reshape(1, 2, 3, 5, 4).sum(axis=2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv_m.reshape(1, 2, 3, 5, 4).sum(axis=2), rtol=0, atol=1e-13)


def _bwd_restated(q, k, v, do, causal, scale, mutation=None):
    """The backward restated in numpy, with an optional planted mistake."""
    B, H_q, N_q, _ = q.shape
    H_kv, N_kv = k.shape[1], k.shape[2]
    g = H_q // H_kv
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    off = N_kv - N_q + (1 if mutation == "mask_off_by_one" else 0)
    vis = (np.arange(N_kv)[None, :] <= np.arange(N_q)[:, None] + off) if causal else \
        np.ones((N_q, N_kv), dtype=bool)
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            # (planted) only the group's first query head reaches dK, dV
            hk_acc = None if mutation == "first_head_only" and h % g else hk
            s = np.where(vis, scale * q[b, h] @ k[b, hk].T, -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            p = e / e.sum(axis=1, keepdims=True)
            o = p @ v[b, hk]
            dp = do[b, h] @ v[b, hk].T
            delta = 0.0 if mutation == "no_delta" else (do[b, h] * o).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dq[b, h] = (1.0 if mutation == "no_scale_dq" else scale) * (ds @ k[b, hk])
            if hk_acc is not None:
                # dV from P, or (planted) from the exponentials before normalising
                dv[b, hk] += (e if mutation == "dv_unnormalised" else p).T @ do[b, h]
                dk[b, hk] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def test_backward_pin_accepts_unmutated_restatement():
    pin_backward_autograd(_bwd_restated)


@pytest.mark.parametrize("mutation", ["no_delta", "no_scale_dq", "first_head_only",
                                      "mask_off_by_one", "dv_unnormalised"])
def test_backward_pin_rejects_planted_mistake(mutation):
    with pytest.raises(AssertionError):
        pin_backward_autograd(lambda *a: _bwd_restated(*a, mutation=mutation))


def test_oracle_reads_bf16_exactly():
    """bf16 inputs are widened exactly: the oracle on bf16 tensors equals the
    oracle on the same values pre-converted to float64."""
    q, k, v = prefill_inputs(1, 2, 1, 4, 4, 8, torch.bfloat16, seed=17)
    o1, _ = oracle.prefill(q, k, v, False, 0.5)
    o2, _ = oracle.prefill(q.double(), k.double(), v.double(), False, 0.5)
    np.testing.assert_array_equal(o1, o2)


def test_oracle_rejects_bad_head_ratio():
    q, k, v = _rand(1, 3, 2, 2, 2, 4, seed=18)
    with pytest.raises(ValueError):
        oracle.prefill(q, k, v, False, 1.0)


# --------------------------------------------------------------------------
# Planted mistakes: a numpy restatement with one error each must fail a pin.
# --------------------------------------------------------------------------

def _np_prefill(q, k, v, causal, scale, mutation=None):
    B, H_q, N_q, d = q.shape
    H_kv, N_kv = k.shape[1], k.shape[2]
    g = H_q // H_kv
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H_q):
            hk = h % H_kv if mutation == "head_modulo" else h // g
            hv = (hk + 1) % H_kv if mutation == "value_head_shifted" else hk
            for i in range(N_q):
                off = 0 if mutation == "causal_top_left" else N_kv - N_q
                n = min(N_kv, i + off + 1) if causal else N_kv
                if mutation == "causal_strict" and causal:
                    n = max(1, n - 1)
                if mutation == "dropped_last_key" and n > 1:
                    n -= 1
                keys = k[b, hk, :n]
                if mutation == "scores_key_reversed":
                    keys = keys[::-1]
                sc = 1.0 if mutation == "scale_ignored" else scale
                s = sc * (keys @ q[b, h, i])
                if mutation == "sign_flipped":
                    s = -s
                m = s.max()
                p = np.exp(s - m)
                l = p.sum()
                o[b, h, i] = p @ v[b, hv, :n] / (1.0 if mutation == "unnormalised" else l)
                lse[b, h, i] = (0.0 if mutation == "lse_without_max" else m) + math.log(l)
    return o, lse


MUTATIONS = ["head_modulo", "value_head_shifted", "causal_top_left", "causal_strict",
             "dropped_last_key", "scores_key_reversed", "scale_ignored", "sign_flipped",
             "unnormalised", "lse_without_max"]


def test_pins_accept_unmutated_restatement():
    for pin in PINS:
        pin(lambda q, k, v, c, s: _np_prefill(q, k, v, c, s))


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_reject_planted_mistake(mutation):
    caught = []
    for pin in PINS:
        try:
            pin(lambda q, k, v, c, s: _np_prefill(q, k, v, c, s, mutation))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{mutation}'"


# ------------------------------------------------------------------ fp8 (e4m3) cache

def test_e4m3_codes_closed_forms():
    """Codes whose values follow from the format's definition by hand."""
    cases = {0x00: 0.0, 0x80: -0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0xB8: -1.0, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0,
             0x77: 240.0, 0x30: 0.5}
    got = oracle.e4m3_value(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values())))
    assert np.isnan(oracle.e4m3_value(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_codes_match_torch_float8():
    """Every code against torch's float8_e4m3fn widening (a library special case)."""
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_decode_fp8_is_decode_of_the_widened_scaled_cache():
    """decode_fp8 equals decode on e4m3(code) * scale, written out here with
    torch's widening; a K scale folds into the softmax scale, a V scale
    multiplies O and leaves the lse alone."""
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_fp8(3, 8, 2, 200, 64, seed=11,
                                                     seqlens=[200, 1, 77])
    o, lse = oracle.decode_fp8(q, k8, v8, ks, vs, sl, 0.125)
    kw = k8.to(torch.float64) * ks.double().view(1, 2, 1, 1)
    vw = v8.to(torch.float64) * vs.double().view(1, 2, 1, 1)
    o2, lse2 = oracle.decode(q, kw, vw, sl, 0.125)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    one = torch.ones(2)
    o_k, lse_k = oracle.decode_fp8(q, k8, v8, torch.full((2,), 0.5), one, sl, 0.125)
    o_ref, lse_ref = oracle.decode_fp8(q, k8, v8, one, one, sl, 0.0625)
    assert np.allclose(o_k, o_ref, atol=1e-13) and np.allclose(lse_k, lse_ref, atol=1e-13)
    o_v, lse_v = oracle.decode_fp8(q, k8, v8, one, torch.full((2,), 3.0), sl, 0.125)
    o_1, lse_1 = oracle.decode_fp8(q, k8, v8, one, one, sl, 0.125)
    assert np.allclose(o_v, 3 * o_1, atol=1e-12) and np.array_equal(lse_v, lse_1)


def test_decode_fp8_planted_mistakes_fail():
    """A decoder that drops the subnormals, or uses bias 8, changes the result."""
    codes = np.arange(256, dtype=np.uint8)
    good = oracle.e4m3_value(codes)
    c = codes.astype(np.int64)
    e, m = (c >> 3) & 0xF, (c & 7) / 8.0
    no_sub = np.where(e == 0, 0.0, np.abs(good))
    bias8 = np.where(e == 0, m * 2.0 ** -7, (1 + m) * np.exp2(e - 8.0))
    ok = ~np.isnan(good)
    assert not np.array_equal(np.abs(good)[ok], no_sub[ok])
    assert not np.array_equal(np.abs(good)[ok], bias8[ok])


# ------------------------------------------------------------------ int8 cache

def test_int8_codes_closed_forms():
    """Two's-complement codes whose values follow by hand."""
    cases = {0x00: 0.0, 0x01: 1.0, 0x7F: 127.0, 0x80: -128.0, 0x81: -127.0, 0xFF: -1.0,
             0xC0: -64.0, 0x40: 64.0, 0x2A: 42.0, 0xD6: -42.0}
    got = oracle.int8_value(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values())))


def test_int8_codes_match_torch_int8():
    """Every code against torch's int8 widening (a library special case)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.int8).to(torch.float64).numpy()
    assert np.array_equal(oracle.int8_value(codes), ref)
    t = torch.from_numpy(codes).view(torch.int8)
    assert np.array_equal(oracle.int8_value(t), ref)


def test_int8_planted_mistakes_fail():
    """Reading the bytes as unsigned, or as offset binary (code - 128),
    gives other values."""
    codes = np.arange(256, dtype=np.uint8)
    good = oracle.int8_value(codes)
    assert not np.array_equal(good, codes.astype(np.float64))
    assert not np.array_equal(good, codes.astype(np.float64) - 128.0)


def test_decode_int8_is_decode_of_the_widened_scaled_cache():
    """decode_int8 equals decode on int8(code) * scale, written out here with
    torch's widening; a K scale folds into the softmax scale, a V scale
    multiplies O and leaves the lse alone; the rows past each sequence
    (code -128) are never used."""
    sl, q, k8, v8, ks, vs = inputs.decode_inputs_int8(3, 8, 2, 200, 64, seed=12,
                                                      seqlens=[200, 1, 77])
    assert int(k8[1, :, 1:].min()) == -128 and int(k8[0].min()) >= -127
    o, lse = oracle.decode_int8(q, k8, v8, ks, vs, sl, 0.125)
    kw = k8.to(torch.float64) * ks.double().view(1, 2, 1, 1)
    vw = v8.to(torch.float64) * vs.double().view(1, 2, 1, 1)
    o2, lse2 = oracle.decode(q, kw, vw, sl, 0.125)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    k_other, v_other = k8.clone(), v8.clone()
    k_other[1, :, 1:] = 5
    v_other[2, :, 77:] = 7
    o3, lse3 = oracle.decode_int8(q, k_other, v_other, ks, vs, sl, 0.125)
    assert np.array_equal(o, o3) and np.array_equal(lse, lse3)
    one = torch.ones(2)
    o_k, lse_k = oracle.decode_int8(q, k8, v8, torch.full((2,), 0.5), one, sl, 0.125)
    o_ref, lse_ref = oracle.decode_int8(q, k8, v8, one, one, sl, 0.0625)
    assert np.allclose(o_k, o_ref, atol=1e-13) and np.allclose(lse_k, lse_ref, atol=1e-13)
    o_v, lse_v = oracle.decode_int8(q, k8, v8, one, torch.full((2,), 3.0), sl, 0.125)
    o_1, lse_1 = oracle.decode_int8(q, k8, v8, one, one, sl, 0.125)
    assert np.allclose(o_v, 3 * o_1, atol=1e-10) and np.array_equal(lse_v, lse_1)


def test_decode_int8_one_dominant_code():
    """Closed form: one key whose codes are q's signs times 127, all other
    keys zero, with a large K scale: that key takes all the weight, so O is
    its V row (codes times the V scale) to double precision."""
    B, H_q, H_kv, L, d = 1, 2, 1, 5, 8
    q = torch.tensor([[[1.0, -1, 1, 1, -1, 1, -1, -1], [2.0, -1, 3, 1, -1, 1, -2, -1]]],
                     dtype=torch.bfloat16)
    k8 = torch.zeros(B, H_kv, L, d, dtype=torch.int8)
    k8[0, 0, 3] = torch.tensor([127, -127, 127, 127, -127, 127, -127, -127], dtype=torch.int8)
    v8 = torch.arange(B * H_kv * L * d).view(B, H_kv, L, d).remainder(251).sub(125).to(torch.int8)
    sl = torch.tensor([L], dtype=torch.int32)
    o, _ = oracle.decode_int8(q, k8, v8, torch.tensor([1.0]), torch.tensor([0.25]), sl, 1.0)
    want = v8[0, 0, 3].double().numpy() * 0.25
    assert np.abs(o[0] - want[None, :]).max() < 1e-12
