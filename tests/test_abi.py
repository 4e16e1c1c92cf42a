"""Host-side checks of the C-ABI library (no GPU needed).

The library is built for sm_103a and loaded with ctypes; every function the
header declares must be exported. Argument validation happens before any
CUDA call, so invalid arguments are checked here with fake, never
dereferenced pointers. The persistent scheduler's work plan is a host
function too: every query tile must be covered exactly once, and units must
come heaviest first under the causal mask.
"""
import ctypes
import os
import re

import pytest

from gqa_flash_attention_02_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")

A = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
MIS = ctypes.c_void_p(0x10008)     # misaligned
SEQ = ctypes.c_void_p(0x20000)


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char \*)\s*(gqa_attn_\w+)\s*\(", text,
                                 re.M)))


def test_library_exports_every_declared_symbol():
    lib = ops.load()
    declared = _declared()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in gqa_attn.h but not exported"
    assert sorted(ops.EXPORTED) == declared


def test_status_strings():
    for code, name in ops.STATUS_NAMES.items():
        assert ops.status_string(code).startswith(name)
    assert "unknown" in ops.status_string(99)


@pytest.mark.parametrize("fn", ["gqa_attn_fwd", "gqa_attn_fwd_f32"])
def test_prefill_validation(fn):
    f = getattr(ops.load(), fn)
    ok = dict(B=1, H_q=4, H_kv=2, N_q=128, N_kv=128, d=64, causal=0, scale=0.125)

    def call(q=A, k=A, v=A, o=A, **kw):
        a = dict(ok, **kw)
        return f(q, k, v, o, a["B"], a["H_q"], a["H_kv"], a["N_q"], a["N_kv"], a["d"],
                 a["causal"], a["scale"], None)

    assert call(q=None) == 1
    assert call(o=MIS) == 1
    assert call(B=0) == 1
    assert call(N_kv=-3) == 1
    assert call(H_q=6, H_kv=4) == 1          # not a whole group
    assert call(scale=float("nan")) == 1
    assert call(scale=float("inf")) == 1
    assert call(causal=1, N_q=256, N_kv=128) == 2   # bottom-right mask undefined
    assert call(d=80) == 2
    assert call(B=1 << 14, H_q=1 << 10, H_kv=1 << 10, N_q=1 << 10, N_kv=1 << 10) == 2


@pytest.mark.parametrize("fn", ["gqa_attn_decode", "gqa_attn_decode_f32"])
def test_decode_validation(fn):
    f = getattr(ops.load(), fn)

    def call(q=A, kc=A, vc=A, s=SEQ, o=A, B=2, H_q=12, H_kv=2, L=2048, d=128, scale=0.088):
        return f(q, kc, vc, s, o, B, H_q, H_kv, L, d, scale, None)

    assert call(s=None) == 1
    assert call(s=ctypes.c_void_p(0x20002)) == 1
    assert call(kc=MIS) == 1
    assert call(L=0) == 1
    assert call(H_q=12, H_kv=5) == 1
    assert call(scale=float("-inf")) == 1
    assert call(d=48) == 2
    assert call(L=(1 << 20) + 1) == 2


@pytest.mark.parametrize("fn", ["gqa_attn_fwd_varlen", "gqa_attn_fwd_varlen_lse"])
def test_varlen_validation(fn):
    f = getattr(ops.load(), fn)
    lse = fn.endswith("_lse")

    def call(q=A, k=A, v=A, o=A, l=None, cq=SEQ, ck=SEQ, B=3, H_q=8, H_kv=2, tq=700, tk=900,
             d=128, causal=1, scale=0.088):
        head = (q, k, v, o) + ((l,) if lse else ())
        return f(*head, cq, ck, B, H_q, H_kv, tq, tk, d, causal, scale, None)

    assert call(cq=None) == 1
    assert call(ck=ctypes.c_void_p(0x20002)) == 1   # offsets not 4-byte aligned
    assert call(v=MIS) == 1
    assert call(B=0) == 1
    assert call(tq=-1) == 1
    assert call(H_q=8, H_kv=3) == 1
    assert call(scale=float("nan")) == 1
    assert call(d=80) == 2   # head dims 32, 64, 96, 128, 256 only
    assert call(d=512) == 2
    assert call(B=4097) == 2                        # above the sequences-per-call limit
    assert call(tq=1 << 22, H_q=1 << 10, H_kv=1 << 8) == 2
    assert call(tq=0) == 0                          # no query rows: nothing launched
    assert call(tk=0) == 1                          # query rows but no keys
    if lse:
        assert call(l=ctypes.c_void_p(0x30002)) == 1


def test_bshd_validation():
    f = ops.load().gqa_attn_fwd_bshd

    def call(q=A, k=A, v=A, o=A, B=2, H_q=8, H_kv=2, N_q=300, N_kv=300, d=128, causal=1,
             scale=0.088):
        return f(q, k, v, o, B, H_q, H_kv, N_q, N_kv, d, causal, scale, None)

    assert call(q=None) == 1
    assert call(o=MIS) == 1
    assert call(N_q=0) == 1
    assert call(H_q=6, H_kv=4) == 1
    assert call(causal=1, N_q=400, N_kv=300) == 2   # bottom-right mask undefined
    assert call(d=48) == 2
    assert call(B=5000, N_q=10, N_kv=10) == 2       # above the sequences-per-call limit


def test_decode_chunk_validation():
    f = ops.load().gqa_attn_decode_chunked
    base = (A, A, A, SEQ, A, 2, 12, 2, 2048, 128, 0.088)
    assert f(*base, 33, None) == 1
    assert f(*base, 96, None) == 1    # not a multiple of the 64-row sub-block
    assert f(*base, 4096, None) == 1  # above the largest split
    assert f(*base, -64, None) == 1


def test_selftest_rejects_bad_limit():
    lib = ops.load()
    assert lib.gqa_attn_selftest_wait_timeout(0, None) == 1
    assert lib.gqa_attn_selftest_wait_timeout(200000, None) == 1


PLAN_CASES = [
    (1, 32, 8, 2048, 2048, True),    # LLaMA-3-8B-shaped layer
    (4, 16, 4, 4096, 4096, True),    # long sequence
    (2, 8, 8, 1024, 1024, True),     # MHA: pairs of q-tiles of one head
    (2, 8, 1, 1024, 1024, False),    # MQA
    (1, 6, 2, 300, 300, True),       # odd group (3) with a ragged tail
    (3, 3, 3, 200, 520, True),       # N_q < N_kv, bottom-right
    (1, 5, 1, 129, 129, False),      # odd tile count: last unit holds one tile
]


@pytest.mark.parametrize("case", PLAN_CASES)
def test_prefill_plan_covers_each_tile_once_heavy_first(case):
    B, H_q, H_kv, N_q, N_kv, causal = case
    units = ops.gqa_attn_prefill_plan(B, H_q, H_kv, N_q, N_kv, causal)
    g = H_q // H_kv
    n_qt = -(-N_q // 128)
    n_kt = -(-N_kv // 128)
    seen = {}
    extents = []
    for (b, h_kv, t0, t1) in units:
        ext = 0
        for (h_q, qt, nb) in (t0, t1):
            if nb == 0:
                assert (h_q, qt) == (-1, -1)
                continue
            assert h_q // g == h_kv, "tile mapped to the wrong K/V head"
            key = (b, h_q, qt)
            assert key not in seen
            seen[key] = nb
            # blocks needed: keys up to the last row's bottom-right limit
            last_row = min(N_q - 1, (qt + 1) * 128 - 1)
            want = min(n_kt, (last_row + N_kv - N_q) // 128 + 1) if causal else n_kt
            assert nb == want
            ext = max(ext, nb)
        assert ext > 0
        extents.append(ext)
    assert len(seen) == B * H_q * n_qt
    assert extents == sorted(extents, reverse=True), "units are not heavy-first"
    if g % 2 == 0:
        for (_, _, t0, t1) in units:
            if t1[2] > 0:
                assert t0[1] == t1[1], "even groups pair tiles of the same q_tile"


@pytest.mark.parametrize("case,tiles_per_unit", [
    ((2, 8, 8, 1024, 1024, 0), 1),     # 64 pairs would leave most of 148 SMs idle
    ((2, 8, 1, 1024, 1024, 1), 1),
    ((1, 32, 8, 2048, 2048, 1), 2),    # the LLaMA-3-8B layer: 256 pairs
    ((4, 16, 4, 4096, 4096, 1), 2),
])
def test_prefill_plan_splits_small_problems_into_single_tiles(case, tiles_per_unit):
    units = ops.gqa_attn_prefill_plan(*case)
    B, H_q, H_kv, N_q = case[:4]
    n_tiles = B * H_q * -(-N_q // 128)
    assert len(units) == -(-n_tiles // tiles_per_unit) if tiles_per_unit == 1 else len(units) >= n_tiles // 2
    if tiles_per_unit == 1:
        assert all(t1[2] == 0 for (_, _, _, t1) in units)


def test_prefill_plan_rejects_bad_sizes():
    lib = ops.load()
    assert lib.gqa_attn_prefill_plan(1, 6, 4, 128, 128, 0, -1, None) == -1
    assert lib.gqa_attn_prefill_plan(1, 4, 4, 256, 128, 1, -1, None) == -1


def test_backward_validation():
    f = ops.load().gqa_attn_bwd
    ok = dict(B=1, H_q=4, H_kv=2, N_q=128, N_kv=128, d=64, causal=0, scale=0.125)
    LSE = ctypes.c_void_p(0x30004)     # 4-byte aligned
    LSE_MIS = ctypes.c_void_p(0x30002)

    def call(q=A, k=A, v=A, o=A, do=A, lse=LSE, dq=A, dk=A, dv=A, **kw):
        a = dict(ok, **kw)
        return f(q, k, v, o, do, lse, dq, dk, dv, a["B"], a["H_q"], a["H_kv"], a["N_q"],
                 a["N_kv"], a["d"], a["causal"], a["scale"], None)

    assert call(do=None) == 1
    assert call(lse=None) == 1
    assert call(dk=None) == 1
    assert call(dv=MIS) == 1
    assert call(lse=LSE_MIS) == 1
    assert call(B=0) == 1
    assert call(H_q=6, H_kv=4) == 1
    assert call(scale=float("nan")) == 1
    assert call(causal=1, N_q=256, N_kv=128) == 2
    assert call(d=48) == 2   # head dims 32, 64, 96, 128 only
    assert call(d=256) == 2


def test_decode_fp8_validation():
    f = ops.load().gqa_attn_decode_fp8
    SC = ctypes.c_void_p(0x40000)
    SC_MIS = ctypes.c_void_p(0x40002)
    ok = dict(B=2, H_q=8, H_kv=2, max_len=256, d=128, scale=0.1)

    def call(q=A, k=A, v=A, ks=SC, vs=SC, sl=SEQ, o=A, lse=None, **kw):
        a = dict(ok, **kw)
        return f(q, k, v, ks, vs, sl, o, lse, a["B"], a["H_q"], a["H_kv"], a["max_len"], a["d"],
                 a["scale"], None)

    assert call(k=None) == 1
    assert call(ks=None) == 1
    assert call(vs=SC_MIS) == 1
    assert call(v=MIS) == 1
    assert call(lse=SC_MIS) == 1
    assert call(H_q=6, H_kv=4) == 1
    assert call(scale=float("nan")) == 1
    assert call(d=48) == 2   # head dims 32, 64, 96, 128 only
    assert call(d=256) == 2
    assert call(max_len=(1 << 20) + 1) == 2


def test_decode_int8_validation():
    """The int8 entry checks what the fp8 one checks."""
    f = ops.load().gqa_attn_decode_int8
    SC = ctypes.c_void_p(0x40000)
    SC_MIS = ctypes.c_void_p(0x40002)
    ok = dict(B=2, H_q=8, H_kv=2, max_len=256, d=128, scale=0.1)

    def call(q=A, k=A, v=A, ks=SC, vs=SC, sl=SEQ, o=A, lse=None, **kw):
        a = dict(ok, **kw)
        return f(q, k, v, ks, vs, sl, o, lse, a["B"], a["H_q"], a["H_kv"], a["max_len"], a["d"],
                 a["scale"], None)

    assert call(q=None) == 1
    assert call(vs=None) == 1
    assert call(ks=SC_MIS) == 1
    assert call(k=MIS) == 1
    assert call(lse=SC_MIS) == 1
    assert call(H_q=6, H_kv=4) == 1
    assert call(scale=float("inf")) == 1
    assert call(B=0) == 1
    assert call(d=48) == 2
    assert call(d=256) == 2
    assert call(max_len=(1 << 20) + 1) == 2


def test_selftest_decode_early_lengths_validation():
    f = ops.load().gqa_attn_selftest_decode_early_lengths
    EARLY = ctypes.c_void_p(0x30000)
    ok = dict(B=2, H_q=8, H_kv=2, max_len=256, d=128, scale=0.1)

    def call(early=EARLY, **kw):
        a = dict(ok, **kw)
        return f(A, A, A, SEQ, early, A, None, a["B"], a["H_q"], a["H_kv"], a["max_len"], a["d"],
                 a["scale"], None)

    assert call(early=None) == 1
    assert call(early=ctypes.c_void_p(0x30002)) == 1
    assert call(H_q=6, H_kv=4) == 1
    assert call(d=48) == 2


def test_strided_validation():
    f = ops.load().gqa_attn_fwd_strided
    dims = dict(B=2, H_q=8, H_kv=2, N_q=300, N_kv=300, d=128, causal=1, scale=0.088)
    # packed [B][H][N][d] strides
    qs = (8 * 300 * 128, 300 * 128, 128)
    ks = (2 * 300 * 128, 300 * 128, 128)

    def call(q=A, k=A, v=A, o=A, q_st=qs, k_st=ks, v_st=ks, o_st=qs, **kw):
        a = dict(dims, **kw)
        return f(q, *q_st, k, *k_st, v, *v_st, o, *o_st, a["B"], a["H_q"], a["H_kv"], a["N_q"],
                 a["N_kv"], a["d"], a["causal"], a["scale"], None)

    assert call(q=None) == 1
    assert call(o=MIS) == 1
    assert call(q_st=(qs[0], qs[1], 100)) == 1       # row stride below d
    assert call(k_st=(ks[0], 12, 128)) == 1           # head stride not a multiple of 8
    assert call(v_st=(0, ks[1], 128)) == 1            # zero batch stride
    assert call(o_st=(qs[0], qs[1], -128)) == 1       # negative row stride
    assert call(d=80) == 2
    assert call(causal=1, N_q=400, N_kv=300) == 2
    assert call(H_q=6, H_kv=4) == 1
