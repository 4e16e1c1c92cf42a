"""Writes the closed-form fixtures in this folder.

Every expected value here is derived by hand from the definition of attention
(softmax-weighted average of V rows) on inputs chosen so the softmax weights
are small rationals: scores such as [0, ln 3] give weights [1/4, 3/4]. The
script imports nothing from the oracle or from the CUDA library; it only
spells the hand derivations out as numbers (ln values and rationals).

Run:  python tests/golden/make_closed_form_fixtures.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
ln2, ln3, ln5 = math.log(2), math.log(3), math.log(5)

FIXTURES = {
    "two_keys_quarter_threequarter.json": {
        "source": "BootstrapAI evolution log, collab-005 'Kernel 2 tiling' (softmax-weighted "
                  "average of V) and collab-014 'Kernel 9 GQA' (MHA case, group size 1)",
        "derivation": "scale=1, q=[1,0]: scores q.k = [0, ln 3]; exp -> [1, 3], sum 4, weights "
                      "[1/4, 3/4]; O = v0/4 + 3 v1/4 = [1+6, -2+3] = [7, 1]; lse = ln 4. With "
                      "q=[0,1] both scores are 0, so O = mean(v) = [6, -2], lse = ln 2. Causal "
                      "row 0 sees key 0 only: O = v0 = [4, -8], lse = 0 (q=[1,0]).",
        "B": 1, "H_q": 1, "H_kv": 1, "d": 2, "scale": 1.0,
        "q": [[[[1.0, 0.0], [0.0, 1.0]]]],
        "k": [[[[0.0, 0.0], [ln3, 0.0]]]],
        "v": [[[[4.0, -8.0], [8.0, 4.0]]]],
        "expect": {
            "full": {"o": [[[[7.0, 1.0], [6.0, -2.0]]]], "lse": [[[math.log(4), math.log(2)]]]},
            "causal": {"o": [[[[4.0, -8.0], [6.0, -2.0]]]], "lse": [[[0.0, math.log(2)]]]},
        },
    },
    "three_keys_scaled.json": {
        "source": "BootstrapAI evolution log, collab-005 'Kernel 2 tiling' (softmax-weighted "
                  "average of V); the scale multiplies the raw dot product",
        "derivation": "scale=0.5, q=[2,0]: raw dots [0, 2 ln 2, 2 ln 5] -> scores [0, ln 2, ln 5]; "
                      "exp -> [1, 2, 5], sum 8; O = (1*[8,0] + 2*[0,8] + 5*[16,-16]) / 8 = "
                      "[88, -64]/8 = [11, -8]; lse = ln 8. q=[0,2]: scores all 0, O = mean(v) = "
                      "[8, -8/3], lse = ln 3.",
        "B": 1, "H_q": 1, "H_kv": 1, "d": 2, "scale": 0.5,
        "q": [[[[2.0, 0.0], [0.0, 2.0]]]],
        "k": [[[[0.0, 0.0], [ln2, 0.0], [ln5, 0.0]]]],
        "v": [[[[8.0, 0.0], [0.0, 8.0], [16.0, -16.0]]]],
        "expect": {
            "full": {"o": [[[[11.0, -8.0], [8.0, -8.0 / 3.0]]]],
                     "lse": [[[math.log(8), math.log(3)]]]},
        },
    },
    "gqa_head_mapping.json": {
        "source": "BootstrapAI evolution log, collab-014 'Kernel 9 GQA': h_kv = h_q / group_size "
                  "with group_size = H_q / H_kv",
        "derivation": "H_q=4, H_kv=2, group 2: heads 0,1 read K/V head 0; heads 2,3 read K/V head "
                      "1. KV head 0: k=[[0,0],[ln3,0]], v=[[4,-8],[8,4]]; KV head 1: "
                      "k=[[0,0],[0,ln3]], v=[[0,4],[4,0]]. Head 0 (q=[1,0]) -> weights "
                      "[1/4,3/4] -> [7,1]. Head 1 (q=[0,1]) -> scores [0,0] -> mean [6,-2]. "
                      "Head 2 (q=[1,0]) -> scores [0,0] -> mean [2,2]. Head 3 (q=[0,1]) -> "
                      "weights [1/4,3/4] -> [0,1]+[3,0] = [3,1]. The modulo mapping "
                      "h_q % H_kv would give [3,1] for head 1 and [7,1] for head 2.",
        "B": 1, "H_q": 4, "H_kv": 2, "d": 2, "scale": 1.0,
        "q": [[[[1.0, 0.0]], [[0.0, 1.0]], [[1.0, 0.0]], [[0.0, 1.0]]]],
        "k": [[[[0.0, 0.0], [ln3, 0.0]], [[0.0, 0.0], [0.0, ln3]]]],
        "v": [[[[4.0, -8.0], [8.0, 4.0]], [[0.0, 4.0], [4.0, 0.0]]]],
        "expect": {
            "full": {"o": [[[[7.0, 1.0]], [[6.0, -2.0]], [[2.0, 2.0]], [[3.0, 1.0]]]],
                     "lse": [[[math.log(4)], [math.log(2)], [math.log(2)], [math.log(4)]]]},
        },
    },
    "bottom_right_causal.json": {
        "source": "Causal alignment for N_q != N_kv is not stated on the pages (microLLM-rocm "
                  "optimisation log, Experiments 044 and 061 use causal GQA with N_q = N_kv); "
                  "the reading taken is bottom-right: row i sees keys j <= i + N_kv - N_q",
        "derivation": "N_q=2, N_kv=3, scale=0.5, both rows q=[2,0], keys and values as in "
                      "three_keys_scaled. Row 0 sees keys 0,1: scores [0, ln 2] -> weights "
                      "[1/3, 2/3] -> O = [8/3, 16/3], lse = ln 3. Row 1 sees all three keys: "
                      "O = [11,-8], lse = ln 8. Top-left alignment would give row 0 = v0 = [8,0].",
        "B": 1, "H_q": 1, "H_kv": 1, "d": 2, "scale": 0.5,
        "q": [[[[2.0, 0.0], [2.0, 0.0]]]],
        "k": [[[[0.0, 0.0], [ln2, 0.0], [ln5, 0.0]]]],
        "v": [[[[8.0, 0.0], [0.0, 8.0], [16.0, -16.0]]]],
        "expect": {
            "causal": {"o": [[[[8.0 / 3.0, 16.0 / 3.0], [11.0, -8.0]]]],
                       "lse": [[[math.log(3), math.log(8)]]]},
        },
    },
    "decode_two_sequences.json": {
        "source": "microLLM-rocm optimisation log, Experiments 064-065 (batched cached GQA "
                  "decode; per-row cache lengths) with the head mapping of BootstrapAI "
                  "evolution log, collab-014 'Kernel 9 GQA'",
        "derivation": "B=2, H_q=2, H_kv=1, max_len=3, scale=1, seqlens=[2,3]. Sequence 0 cache "
                      "k=[[0,0],[ln3,0],pad], v=[[4,-8],[8,4],pad]: head 0 q=[1,0] -> [7,1]; "
                      "head 1 q=[0,1] -> mean [6,-2]. Sequence 1 cache k=[[0,0],[ln2,0],[ln5,0]], "
                      "v=[[8,0],[0,8],[16,-16]]: head 0 q=[1,0] -> weights [1,2,5]/8 -> [11,-8]; "
                      "head 1 q=[0,1] -> mean [8,-8/3]. Pad rows are NaN and must not be read.",
        "B": 2, "H_q": 2, "H_kv": 1, "d": 2, "max_len": 3, "scale": 1.0, "seqlens": [2, 3],
        "q": [[[1.0, 0.0], [0.0, 1.0]], [[1.0, 0.0], [0.0, 1.0]]],
        "k_cache": [[[[0.0, 0.0], [ln3, 0.0], ["nan", "nan"]]],
                    [[[0.0, 0.0], [ln2, 0.0], [ln5, 0.0]]]],
        "v_cache": [[[[4.0, -8.0], [8.0, 4.0], ["nan", "nan"]]],
                    [[[8.0, 0.0], [0.0, 8.0], [16.0, -16.0]]]],
        "expect": {"o": [[[7.0, 1.0], [6.0, -2.0]], [[11.0, -8.0], [8.0, -8.0 / 3.0]]],
                   "lse": [[math.log(4), math.log(2)], [math.log(8), math.log(3)]]},
    },
}


def main():
    for name, fx in FIXTURES.items():
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
