"""Writes worked_examples.json: worked examples derived by hand from the rule each
cites (see each entry's 'derivation').  It calls neither the oracle nor the CUDA
library; the only arithmetic here is the derivation's own (the attention output
v0/4 + 3 v1/4).  Run from the repository root: python tests/golden/make_worked_examples.py
"""
import json
import math
import os

v0 = [float(i % 4) for i in range(16)]  # 0,1,2,3,... : min 0, max 3 -> s = 1
v1 = [3.0 if i < 8 else 0.0 for i in range(16)]  # 3 x8, 0 x8 : min 0, max 3 -> s = 1
out = [0.25 * a + 0.75 * b for a, b in zip(v0, v1)]

FX = {
    "about": ("Worked examples whose results the quantization rule and the attention definition fix exactly. "
              "The page prints no worked example or table (it is prose only), so every value here is derived by "
              "hand in its 'derivation' field from the rule it cites; none comes from the oracle or the CUDA path."),
    "source": "KIVI page 'Makale Bulteni -- KIVI' (cmlonder.com radar / paper-to-prod, 2026-11-01)",
    "quantize_group": [
        {"name": "four levels on a 0.5 grid",
         "citation": "headline paragraph (asymmetric 2-bit: zero = min, scale = (max - min)/3); "
                     "section 'Iddia ve Gerceklik' paragraph 2",
         "bits": 2, "x": [-1.0, -0.5, 0.0, 0.5],
         "derivation": "min = -1, max = 0.5, s = 1.5/3 = 0.5 (fp16 0x3800), z = -1 (fp16 0xBC00); "
                       "(x - min)/s = 0, 1, 2, 3",
         "s16": 0x3800, "z16": 0xBC00, "codes": [0, 1, 2, 3]},
        {"name": "half-way values round to even",
         "citation": "headline paragraph; rounding to nearest with ties to even (reading R3)",
         "bits": 2, "x": [0.0, 0.25, 0.75, 1.25, 1.5],
         "derivation": "min = 0, max = 1.5, s = 0.5 (0x3800), z = 0; (x - min)/s = 0, 0.5, 1.5, 2.5, 3 "
                       "-> 0, 0, 2, 2, 3",
         "s16": 0x3800, "z16": 0, "codes": [0, 0, 2, 2, 3]},
        {"name": "constant group",
         "citation": "headline paragraph; a zero range gives scale 0 and all codes 0 (reading R3)",
         "bits": 2, "x": [2.0, 2.0, 2.0],
         "derivation": "min = max = 2, s = 0 (0x0000), z = 2 (0x4000), codes 0",
         "s16": 0, "z16": 0x4000, "codes": [0, 0, 0]},
        {"name": "signed zeros",
         "citation": "headline paragraph; a zero point of -0 is stored as +0 (reading R4)",
         "bits": 2, "x": [-0.0, 0.0],
         "derivation": "min = -0 = max, s = 0, z = +0 (0x0000), codes 0",
         "s16": 0, "z16": 0, "codes": [0, 0]},
        {"name": "sixteen levels on a unit grid (4-bit variant)",
         "citation": "reading R10: the same rule with 2^4 - 1 = 15 levels",
         "bits": 4, "x": [float(i) for i in range(16)],
         "derivation": "min = 0, max = 15, s = 15/15 = 1 (0x3C00), z = 0; (x - min)/s = 0 .. 15",
         "s16": 0x3C00, "z16": 0, "codes": list(range(16))},
    ],
    "pack_row": [
        {"name": "2-bit codes 0,1,2,3 repeated",
         "citation": "reading R7: channel 16w+i in bits [2i, 2i+1] of word w",
         "bits": 2, "codes": [0, 1, 2, 3] * 4,
         "derivation": "byte = 0 | 1<<2 | 2<<4 | 3<<6 = 0xE4, four times",
         "words": [0xE4E4E4E4]},
        {"name": "4-bit codes 0..7",
         "citation": "reading R10: channel 8w+i in bits [4i, 4i+3] of word w",
         "bits": 4, "codes": list(range(8)),
         "derivation": "nibble i holds i: 0x76543210",
         "words": [0x76543210]},
    ],
    "attention": [
        {"name": "two tokens, weights 1/4 and 3/4",
         "citation": "section 'Iddia ve Gerceklik' paragraph 2 (the output is a weighted sum of values); reading R8",
         "D": 16, "G": 2, "sigma": math.log(3.0) / 0.75,
         "k": [[0.0] * 16, [0.75] + [0.0] * 15],
         "v": [v0, v1],
         "q": [1.0] + [0.0] * 15,
         "derivation": ("keys: channel 0 spans 0..0.75 = 3 * 0.25, so s = 0.25 and both keys dequantize exactly; "
                        "the other channels are constant 0. Values: each token spans 0..3, s = 1, exact. Scores: "
                        "sigma * q.k = 0 and sigma * 0.75 = ln 3, so softmax = (1/4, 3/4) and out = v0/4 + 3 v1/4"),
         "out": out, "atol": 1e-12},
    ],
}

if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_examples.json")
    with open(path, "w") as f:
        json.dump(FX, f, indent=1)
