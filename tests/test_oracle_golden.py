"""The oracle against the hand-derived worked examples in tests/golden/ (CPU only).

Each example cites the passage of the KIVI page (or the reading of it) that fixes
its result, and carries its derivation; the expected values are derived by hand,
not produced by the oracle or the CUDA path.
"""
import json
import os

import numpy as np
import pytest

import oracle

FX = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


@pytest.mark.parametrize("ex", FX["quantize_group"], ids=lambda e: e["name"])
def test_quantize_group_worked_examples(ex):
    s, z, codes = oracle.quantize_group(np.array(ex["x"], np.float16), bits=ex["bits"])
    assert (s, z) == (ex["s16"], ex["z16"]), ex["derivation"]
    assert codes.tolist() == ex["codes"], ex["derivation"]


@pytest.mark.parametrize("ex", FX["pack_row"], ids=lambda e: e["name"])
def test_pack_row_worked_examples(ex):
    assert oracle.pack_row(np.array(ex["codes"], np.uint8), bits=ex["bits"]).tolist() == ex["words"]


@pytest.mark.parametrize("ex", FX["attention"], ids=lambda e: e["name"])
def test_attention_worked_examples(ex):
    D, G = ex["D"], ex["G"]
    k = np.array(ex["k"], np.float16)[None, None]
    v = np.array(ex["v"], np.float16)[None, None]
    q = np.array(ex["q"], np.float16)[None, None]
    c = oracle.prefill(k, v, G, k.shape[2])
    out = oracle.attention(c, q, ex["sigma"])
    assert np.allclose(out[0, 0], np.array(ex["out"]), rtol=0, atol=ex["atol"]), ex["derivation"]
