"""The oracle against the hand-derived closed forms in tests/golden/closed_forms.json."""
import json
import os

import numpy as np
import pytest

import oracle

_CASES = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))["cases"]


@pytest.mark.parametrize("case", _CASES, ids=[f"{c['op']}-{i}" for i, c in enumerate(_CASES)])
def test_oracle_matches_closed_form(case):
    x = np.array(case["x"], np.float32)
    atol = case.get("atol", 1e-15)
    op = case["op"]
    if op == "softmax":
        got = oracle.softmax(x)
    elif op == "layernorm":
        g = None if "gamma" not in case else np.array(case["gamma"], np.float32)
        b = None if "beta" not in case else np.array(case["beta"], np.float32)
        got = oracle.layernorm(x, g, b, case["eps"])
    elif op == "rmsnorm":
        w = None if "w" not in case else np.array(case["w"], np.float32)
        got = oracle.rmsnorm(x, w, case["eps"])
    else:
        got = oracle.cross_entropy(x, np.array(case["labels"], np.int64))
    assert np.allclose(got, np.array(case["expect"]), rtol=1e-15, atol=atol)
