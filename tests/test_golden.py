"""Regression check of the oracle against the stored fixtures in tests/golden
(written by tests/golden/make_golden.py, which calls only the oracle)."""
import json
import os

import numpy as np
import pytest

from tests.golden.make_golden import small_stochastic, tiny_greedy

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name,fn", [("tiny_greedy.json", tiny_greedy),
                                     ("small_stochastic.json", small_stochastic)])
def test_golden_fixture(orc, name, fn):
    with open(os.path.join(HERE, name)) as f:
        stored = json.load(f)
    now = fn()
    if now["input_sha256"] != stored["input_sha256"]:
        pytest.skip("seeded generator produced different inputs on this numpy build")
    for key, val in stored.items():
        if key in ("workload", "input_sha256"):
            continue
        if key == "row_lse":
            np.testing.assert_allclose(now[key], val, rtol=1e-13)
        else:
            assert now[key] == val, key
