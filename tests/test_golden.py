"""Regression check of the oracle against the stored fixtures in tests/golden
(written by tests/golden/make_golden.py, which calls only the oracle), and of
the step controller against the values the pages print
(tests/golden/page_step_controller.json, with its citation)."""
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


def test_page_values_of_the_step_controller():
    import inspect
    import speculative_decoding_verification_ragged_gb300 as sv
    from oracle.step_policy import StepController, step_cost_sps
    with open(os.path.join(HERE, "page_step_controller.json")) as f:
        page = json.load(f)
    d = page["policy_defaults"]
    for cls in (StepController, sv.StepController):
        sig = inspect.signature(cls.__init__).parameters
        for key in ("window_size", "update_interval", "switch_min_gain"):
            assert sig[key].default == d[key], (cls, key)
    # the bucket example: with exactly the page's graphs captured, the rows
    # of steps k = 0, 1, 3 and 5 (B, 2B, 4B, 6B) bind those graphs in order
    ex = page["bucket_example"]
    g = ex["graph_rows"]
    sps = [1000.0 / (i + 1) for i in range(len(g))]          # cost i + 1 ms marks graph i
    for cost in (step_cost_sps(ex["B"], ex["draft_width"], g, sps),
                 list(sv.step_cost_sps(ex["B"], ex["draft_width"], g, sps))):
        chosen = [g[int(round(cost[k])) - 1] for k in (0, 1, 3, 5)]
        assert chosen == ex["graph_rows"]
        assert [ex["B"] * (k + 1) for k in (0, 1, 3, 5)] == ex["rows_covered"]
