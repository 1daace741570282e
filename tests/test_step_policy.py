"""Parity of the library's adaptive draft-step controller (host code behind
the C ABI, include/spec_step.h) with the oracle, on CPU.

Closed-loop runs: each batch drafts with the step the controller chose,
accepted lengths follow a drifting per-position acceptance rate, and the
costs come from SPS and additive tables.  Decisions must be identical; the
windowed prefix acceptance and the scores bit-identical (both sides take the
same fp64 operations).
"""
import math

import numpy as np
import pytest

from oracle.step_policy import StepController as OracleController
from oracle.step_policy import step_cost_additive as o_additive
from oracle.step_policy import step_cost_sps as o_sps


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_ragged_gb300 as sv
    sv.build()
    return sv


def _counters(a, k_per_request, k_max):
    acc = np.array([(a > j).sum() for j in range(k_max)], np.int64)
    ver = np.array([(k_per_request > j).sum() for j in range(k_max)], np.int64)
    return acc, ver


def _tables(rng, k_max):
    g = np.cumsum(rng.integers(1, 64, size=int(rng.integers(2, 8)))).astype(np.int32)
    sps = np.sort(rng.uniform(20, 400, size=g.size))[::-1].copy()
    bb = np.cumsum(rng.integers(1, 32, size=int(rng.integers(1, 5)))).astype(np.int32)
    alpha = rng.uniform(0, 2e-3, size=bb.size)
    theta = np.sort(rng.uniform(1e-3, 2e-2, size=g.size))
    return g, sps, bb, alpha, theta


@pytest.mark.parametrize("seed", range(12))
def test_closed_loop_parity(sv, seed):
    rng = np.random.default_rng(seed)
    k_max = int(rng.integers(1, 9))
    k_min = int(rng.integers(0, k_max + 1))
    k_init = int(rng.integers(k_min, k_max + 1))
    policy = dict(window_size=int(rng.integers(1, 30)), update_interval=int(rng.integers(1, 7)),
                  switch_min_gain=float(rng.choice([0.0, 0.05, 0.2])))
    lib = sv.StepController(k_min, k_max, k_init, **policy)
    orc = OracleController(k_min, k_max, k_init, **policy)
    g, sps, bb, alpha, theta = _tables(rng, k_max)
    k = k_init
    switches = 0
    for t in range(120):
        B = int(rng.integers(1, 40))
        alpha_t = 0.5 + 0.45 * math.sin(t / 9.0 + seed)         # drifting acceptance
        ragged = rng.random() < 0.2
        kb = rng.integers(0, k + 1, size=B) if ragged else np.full(B, k)
        a = np.minimum(rng.geometric(1 - alpha_t, size=B) - 1, kb)
        acc, ver = _counters(a, kb, k_max)
        if t % 2:
            cost = sv.step_cost_sps(B, k_max, g, sps)
            ref_cost = o_sps(B, k_max, list(g), list(sps))
        else:
            cost = sv.step_cost_additive(B, k_max, 2e-3, bb, alpha, g, theta)
            ref_cost = o_additive(B, k_max, 2e-3, list(bb), list(alpha), list(g), list(theta))
        np.testing.assert_array_equal(cost, np.array(ref_cost))
        k_new = lib.update(acc, ver, cost, B)
        assert k_new == orc.update(acc, ver, ref_cost, B), t
        switches += k_new != k
        k = k_new
        pa, score, kc = lib.query()
        assert kc == k
        np.testing.assert_array_equal(pa, np.array(orc.prefix_acceptance))
        np.testing.assert_array_equal(score, np.array(orc.score))
    if k_max > k_min and policy["switch_min_gain"] == 0.0:
        assert switches > 0                      # the drift moves the step


def test_page_defaults_follow_a_regime_change(sv):
    """Window 20, re-scoring every 5, gain 5 %: high acceptance pushes the
    step up, a collapse brings it down within one window."""
    lib = sv.StepController(1, 5, 3)
    orc = OracleController(1, 5, 3)
    B = 32
    cost = [10.0 + 2.0 * k for k in range(6)]
    hist = []
    for t in range(60):
        k = hist[-1] if hist else 3
        a = np.full(B, k) if t < 30 else np.zeros(B, np.int64)
        acc, ver = _counters(a, np.full(B, k), 5)
        k1 = lib.update(acc, ver, cost, B)
        assert k1 == orc.update(acc, ver, cost, B)
        hist.append(k1)
    assert hist[4] == 5 and hist[29] == 5               # all accepted: the longest step
    assert hist[-1] == 1                                 # nothing accepted: the shortest
    assert all(h == hist[i - 1] for i, h in enumerate(hist) if i % 5 != 4 and i > 0)


def test_rejected_inputs_leave_the_state_alone(sv):
    from speculative_decoding_verification_ragged_gb300 import SpecError
    lib = sv.StepController(0, 2, 1, update_interval=2)
    orc = OracleController(0, 2, 1, update_interval=2)
    for acc, ver in [([3, 1], [2, 2]), ([1, 2], [2, 2]), ([1, 1], [1, 2]), ([-1, 0], [1, 0])]:
        with pytest.raises(SpecError):
            lib.update(acc, ver, [1.0] * 3, 2)
    assert lib.update([1, 0], [2, 0], [1.0] * 3, 2) == orc.update([1, 0], [2, 0], [1.0] * 3, 2)
    with pytest.raises(SpecError):                   # due now: a bad cost is rejected
        lib.update([2, 1], [2, 2], [1.0, float("nan"), 1.0], 2)
    with pytest.raises(SpecError):
        lib.update([2, 1], [2, 2], [1.0, 0.0, 1.0], 2)
    with pytest.raises(SpecError):
        lib.update([2, 1], [2, 2], [1.0] * 3, 0)
    k = lib.update([2, 1], [2, 2], [1.0, 0.5, 0.25], 2)
    assert k == orc.update([2, 1], [2, 2], [1.0, 0.5, 0.25], 2)
    np.testing.assert_array_equal(lib.query()[1], np.array(orc.score))
    for args in [(2, 1, 1), (0, 32, 1), (0, 3, 4)]:
        with pytest.raises(SpecError):
            sv.StepController(*args)
    with pytest.raises(SpecError):
        sv.StepController(0, 3, 1, window_size=65)
    with pytest.raises(SpecError):
        sv.StepController(0, 3, 1, switch_min_gain=-0.1)
    with pytest.raises(SpecError):
        sv.step_cost_sps(8, 3, [8, 8], [1.0, 1.0])
    with pytest.raises(SpecError):
        sv.step_cost_sps(8, 3, [8, 16], [1.0, 0.0])
    with pytest.raises(SpecError):
        sv.step_cost_additive(8, 3, float("inf"), [8], [0.0], [8], [0.0])


def test_abi_state_checks(sv):
    import ctypes as C
    L = sv.load_library()
    n = L.spec_step_state_bytes()
    assert n > 0
    buf = np.zeros(n // 8 + 2, np.uint64)
    pol = sv.binding.StepPolicy(0, 3, 1, 20, 5, 0.05)
    p = buf.ctypes.data_as(C.c_void_p)
    assert L.spec_step_init(p, n - 1, C.byref(pol)) == 1
    assert L.spec_step_init(C.c_void_p(buf.ctypes.data + 4), n, C.byref(pol)) == 1
    k = C.c_int32(-1)
    assert L.spec_step_update(p, None, None, None, 4, C.byref(k)) == 1     # not initialised
    assert L.spec_step_init(p, n, C.byref(pol)) == 0
    assert L.spec_step_query(p, None, None, C.byref(k)) == 0 and k.value == 1
    assert L.spec_step_update(p, None, None, None, 4, C.byref(k)) == 1     # k_max 3: counters
    acc = np.array([2, 1, 0], np.int64)
    ver = np.array([4, 4, 4], np.int64)
    assert L.spec_step_update(p, acc.ctypes.data_as(C.c_void_p), ver.ctypes.data_as(C.c_void_p),
                              None, 4, C.byref(k)) == 0                   # not due: no costs
    assert k.value == 1


def test_bench_times_the_controller_on_the_host(sv):
    """The benchmark's controller timing runs without a GPU and ends on a
    valid step."""
    import bench
    r = bench.time_step_controller(sv, batches=200)
    assert r["batches"] == 200 and 1 <= r["k_final"] <= 5
    assert r["us_per_batch_c_call"] > 0 and r["us_per_batch_binding"] > 0
