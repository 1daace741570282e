"""Pins for the oracle of the adaptive draft-step controller (xLLM
"自适应投机推理" §"自适应 draft 步长（MTP）", §"可选的步长配置文件",
§"成本模型与覆盖范围").

Each pin checks the oracle against something other than itself: the page's
worked bucket example, closed forms of the objective (every draft accepted:
B (1 + k) / cost(k); i.i.d. acceptance 1/2: B (2 - 2^-k) / cost(k)), and
hand-worked windows, intervals, ties and gains.
"""
import math

import pytest

from oracle.step_policy import StepController, step_cost_additive, step_cost_sps


def test_sps_buckets_follow_the_page_example():
    # B = 8 with 5 drafts binds target graphs G = 8, 16, 32, 48 for the rows
    # of B, 2B, 4B and B (5 + 1)
    g = [8, 16, 32, 48]
    sps = [400.0, 250.0, 125.0, 80.0]
    c = step_cost_sps(8, 6, g, sps)
    assert c[:6] == [2.5, 4.0, 8.0, 8.0, 12.5, 12.5]     # rows 8 16 24 32 40 48
    assert c[6] == math.inf                               # 56 rows: no captured graph


def test_additive_costs_by_hand():
    c = step_cost_additive(5, 3, 0.001, [4, 8, 16], [0.0005, 0.001, 0.002],
                           [8, 16, 32], [0.002, 0.003, 0.005])
    # Bcap = 8; rows 5 10 15 20 -> G = 8 16 16 32
    assert c == pytest.approx([4.0, 5.0, 5.0, 7.0], rel=1e-15)
    assert step_cost_additive(17, 1, 0.0, [4, 8, 16], [0, 0, 0], [64], [1e-3]) == [math.inf] * 2
    with pytest.raises(ValueError):
        step_cost_additive(5, 1, 0.0, [8, 4], [0, 0], [8], [0])


def _feed(ctl, n, acc, ver, cost, B):
    return [ctl.update(acc, ver, cost, B) for _ in range(n)]


def test_all_accepted_closed_form():
    # acc = ver: prefix acceptance 1, so score(k) = B (1 + k) / cost(k)
    B, K = 64, 5
    cost = [10.0 + k for k in range(K + 1)]
    ctl = StepController(1, K, 1)
    ks = _feed(ctl, 5, [B] * K, [B] * K, cost, B)
    assert ks == [1, 1, 1, 1, 5]                 # re-scored at the 5th batch only
    assert ctl.prefix_acceptance == [1.0] * K
    for k in range(1, K + 1):
        assert ctl.score[k] == B * (1 + k) / (10.0 + k)
    assert ctl.score[0] == 0.0                    # below k_min


@pytest.mark.parametrize("k_init,expect", [(2, 5), (4, 4), (3, 5)])
def test_geometric_acceptance_and_the_switch_gain(k_init, expect):
    # half of the prefixes survive each position: pa[j] = 2^-(j+1) and, at
    # constant cost, score(k) = B (2 - 2^-k).  From k = 2 the best (k = 5)
    # gains 12.5 %: switch.  From k = 4 it gains 1.6 %: hold.  From k = 3 the
    # gain is 5 % exactly in real numbers, which 1.05 (not a binary fraction)
    # cannot decide, so there k = 5 is made 0.1 % cheaper (gain 5.1 %)
    B = 1024
    acc, ver = [512, 256, 128, 64, 32], [1024] * 5
    cost = [1.0] * 6
    if k_init == 3:
        cost[5] = 0.999
    ctl = StepController(0, 5, k_init)
    assert _feed(ctl, 5, acc, ver, cost, B)[-1] == expect
    for j in range(5):
        assert ctl.prefix_acceptance[j] == 2.0 ** -(j + 1)
    assert ctl.score[4] == B * (2 - 2.0 ** -4)


def test_gain_equal_to_the_threshold_does_not_switch():
    # every draft accepted: score(1) = 2B / cost(1), score(0) = B / cost(0).
    # With gain 1 (a binary fraction) equal costs give a ratio of exactly 2:
    # the gain is not exceeded.  A 0.1 % cheaper k = 1 exceeds it.
    B = 16
    ctl = StepController(0, 1, 0, update_interval=1, switch_min_gain=1.0)
    assert ctl.update([B], [B], [1.0, 1.0], B) == 0
    assert ctl.score == [B, 2 * B]
    assert ctl.update([B], [B], [1.0, 0.999], B) == 1


def test_window_forgets_old_batches():
    B, K = 8, 3
    cost = [1.0 + k for k in range(K + 1)]        # more drafts cost more
    ctl = StepController(0, K, K)
    ks = _feed(ctl, 20, [B] * K, [B] * K, cost, B)          # all accepted
    # score(k) = B (1 + k) / (1 + k) = B for every k: ties keep k = 3
    assert ks[-1] == 3 and ctl.score == [B] * (K + 1)
    ks = _feed(ctl, 5, [0] * K, [B] * K, cost, B)           # nothing accepted
    # window = 15 all-accepted batches + 5 none: pa = 15/20 = 0.75 everywhere
    assert ctl.prefix_acceptance == [0.75] * K
    assert ctl.score == [B / 1.0, B * 1.75 / 2, B * 2.5 / 3, B * 3.25 / 4]
    # best k = 0 (8 > 7 > 6.67 > 6.5): gain 8 / 6.5 - 1 = 23 % > 5 %
    assert ks[-1] == 0
    _feed(ctl, 15, [0] * K, [B] * K, cost, B)
    assert ctl.prefix_acceptance == [0.0] * K               # the old regime is gone


def test_unverified_positions_extrapolate():
    # only positions 0 and 1 verified (k = 2): pa = [0.8, 0.64], rate 0.8
    ctl = StepController(1, 5, 2)
    _feed(ctl, 5, [80, 64, 0, 0, 0], [100, 100, 0, 0, 0], [1.0] * 6, 10)
    assert ctl.prefix_acceptance == pytest.approx([0.8, 0.64, 0.512, 0.4096, 0.32768],
                                                  rel=1e-15)
    # only position 0 verified: pa[j] = 0.6^(j+1)
    ctl = StepController(1, 4, 1)
    _feed(ctl, 5, [60, 0, 0, 0], [100, 0, 0, 0], [1.0] * 5, 10)
    assert ctl.prefix_acceptance == pytest.approx([0.6, 0.36, 0.216, 0.1296], rel=1e-15)
    # a verified position with no acceptance ends the tail
    ctl = StepController(1, 4, 2)
    _feed(ctl, 5, [0, 0, 0, 0], [100, 100, 0, 0], [1.0] * 5, 10)
    assert ctl.prefix_acceptance == [0.0] * 4


def test_empty_window_and_infeasible_steps():
    ctl = StepController(0, 3, 2)
    assert _feed(ctl, 5, [0, 0, 0], [0, 0, 0], [1.0] * 4, 4)[-1] == 2   # nothing verified
    assert ctl.score == [0.0] * 4
    # the current k is not covered by any captured graph: any feasible k wins
    ctl = StepController(0, 3, 3)
    inf = math.inf
    assert _feed(ctl, 5, [4, 2, 1], [4, 4, 4], [1.0, 1.5, inf, inf], 4)[-1] == 1
    # ties go to the smaller k: pa = 1, cost(k) = 1 + k gives B for every k
    ctl = StepController(1, 3, 1, update_interval=1)
    assert ctl.update([4] * 3, [4] * 3, [1.0, 2.0, 3.0, 4.0], 4) == 1


def test_invalid_batches_are_rejected():
    ctl = StepController(0, 2, 1)
    for acc, ver in [([3, 1], [2, 2]), ([1, 2], [2, 2]), ([1, 1], [1, 2]), ([-1, 0], [1, 0])]:
        with pytest.raises(ValueError):
            ctl.update(acc, ver, [1.0] * 3, 2)
    with pytest.raises(ValueError):
        ctl.update([1, 0], [1, 0], [1.0] * 3, 0)
    with pytest.raises(ValueError):
        StepController(2, 1, 1)
    with pytest.raises(ValueError):
        StepController(0, 3, 1, window_size=65)
    assert ctl.batches == []
