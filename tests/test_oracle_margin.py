"""Pins for the oracle's confidence-margin acceptance.

The margin loosens greedy acceptance (vSpec README §"启动" approximate
acceptance preset, §"通用参数" --confidence-accept-margin and its position,
token-count and protected-id options).  Each pin checks the oracle against
something other than itself: hand-worked rows, the special cases that reduce
to the separately pinned greedy and relaxed top-K rules, and invariants.
"""
import numpy as np
import pytest

import workloads as W


# row0: max 5 at index 1, draft 2 sits 1.5 below it
# row1: max 2 at index 0, draft 2 sits 0.75 below it
# row2: bonus row, argmax 3
Z = np.array([[0, 5, 3.5, 1, 4], [2, 0, 1.25, 0, 0], [0, 0, 0, 9, 0]], dtype=np.float32)
CU = np.array([0, 3])
D = np.array([2, 2, -1])


def _run(orc, margin, **kw):
    return orc.verify_margin(Z, "f32", 5, 1, 2, CU, D, np.array([margin], np.float32), **kw)


def test_margin_worked_example(orc):
    r = _run(orc, 1.5)                       # both gaps (1.5, 0.75) within the margin
    assert r.accepted_len.tolist() == [2] and r.out_tokens.tolist() == [[2, 2, 3]]
    assert r.status == 0
    r = _run(orc, 1.0)                       # row0's gap 1.5 > 1: stop there, emit its argmax
    assert r.accepted_len.tolist() == [0] and r.out_tokens.tolist() == [[1, -1, -1]]
    r = _run(orc, 1.49)
    assert r.accepted_len.tolist() == [0] and r.next_token.tolist() == [1]
    r = _run(orc, 0.75)                      # row0 fails first even though row1 would pass
    assert r.accepted_len.tolist() == [0]
    assert r.rows["row_ok"].tolist() == [0, 1, 0]          # the bonus row has no draft


def test_margin_positions_and_token_count(orc):
    # position 0 kept strict: the draft 2 is not row0's argmax
    assert _run(orc, 1.5, from_position=1).accepted_len.tolist() == [0]
    # 3 tokens generated before this step: position j is output token 3 + j
    gen = np.array([3], np.int32)
    assert _run(orc, 1.5, generated=gen, after_tokens=4).accepted_len.tolist() == [0]
    r = _run(orc, 1.5, generated=gen, after_tokens=3)
    assert r.accepted_len.tolist() == [2] and r.next_token.tolist() == [3]
    # without a count of generated tokens, position j itself is the count
    assert _run(orc, 1.5, after_tokens=1).accepted_len.tolist() == [0]


def test_margin_protected_ids(orc):
    assert _run(orc, 1.5, protected_ids=np.array([2])).accepted_len.tolist() == [0]
    assert _run(orc, 1.5, protected_ids=np.array([7, 0, 4])).accepted_len.tolist() == [2]
    # a protected draft that is the argmax is still accepted (strict rule)
    r = orc.verify_margin(Z, "f32", 5, 1, 2, CU, np.array([1, 0, -1]), np.array([1.5], np.float32),
                          protected_ids=np.array([0, 1]))
    assert r.accepted_len.tolist() == [2] and r.next_token.tolist() == [3]


def test_margin_gap_is_rounded_to_fp32(orc):
    # max 2^25 and draft value 3: the exact gap 33554429 lies halfway between
    # the fp32 neighbours 33554428 and 33554430 and rounds to even, 33554428
    z = np.array([[2.0 ** 25, 3, 0, 0], [0, 1, 0, 0]], dtype=np.float32)
    cu, d = np.array([0, 2]), np.array([1, -1])
    ok = orc.verify_margin(z, "f32", 4, 1, 1, cu, d, np.array([33554428.0], np.float32))
    assert ok.accepted_len.tolist() == [1] and ok.next_token.tolist() == [1]
    no = orc.verify_margin(z, "f32", 4, 1, 1, cu, d, np.array([33554426.0], np.float32))
    assert no.accepted_len.tolist() == [0] and no.next_token.tolist() == [0]


def test_margin_bad_values_and_out_of_vocab(orc):
    r = _run(orc, float("nan"))
    assert r.status & orc.BAD_MARGIN
    assert r.accepted_len.tolist() == [0]
    z = np.array([[1, 2, 3], [3, 2, 1]], dtype=np.float32)
    r = orc.verify_margin(z, "f32", 3, 1, 1, np.array([0, 2]), np.array([7, -1]),
                          np.array([np.inf], np.float32))
    assert r.status == 0 and r.accepted_len.tolist() == [0] and r.next_token.tolist() == [2]


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_margin_special_cases_reduce_to_pinned_rules(orc, seed, dtype):
    vb = W.ragged_batch(20 + seed, B=9, k_max=6, V=700, dtype=dtype, tie_top=(seed != 1), p_top=0.5)
    args = (vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    g = orc.verify_greedy(*args)
    # a negative margin, or every token protected, is strict greedy
    for kw in [dict(margin=np.full(vb.B, -1.0, np.float32)),
               dict(margin=np.full(vb.B, 1e30, np.float32), protected_ids=np.arange(vb.V))]:
        m = orc.verify_margin(*args, **kw)
        np.testing.assert_array_equal(m.out_tokens, g.out_tokens)
        np.testing.assert_array_equal(m.accepted_len, g.accepted_len)
    # margin 0 accepts exactly the drafts with no larger logit: relaxed K = 1
    m0 = orc.verify_margin(*args, margin=np.zeros(vb.B, np.float32))
    r1 = orc.verify_relaxed(*args, np.ones(vb.B, np.int32))
    np.testing.assert_array_equal(m0.out_tokens, r1.out_tokens)
    # an infinite margin accepts every in-vocabulary draft: relaxed K = V
    mi = orc.verify_margin(*args, margin=np.full(vb.B, np.inf, np.float32))
    rv = orc.verify_relaxed(*args, np.full(vb.B, vb.V, np.int32))
    np.testing.assert_array_equal(mi.out_tokens, rv.out_tokens)


def test_margin_monotone(orc):
    vb = W.ragged_batch(31, B=40, k_max=5, V=300, dtype="bf16", p_top=0.3)
    args = (vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    prev = None
    for mg in [0.0, 0.5, 1.0, 2.0, 4.0, 8.0]:
        a = orc.verify_margin(*args, margin=np.full(vb.B, mg, np.float32)).accepted_len
        if prev is not None:
            assert (a >= prev).all()
        prev = a
    assert prev.sum() > orc.verify_greedy(*args).accepted_len.sum()
    prev = None
    for fp in range(0, 7):
        a = orc.verify_margin(*args, margin=np.full(vb.B, 4.0, np.float32),
                              from_position=fp).accepted_len
        if prev is not None:
            assert (a <= prev).all()
        prev = a
    # the chain keeps its shape: drafts up to a, then the stopping row's argmax
    m = orc.verify_margin(*args, margin=np.full(vb.B, 2.0, np.float32))
    am = m.rows["row_argmax"]
    for b in range(vb.B):
        r0, a = int(vb.cu_rows[b]), int(m.accepted_len[b])
        assert m.out_tokens[b, :a].tolist() == vb.draft_ids[r0:r0 + a].tolist()
        assert m.next_token[b] == am[r0 + a] == m.out_tokens[b, a]
        assert m.rows["row_ok"][r0:r0 + a].all()
