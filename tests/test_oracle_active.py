"""Pins for the oracle's greedy verification over an active vocabulary
(vSpec README §"EAGLE 功能", §"代码所有权": the target LM head scores a
subset of token ids, mapped back to full ids).

Checked against a hand-worked example and against the separately pinned
greedy rule: the identity map, and a permuted full vocabulary with its
logits permuted alike, must give greedy verification's results.
"""
import numpy as np
import pytest

import workloads as W


def test_active_worked_example(orc):
    # 4 active columns standing for full ids 17, 3, 250, 9
    ids = np.array([17, 3, 250, 9])
    z = np.array([[0, 1, 5, 2],      # column 2 -> token 250
                  [4, 4, 0, 1],      # tie of columns 0 and 1: the first, token 17
                  [0, 0, 0, 3]],     # bonus row: column 3 -> token 9
                 dtype=np.float32)
    cu = np.array([0, 3])
    r = orc.verify_greedy_active(z, "f32", 4, 1, 2, cu, np.array([250, 17, -1]), ids)
    assert r.accepted_len.tolist() == [2] and r.out_tokens.tolist() == [[250, 17, 9]]
    assert r.rows["row_argmax"].tolist() == [2, 0, 3]
    assert r.rows["row_token"].tolist() == [250, 17, 9]
    # drafts are full ids: the column index 2 is not the token 250
    r = orc.verify_greedy_active(z, "f32", 4, 1, 2, cu, np.array([2, 17, -1]), ids)
    assert r.accepted_len.tolist() == [0] and r.next_token.tolist() == [250]
    # a draft outside the active set never matches
    r = orc.verify_greedy_active(z, "f32", 4, 1, 2, cu, np.array([250, 4, -1]), ids)
    assert r.accepted_len.tolist() == [1] and r.out_tokens.tolist() == [[250, 17, -1]]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_map_is_greedy(orc, dtype):
    vb = W.ragged_batch(50, B=9, k_max=6, V=700, dtype=dtype, tie_top=True)
    args = (vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    g = orc.verify_greedy(*args)
    a = orc.verify_greedy_active(*args, np.arange(vb.V))
    np.testing.assert_array_equal(a.out_tokens, g.out_tokens)
    np.testing.assert_array_equal(a.accepted_len, g.accepted_len)
    np.testing.assert_array_equal(a.rows["row_argmax"], g.rows["row_argmax"])
    assert a.status == g.status


def test_permuted_vocabulary_is_greedy(orc):
    # every id active, in a shuffled column order, with the logits shuffled
    # alike: the full-id result is greedy's (values distinct, no ties)
    vb = W.ragged_batch(51, B=11, k_max=5, V=500, dtype="f32", p_top=0.5)
    rng = np.random.default_rng(52)
    perm = rng.permutation(vb.V).astype(np.int32)
    z = vb.logits[:, :vb.V]
    assert all(len(np.unique(row)) == vb.V for row in z)
    g = orc.verify_greedy(z, "f32", vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    a = orc.verify_greedy_active(z[:, perm], "f32", vb.V, vb.B, vb.k_max, vb.cu_rows,
                                 vb.draft_ids, perm)
    np.testing.assert_array_equal(a.out_tokens, g.out_tokens)
    np.testing.assert_array_equal(a.rows["row_token"], g.rows["row_argmax"])
    np.testing.assert_array_equal(perm[a.rows["row_argmax"]], g.rows["row_argmax"])


def test_subset_chain_invariants(orc):
    full_v, v = 5000, 700
    rng = np.random.default_rng(53)
    ids = np.sort(rng.choice(full_v, size=v, replace=False)).astype(np.int32)
    vb = W.ragged_batch(54, B=20, k_max=6, V=v, dtype="bf16", p_top=0.6)
    # drafts as full ids: the chosen column's id, or any full id
    d = np.where(vb.draft_ids >= 0, ids[np.clip(vb.draft_ids, 0, v - 1)], -1)
    d = np.where(rng.random(d.size) < 0.2, rng.integers(0, full_v, size=d.size), d).astype(np.int32)
    r = orc.verify_greedy_active(vb.logits, vb.dtype, v, vb.B, vb.k_max, vb.cu_rows, d, ids)
    tok = r.rows["row_token"]
    assert set(tok.tolist()) <= set(ids.tolist())
    for b in range(vb.B):
        r0, r1 = int(vb.cu_rows[b]), int(vb.cu_rows[b + 1])
        k, a = r1 - r0 - 1, int(r.accepted_len[b])
        assert r.out_tokens[b, :a].tolist() == d[r0:r0 + a].tolist()
        assert r.next_token[b] == tok[r0 + a]
        if a < k:
            assert d[r0 + a] != tok[r0 + a]
    assert r.accepted_len.sum() > 0
