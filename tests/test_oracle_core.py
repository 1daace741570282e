"""Pins for the oracle's Philox generator and its fused row reduction (A1),
greedy chain (A2) and relaxed top-K acceptance (A5).

Each pin checks the oracle against something other than itself: published
known answers, closed forms, library routines, hand-worked special cases and
invariants.
"""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import workloads as W
from tests import _brute


# ---------------------------------------------------------------- Philox -----

# Known-answer vectors distributed with the Random123 library by the authors of
# "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11) for Philox4x32-10:
# (counter, key) -> output.
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", PHILOX_KAT)
def test_philox_known_answers(orc, ctr, key, out):
    assert tuple(int(x) for x in orc.philox4x32_10(ctr, key)) == out


def test_uniform_mapping(orc):
    # u = (2*(x>>9)+1) * 2^-24: endpoints and an interior point
    assert orc.uniform(0) == 2.0 ** -24
    assert orc.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert orc.uniform(0x80000000) == 0.5 + 2.0 ** -24
    assert orc.uniform(0x1FF) == 2.0 ** -24          # low 9 bits are dropped


def test_token_uniform_counter_layout(orc):
    seed = 0x0123456789ABCDEF
    for i in [0, 1, 2, 3, 4, 7, 151_999, 152_063]:
        words = orc.philox4x32_10([i >> 2, 5, 77, 9], [seed & 0xFFFFFFFF, seed >> 32])
        assert orc.token_uniform(seed, 77, 5, 9, i) == orc.uniform(int(words[i & 3]))


def test_uniforms_are_uniform(orc):
    u = np.array([orc.token_uniform(42, 3, 1, 0, i) for i in range(40_000)])
    assert 0.0 < u.min() and u.max() < 1.0
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
    # different positions / requests / steps give unrelated streams
    v = np.array([orc.token_uniform(42, 3, 2, 0, i) for i in range(4_000)])
    assert abs(np.corrcoef(u[:4000], v)[0, 1]) < 0.06


# ------------------------------------------------------------- A1 reduce -----

def _row(vals, dtype="f32", ld=None):
    vals = np.asarray(vals, dtype=np.float32)[None, :]
    if ld is not None:
        pad = np.full((1, ld), 1e30, dtype=np.float32)   # poison beyond V
        pad[:, :vals.shape[1]] = vals
        vals = pad
    return W.bf16_bits(vals) if dtype == "bf16" else vals


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_constant_row(orc, dtype):
    V = 1000
    mx, lse, am = orc.row_reduce(_row([2.5] * V, dtype, ld=1024), dtype, V=V)
    assert am[0] == 0 and mx[0] == 2.5
    assert lse[0] == pytest.approx(2.5 + math.log(V), rel=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_one_hot(orc, dtype):
    V, L, p = 777, 6.0, 500
    z = [0.0] * V
    z[p] = L
    mx, lse, am = orc.row_reduce(_row(z, dtype), dtype)
    assert am[0] == p and mx[0] == L
    assert lse[0] == pytest.approx(math.log(math.exp(L) + V - 1), rel=1e-13)


def test_reduce_ties_and_signed_zero(orc):
    _, _, am = orc.row_reduce(_row([0, 3, 1, 3, -1]), "f32")
    assert am[0] == 1                                    # first of the tied maxima
    _, _, am = orc.row_reduce(_row([-0.0, 0.0, -1.0]), "f32")
    assert am[0] == 0                                    # -0.0 == +0.0
    _, _, am = orc.row_reduce(_row([-5.0, 0.0, -0.0]), "f32")
    assert am[0] == 1


def test_reduce_neg_inf(orc):
    mx, lse, am = orc.row_reduce(_row([-np.inf] * 5), "f32")
    assert mx[0] == -np.inf and lse[0] == -np.inf and am[0] == 0
    mx, lse, am = orc.row_reduce(_row([-np.inf, 1.0, -np.inf, 1.0]), "f32")
    assert am[0] == 1 and lse[0] == pytest.approx(1.0 + math.log(2.0), rel=1e-14)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_matches_library(orc, dtype):
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((6, 3001)) * 3).astype(np.float32)
    x = W.bf16_bits(z) if dtype == "bf16" else z
    vals = W.bf16_bits_to_f32(x).astype(np.float64) if dtype == "bf16" else z.astype(np.float64)
    mx, lse, am = orc.row_reduce(x, dtype)
    np.testing.assert_array_equal(am, np.argmax(vals, axis=1))
    np.testing.assert_array_equal(mx, vals.max(axis=1))
    np.testing.assert_allclose(lse, scipy.special.logsumexp(vals, axis=1), rtol=1e-13)
    for r in range(2):
        assert lse[r] == pytest.approx(_brute.lse_direct(list(vals[r])), rel=1e-14)


def test_reduce_shift_invariance(orc):
    rng = np.random.default_rng(1)
    z = rng.integers(-40, 40, size=(3, 500)).astype(np.float32) / 4
    _, l0, a0 = orc.row_reduce(z, "f32")
    _, l1, a1 = orc.row_reduce(z + np.float32(16.0), "f32")
    np.testing.assert_array_equal(a0, a1)
    np.testing.assert_allclose(l1 - l0, 16.0, rtol=1e-12)


def test_bf16_decode_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    z = (rng.standard_normal(4096) * 5).astype(np.float32)
    bits = W.bf16_bits(z)
    ref = torch.from_numpy(z).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(W.bf16_bits_to_f32(bits), ref)
    mx, _, _ = orc.row_reduce(bits[None, :], "bf16")
    assert mx[0] == ref.max()


# ------------------------------------------------------------- A2 greedy -----

def test_greedy_worked_example(orc):
    # request with k = 2: row0 = [0,3,1,3,-1] -> first argmax 1 = d0 (accept);
    # row1 = [2,0,0,0,0] -> argmax 0 != d1 = 3 (reject): a = 1, emits [1, 0]
    z = np.array([[0, 3, 1, 3, -1], [2, 0, 0, 0, 0], [0, 0, 0, 0, 9]], dtype=np.float32)
    res = orc.verify_greedy(z, "f32", 5, 1, 2, np.array([0, 3]), np.array([1, 3, -1]))
    assert res.accepted_len.tolist() == [1]
    assert res.out_tokens.tolist() == [[1, 0, -1]]
    assert res.next_token.tolist() == [0]
    # same rows, all drafts match: a = k and the bonus is the last row's argmax
    res = orc.verify_greedy(z, "f32", 5, 1, 2, np.array([0, 3]), np.array([1, 0, -1]))
    assert res.accepted_len.tolist() == [2]
    assert res.out_tokens.tolist() == [[1, 0, 4]]
    assert res.next_token.tolist() == [4]


def _check_chain_invariants(vb, res, row_tok):
    for b in range(vb.B):
        r0, r1 = int(vb.cu_rows[b]), int(vb.cu_rows[b + 1])
        k, a = r1 - r0 - 1, int(res.accepted_len[b])
        assert 0 <= a <= k
        out = res.out_tokens[b]
        assert out[:a].tolist() == vb.draft_ids[r0:r0 + a].tolist()
        assert out[a] == res.next_token[b] == row_tok[r0 + a]   # one non-draft token
        assert (out[a + 1:] == -1).all()
        if a < k:
            assert row_tok[r0 + a] != vb.draft_ids[r0 + a]


@pytest.mark.parametrize("seed", range(4))
def test_greedy_invariants_ragged(orc, seed):
    vb = W.ragged_batch(seed, B=9, k_max=6, V=700, dtype="bf16", tie_top=(seed % 2 == 0))
    res = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    assert res.status == 0
    _check_chain_invariants(vb, res, res.rows["row_argmax"])


def test_greedy_all_match_and_k0(orc):
    vb = W.ragged_batch(11, B=5, k_max=4, V=300, dtype="f32", p_top=1.0,
                        k_values=np.array([4, 0, 2, 4, 1]))
    res = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    assert res.accepted_len.tolist() == [4, 0, 2, 4, 1]
    am = res.rows["row_argmax"]
    assert res.next_token.tolist() == [int(am[vb.cu_rows[b + 1] - 1]) for b in range(5)]


def test_greedy_invalid_request(orc):
    z = np.zeros((6, 8), dtype=np.float32)
    cu = np.array([0, 1, 6])          # request 1 has k = 4 > k_max = 2
    res = orc.verify_greedy(z, "f32", 8, 2, 2, cu, np.array([-1, 0, 0, 0, 0, -1]))
    assert res.status & orc.BAD_ROWS
    assert res.accepted_len.tolist() == [0, 0]
    assert res.next_token.tolist() == [0, -1]
    assert res.out_tokens[1].tolist() == [-1, -1, -1]


def test_greedy_expected_acceptance_closed_form(orc):
    # planted workload: the planted token is the unique argmax, the draft
    # copies it with prob p_j, so E[a] = sum_m prod_{j<m} p_j
    p = (0.8, 0.65, 0.5, 0.4)
    vb = W.planted_greedy(seed=99, B=3000, k=4, V=64, p_pos=p, dtype="f32")
    res = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    expect = sum(np.prod(p[:m]) for m in range(1, 5))
    assert abs(res.accepted_len.mean() - expect) < 4 * 1.2 / math.sqrt(vb.B)


# ------------------------------------------------------------ A5 relaxed -----

def test_relaxed_worked_example(orc):
    # row1 = [2,0,0,0,0], draft 3: only z[0] > z[3], so rank 1 -> accepted iff K >= 2
    z = np.array([[0, 3, 1, 3, -1], [2, 0, 0, 0, 0], [0, 0, 0, 0, 9]], dtype=np.float32)
    cu, d = np.array([0, 3]), np.array([1, 3, -1])
    r2 = orc.verify_relaxed(z, "f32", 5, 1, 2, cu, d, np.array([2]))
    assert r2.accepted_len.tolist() == [2] and r2.next_token.tolist() == [4]
    r1 = orc.verify_relaxed(z, "f32", 5, 1, 2, cu, d, np.array([1]))
    assert r1.accepted_len.tolist() == [1] and r1.next_token.tolist() == [0]
    # draft 3 in row0 (tied maximum 3 at index 3) is accepted at K = 1
    r = orc.verify_relaxed(z, "f32", 5, 1, 2, cu, np.array([3, 0, -1]), np.array([1]))
    assert r.accepted_len.tolist() == [2]


def test_relaxed_rank_matches_sort(orc):
    vb = W.ragged_batch(5, B=7, k_max=5, V=257, dtype="bf16", tie_top=True, p_top=0.3)
    K = np.array([1, 2, 3, 4, 10, 257, 1], dtype=np.int32)
    res = orc.verify_relaxed(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                             vb.draft_ids, K)
    vals = vb.values_f32().astype(np.float64)
    for r in range(vb.R):
        d = int(vb.draft_ids[r])
        if 0 <= d < vb.V:
            assert res.rows["row_rank"][r] == _brute.draft_rank(list(vals[r, :vb.V]), d)
    _check_chain_invariants(vb, res, res.rows["row_argmax"])
    # K = V accepts every in-vocabulary draft
    for b in [5]:
        r0, r1 = vb.cu_rows[b], vb.cu_rows[b + 1]
        assert res.accepted_len[b] == r1 - r0 - 1


def test_relaxed_k1_equals_greedy_without_ties(orc):
    vb = W.ragged_batch(8, B=12, k_max=5, V=999, dtype="f32")
    g = orc.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    r = orc.verify_relaxed(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids,
                           np.ones(vb.B, np.int32))
    np.testing.assert_array_equal(g.out_tokens, r.out_tokens)


def test_relaxed_bad_k_and_out_of_vocab(orc):
    z = np.array([[1, 2, 3], [3, 2, 1]], dtype=np.float32)
    r = orc.verify_relaxed(z, "f32", 3, 1, 1, np.array([0, 2]), np.array([7, -1]), np.array([0]))
    assert r.status & orc.BAD_RELAXED_K
    assert r.accepted_len.tolist() == [0] and r.next_token.tolist() == [2]
