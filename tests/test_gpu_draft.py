"""GPU parity (through the C ABI) of the draft confidence and the device-side
prefix-budget allocation / packing, against the CPU oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests._gpu import host, logits_tensor, need_gpu, run_greedy, t, torch

pytestmark = pytest.mark.gpu

CONF_RTOL = 1e-5


def run_conf(sv, db, selected=None, threshold=0.3, max_rows=0, x=None):
    x = db.draft_logits if x is None else x
    return host(sv.draft_confidence(logits_tensor(x, db.dtype), V=db.V, B=db.B, k=db.k,
                                    selected=None if selected is None else t(selected),
                                    threshold=threshold, max_rows=max_rows))


U32 = 2.0 ** -24


def near_requests(ref, B, k, threshold, max_rows):
    """Requests whose allocation may legitimately differ from the oracle's.
    Every confidence is checked within CONF_RTOL, so the cumulative product
    c_bj of j + 1 of them is within (j + 1) CONF_RTOL + j U of exact (1%
    slack for the compounding).  A threshold decision can flip only where
    |c_bj - threshold| / threshold is below that; a budget cut only where
    the relative gap between the last kept and the first dropped c is below
    twice it (then both of their requests are excused)."""
    cum = np.cumprod(ref.conf.reshape(B, k).astype(np.float64), axis=1)
    band = 1.01 * (np.arange(1, k + 1) * CONF_RTOL + np.arange(k) * U32)
    near = np.zeros(B, bool)
    if threshold > 0:
        near |= (np.abs(cum - threshold) / threshold < band[None, :]).any(axis=1)
    want = (cum >= threshold).sum(axis=1)
    if max_rows > 0 and want.sum() + B > max_rows >= B:
        e = sorted(((cum[b, j], b, j) for b in range(B) for j in range(want[b])),
                   key=lambda x: (-x[0], x[1], x[2]))
        keep = max_rows - B
        if 0 < keep < len(e) and e[keep - 1][0] > 0:
            if (e[keep - 1][0] - e[keep][0]) / e[keep - 1][0] < 2 * band[-1]:
                near[e[keep - 1][1]] = near[e[keep][1]] = True
    return near


def check_alloc(got, ref, B, k, threshold, max_rows, expect_no_tie=False):
    """Allocations request by request: every request outside a float tie
    gets the oracle's k_alloc and the oracle's packed rows (drafts, owner,
    position) at its own offset; with no tie at all the whole layout agrees."""
    near = near_requests(ref, B, k, threshold, max_rows)
    print("allocation check: %d requests, %d inside a tie band" % (B, near.sum()))
    if expect_no_tie:
        assert not near.any(), "the fixed-seed workload has a decision inside a tie band"
    cu, rcu = got["cu_rows"], ref.cu_rows
    for b in np.nonzero(~near)[0]:
        assert got["k_alloc"][b] == ref.k_alloc[b], "request %d" % b
        g = slice(cu[b], cu[b + 1])
        o = slice(rcu[b], rcu[b + 1])
        np.testing.assert_array_equal(got["packed_draft"][g], ref.packed_draft[o], err_msg="request %d" % b)
        np.testing.assert_array_equal(got["row_owner"][g], ref.row_owner[o], err_msg="request %d" % b)
        np.testing.assert_array_equal(got["row_pos"][g], ref.row_pos[o], err_msg="request %d" % b)
    if not near.any():
        np.testing.assert_array_equal(got["k_alloc"], ref.k_alloc)
        np.testing.assert_array_equal(got["cu_rows"], ref.cu_rows)
        np.testing.assert_array_equal(got["row_owner"], ref.row_owner)
        np.testing.assert_array_equal(got["row_pos"], ref.row_pos)
        np.testing.assert_array_equal(got["packed_draft"], ref.packed_draft)
        assert got["total_rows"][0] == ref.total_rows
    # structural invariants always hold
    assert cu[0] == 0 and (np.diff(cu) == got["k_alloc"] + 1).all()
    assert (got["row_owner"][cu[-1]:] == -1).all()
    return near


@pytest.mark.parametrize("planted", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_mtp_confidence_workload(planted, dtype):
    """MTP/DSpark-shaped: B=16, k=7, V=151552, threshold 0.3, no budget."""
    sv = need_gpu()
    db = W.mtp_adaptive(planted_draft=planted, dtype=dtype)
    ref = oracle.draft_confidence(db.draft_logits, dtype, db.V, db.B, db.k, threshold=0.3)
    got = run_conf(sv, db)
    np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=0)
    vals = W.bf16_bits_to_f32(db.draft_logits) if dtype == "bf16" else db.draft_logits
    np.testing.assert_array_equal(got["draft_token"], np.argmax(vals[:, :db.V], axis=1))
    check_alloc(got, ref, db.B, db.k, 0.3, 0, expect_no_tie=True)
    assert got["status"][0] == 0


@pytest.mark.parametrize("G", [16, 20, 40, 64, 128])
def test_budgeted_allocation(G):
    sv = need_gpu()
    db = W.mtp_adaptive(seed=44, B=16, k=7, V=5000, planted_draft=True)
    ref = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, threshold=0.05,
                                  max_rows=G)
    got = run_conf(sv, db, threshold=0.05, max_rows=G)
    np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=0)
    check_alloc(got, ref, db.B, db.k, 0.05, G)
    assert got["total_rows"][0] <= max(G, db.B)


def test_selected_tokens_and_bad_selection():
    sv = need_gpu()
    db = W.mtp_adaptive(seed=45, B=3, k=4, V=3001, planted_draft=True)
    sel = np.random.default_rng(0).integers(0, 3001, size=12).astype(np.int32)
    sel[5] = 3001                                  # out of range: confidence 0 + status
    ref = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, selected=sel,
                                  threshold=0.0)
    got = run_conf(sv, db, selected=sel, threshold=0.0)
    np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=1e-30)
    assert got["status"][0] == ref.status == 0x20
    check_alloc(got, ref, db.B, db.k, 0.0, 0)


def test_budget_below_batch_is_reported():
    sv = need_gpu()
    db = W.mtp_adaptive(seed=46, B=8, k=3, V=800, planted_draft=True)
    ref = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, threshold=0.0,
                                  max_rows=5)
    got = run_conf(sv, db, threshold=0.0, max_rows=5)
    assert got["status"][0] == ref.status == 0x80
    check_alloc(got, ref, db.B, db.k, 0.0, 5)


def test_adaptive_verify_pipeline_on_device():
    """Confidence -> allocation -> packed greedy verification, all device
    side: the packed layout from the allocation drives the verifier."""
    sv = need_gpu()
    db = W.mtp_adaptive(seed=47, planted_draft=True)
    alloc = sv.draft_confidence(logits_tensor(db.draft_logits, "bf16"), V=db.V, B=db.B, k=db.k,
                                threshold=0.3)
    tgt = logits_tensor(db.target_logits, "bf16")
    res = sv.verify_greedy(tgt, alloc["cu_rows"], alloc["packed_draft"], V=db.V, B=db.B,
                           k_max=db.k, R_cap=db.B * (db.k + 1))
    a = host(alloc)
    got = host(res)
    ref_a = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, threshold=0.3)
    ref = oracle.verify_greedy(db.target_logits, "bf16", db.V, db.B, db.k, ref_a.cu_rows,
                               ref_a.packed_draft)
    # the target rows are indexed by packed row, so the two sides see the
    # same rows only with the same layout: the fixed seed has no tie
    check_alloc(a, ref_a, db.B, db.k, 0.3, 0, expect_no_tie=True)
    np.testing.assert_array_equal(got["out_tokens"], ref.out_tokens)
    np.testing.assert_array_equal(got["accepted_len"], ref.accepted_len)
    np.testing.assert_array_equal(got["next_token"], ref.next_token)
    assert (got["accepted_len"] <= a["k_alloc"]).all()


@pytest.mark.parametrize("dtype,V", [("bf16", 1_048_000), ("f32", 524_000), ("bf16", 1000),
                                     ("bf16", 16_385), ("bf16", 262_144), ("bf16", 262_145),
                                     ("f32", 131_072), ("f32", 131_073)])
def test_confidence_row_lengths(dtype, V):
    """Draft rows near the 2 MiB limit (64 chunks), far below one chunk, of
    exactly 16 chunks and one element more (a last chunk of one element, as
    in the 16 385-element bf16 row); the chunk-major grid and the combine
    over every chunk."""
    sv = need_gpu()
    db = W.mtp_adaptive(seed=V % 997, B=3, k=4, V=V, planted_draft=True, dtype=dtype)
    ref = oracle.draft_confidence(db.draft_logits, dtype, db.V, db.B, db.k, threshold=0.3)
    got = run_conf(sv, db)
    np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=0)
    vals = W.bf16_bits_to_f32(db.draft_logits) if dtype == "bf16" else db.draft_logits
    np.testing.assert_array_equal(got["draft_token"], np.argmax(vals[:, :db.V], axis=1))
    check_alloc(got, ref, db.B, db.k, 0.3, 0)
    assert got["status"][0] == 0


@pytest.mark.parametrize("dtype,V,off", [("bf16", 151_552, 3), ("bf16", 20_000, 1), ("f32", 70_001, 2)])
def test_confidence_unaligned_rows(dtype, V, off):
    """Rows that start off a 16-byte boundary (a view into wider rows): every
    chunk's head and tail elements come from plain loads, and the selected
    tokens' logits from the unaligned rows."""
    sv = need_gpu()
    db = W.mtp_adaptive(seed=V % 991, B=4, k=3, V=V, planted_draft=True, dtype=dtype)
    x = logits_tensor(db.draft_logits, dtype)
    # rows of V + 8 elements whose first starts `off` elements into the
    # allocation (one spare row keeps the last one inside it)
    Q, ld = x.shape[0], V + 8
    wide = torch.zeros(((Q + 1) * ld,), dtype=x.dtype, device=x.device)
    view = torch.as_strided(wide, (Q, ld), (ld, 1), off)
    view[:, :V] = x[:, :V]
    sel = np.random.default_rng(V).integers(0, V, size=db.B * db.k).astype(np.int32)
    for selected in (None, sel):
        ref = oracle.draft_confidence(db.draft_logits, dtype, db.V, db.B, db.k, selected=selected,
                                      threshold=0.3)
        got = host(sv.draft_confidence(view, V=V, B=db.B, k=db.k,
                                       selected=None if selected is None else t(selected),
                                       threshold=0.3))
        np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=1e-30)
        check_alloc(got, ref, db.B, db.k, 0.3, 0)
        assert got["status"][0] == 0
