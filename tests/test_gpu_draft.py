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


def check_alloc(got, ref, B, k):
    near = ref.margin < 1e-5      # a threshold or budget decision at a float tie
    if not near:
        np.testing.assert_array_equal(got["k_alloc"], ref.k_alloc)
        np.testing.assert_array_equal(got["cu_rows"], ref.cu_rows)
        np.testing.assert_array_equal(got["row_owner"], ref.row_owner)
        np.testing.assert_array_equal(got["row_pos"], ref.row_pos)
        np.testing.assert_array_equal(got["packed_draft"], ref.packed_draft)
        assert got["total_rows"][0] == ref.total_rows
    # structural invariants always hold
    cu = got["cu_rows"]
    assert cu[0] == 0 and (np.diff(cu) == got["k_alloc"] + 1).all()
    assert (got["row_owner"][cu[-1]:] == -1).all()


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
    check_alloc(got, ref, db.B, db.k)
    assert got["status"][0] == 0


@pytest.mark.parametrize("G", [16, 20, 40, 64, 128])
def test_budgeted_allocation(G):
    sv = need_gpu()
    db = W.mtp_adaptive(seed=44, B=16, k=7, V=5000, planted_draft=True)
    ref = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, threshold=0.05,
                                  max_rows=G)
    got = run_conf(sv, db, threshold=0.05, max_rows=G)
    np.testing.assert_allclose(got["conf"], ref.conf, rtol=CONF_RTOL, atol=0)
    check_alloc(got, ref, db.B, db.k)
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
    check_alloc(got, ref, db.B, db.k)


def test_budget_below_batch_is_reported():
    sv = need_gpu()
    db = W.mtp_adaptive(seed=46, B=8, k=3, V=800, planted_draft=True)
    ref = oracle.draft_confidence(db.draft_logits, "bf16", db.V, db.B, db.k, threshold=0.0,
                                  max_rows=5)
    got = run_conf(sv, db, threshold=0.0, max_rows=5)
    assert got["status"][0] == ref.status == 0x80
    check_alloc(got, ref, db.B, db.k)


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
    if ref_a.margin >= 1e-5:
        np.testing.assert_array_equal(got["out_tokens"], ref.out_tokens)
        np.testing.assert_array_equal(got["accepted_len"], ref.accepted_len)
    assert (got["accepted_len"] <= a["k_alloc"]).all()
