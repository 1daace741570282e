"""GPU parity (through the C ABI) of greedy verification over an active
vocabulary and of the restore of compact rows to request slots, against the
CPU oracle.  Bit-exact.  This file is collected last: its paths are the
newest, so a run stopping at the first failure has run every other test
before it."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests._gpu import (assert_requests_equal, host, logits_tensor, need_gpu, run_active, t,
                        torch)

pytestmark = pytest.mark.gpu


def _active_case(seed, B, k_max, V, full_v, dtype, ld=None, sort_ids=True, tie_top=False):
    """Logits over V active columns standing for V distinct ids of a full
    vocabulary; drafts are full ids: the top column's id, another active
    column's id, or an id outside the active set."""
    vb = W.ragged_batch(seed=seed, B=B, k_max=k_max, V=V, dtype=dtype, ld=ld, tie_top=tie_top)
    rng = np.random.default_rng(seed + 1)
    ids = rng.choice(full_v, size=V, replace=False).astype(np.int32)
    if sort_ids:
        ids.sort()
    d = np.where(vb.draft_ids >= 0, ids[np.clip(vb.draft_ids, 0, V - 1)], -1).astype(np.int32)
    off = rng.random(d.size) < 0.15
    d[off] = rng.integers(0, full_v, size=int(off.sum()))
    d[vb.cu_rows[1:] - 1] = -1
    return vb, d, ids


@pytest.mark.parametrize("dtype,V,ld,full_v,sort_ids", [
    ("bf16", 50_000, 50_003, 152_064, True), ("f32", 33, 33, 1_000, False),
    ("bf16", 4_099, 4_099, 151_552, False)])
def test_active_vocabulary_ragged(dtype, V, ld, full_v, sort_ids):
    """Active columns as sorted or shuffled subsets of the full vocabulary,
    odd leading dimensions, exact ties at the top; row outputs give the
    argmax column and its full id."""
    sv = need_gpu()
    vb, d, ids = _active_case(60 + V % 11, 12, 7, V, full_v, dtype, ld, sort_ids, tie_top=True)
    ref = oracle.verify_greedy_active(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                      d, ids)
    got = host(run_active(sv, vb, d, ids))
    assert_requests_equal(got, ref)
    np.testing.assert_array_equal(got["row_argmax"][:vb.R], ref.rows["row_argmax"])
    np.testing.assert_array_equal(got["row_token"][:vb.R], ref.rows["row_token"])
    assert got["status"][0] == ref.status == 0


def test_active_vocabulary_32k_columns_with_fused_stats():
    """B=128, ragged k <= 4, over 32000 active columns of a 152064-token vocabulary
    (bf16), counters fused."""
    sv = need_gpu()
    dev = "cuda"
    vb, d, ids = _active_case(W.data_seed(2, 8), 128, 4, 32_000, 152_064, "bf16")
    ref = oracle.verify_greedy_active(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                      d, ids)
    acc = torch.zeros(4, dtype=torch.int64, device=dev)
    ver = torch.zeros(4, dtype=torch.int64, device=dev)
    hist = torch.zeros(5, dtype=torch.int64, device=dev)
    got = host(run_active(sv, vb, d, ids, stats=(acc, ver, hist)))
    assert_requests_equal(got, ref)
    racc, rver, rhist, _ = oracle.prefix_stats(ref.accepted_len, vb.cu_rows, vb.B, vb.k_max)
    for a, b in [(acc, racc), (ver, rver), (hist, rhist)]:
        np.testing.assert_array_equal(a.cpu().numpy(), b)


def _bytes(x: torch.Tensor) -> np.ndarray:
    """Host copy of a 2-D tensor's rows as bytes."""
    torch.cuda.synchronize()
    return x.contiguous().cpu().view(torch.uint8).numpy()


def test_restore_hidden_rows_after_the_allocation():
    """Target hidden states (bf16, H=5120) packed by the device allocation of
    the MTP-shaped workload come back to their request slots."""
    sv = need_gpu()
    db = W.mtp_adaptive(seed=W.data_seed(4, 5), planted_draft=True)
    al = sv.draft_confidence(logits_tensor(db.draft_logits, "bf16"), V=db.V, B=db.B, k=db.k)
    k1 = db.k + 1
    g = torch.Generator(device="cuda").manual_seed(11)
    compact = torch.randn(db.B * k1, 5120, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.full((db.B * k1, 5120), -7.0, device="cuda", dtype=torch.bfloat16)
    before = _bytes(out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.restore_rows(compact, al["cu_rows"], out, B=db.B, k_max=db.k, status=status)
    cu = al["cu_rows"].cpu().numpy()
    ref, st = oracle.restore_rows(_bytes(compact), cu, db.B, db.k, before)
    np.testing.assert_array_equal(_bytes(out), ref)
    assert int(status.item()) == st == 0
    assert 0 < int(cu[-1]) < db.B * k1                       # some slots stay untouched


def test_restore_ragged_padded_rows_and_a_malformed_request():
    """Rows of 8224 bytes (two 8 KiB pieces, the second short) read from a
    padded source stride; one request claims k > k_max and is skipped."""
    sv = need_gpu()
    rng = np.random.default_rng(12)
    B, k_max, width, ld = 23, 5, 8224, 8240
    kb = rng.integers(0, k_max + 1, size=B)
    kb[7] = k_max + 2                                        # malformed
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(kb + 1)
    R_cap = int(cu[-1]) + 3
    src = torch.from_numpy(rng.integers(0, 256, size=(R_cap, ld), dtype=np.uint8)).cuda()
    compact = src[:, :width]
    out = torch.from_numpy(rng.integers(0, 256, size=(B * (k_max + 1), width),
                                        dtype=np.uint8)).cuda()
    before = _bytes(out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.restore_rows(compact, t(cu), out, B=B, k_max=k_max, status=status)
    ref, st = oracle.restore_rows(_bytes(compact), cu, B, k_max, before)
    np.testing.assert_array_equal(_bytes(out), ref)
    assert int(status.item()) == st == oracle.BAD_ROWS


def test_restore_more_slots_than_a_grid_dimension_holds():
    """72000 slots of 16-byte rows (fp32 x 4): the slot loop strides."""
    sv = need_gpu()
    rng = np.random.default_rng(13)
    B, k_max = 9000, 7
    kb = rng.integers(0, k_max + 1, size=B)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(kb + 1)
    compact = torch.from_numpy(rng.standard_normal((int(cu[-1]), 4)).astype(np.float32)).cuda()
    out = torch.zeros(B * (k_max + 1), 4, device="cuda")
    sv.restore_rows(compact, t(cu), out, B=B, k_max=k_max)
    ref, st = oracle.restore_rows(_bytes(compact), cu, B, k_max, _bytes(torch.zeros_like(out)))
    np.testing.assert_array_equal(_bytes(out), ref)
    assert st == 0
