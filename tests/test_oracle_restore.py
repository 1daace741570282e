"""Pins for the oracle's restore of compact rows to request slots (xLLM
"自适应投机推理" §"基于 MTP logits 的自适应 target 验证": compact target
outputs restored by device offsets).

The restore is checked on a hand-worked layout and as the inverse of the
packing that the separately pinned prefix allocation produces: rows packed
by (row owner, row position) and restored by the allocation's offsets come
back to their slots.
"""
import numpy as np

import workloads as W


def test_restore_worked_example(orc):
    # k_0 = 1 (rows 0-1), k_1 = 2 (rows 2-4); k_max = 2: three slots each
    compact = np.arange(5 * 4, dtype=np.uint8).reshape(5, 4)
    out = np.full((6, 4), 255, np.uint8)
    res, st = orc.restore_rows(compact, [0, 2, 5], 2, 2, out)
    assert st == 0
    assert res[:, 0].tolist() == [0, 4, 255, 8, 12, 16]
    np.testing.assert_array_equal(res[4], compact[3])
    np.testing.assert_array_equal(out, np.full((6, 4), 255, np.uint8))   # input untouched


def test_restore_skips_malformed_requests(orc):
    compact = np.arange(6 * 2, dtype=np.uint8).reshape(6, 2)
    out = np.zeros((9, 2), np.uint8)
    # request 1 has k = 3 > k_max = 2; request 2 reads beyond the buffer
    res, st = orc.restore_rows(compact, [0, 1, 5, 7], 3, 2, out)
    assert st & orc.BAD_ROWS
    np.testing.assert_array_equal(res[0], compact[0])
    assert (res[1:].sum() == 0)
    res, st = orc.restore_rows(compact, [1, 2], 1, 2, out)          # cu_rows[0] != 0
    assert st & orc.BAD_ROWS and res.sum() == 0


def test_restore_inverts_the_allocation_packing(orc):
    db = W.mtp_adaptive(seed=W.data_seed(4, 3), planted_draft=True)
    al = orc.draft_confidence(db.draft_logits, db.dtype, db.V, db.B, db.k, threshold=0.3)
    k1 = db.k + 1
    assert 0 < al.total_rows < db.B * k1
    rng = np.random.default_rng(5)
    dense = rng.integers(0, 256, size=(db.B * k1, 48), dtype=np.uint8)
    # pack: compact row r holds the slot of (row_owner[r], row_pos[r])
    owner, pos = al.row_owner[:al.total_rows], al.row_pos[:al.total_rows]
    compact = dense[owner * k1 + pos]
    sentinel = np.full_like(dense, 7)
    res, st = orc.restore_rows(compact, al.cu_rows, db.B, db.k, sentinel)
    assert st == 0
    kept = np.zeros(db.B * k1, bool)
    kept[owner * k1 + pos] = True
    np.testing.assert_array_equal(res[kept], dense[kept])
    assert (res[~kept] == 7).all()
    # every request keeps its first k_alloc + 1 slots
    for b in range(db.B):
        assert kept[b * k1: b * k1 + al.k_alloc[b] + 1].all()
        assert not kept[b * k1 + al.k_alloc[b] + 1: (b + 1) * k1].any()
