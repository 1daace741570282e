"""Host-side model of the compact-row restore kernel's launch: grid shape,
slot striding and per-thread addressing, checked before any GPU run for the
shapes the GPU tests and the benchmark use.

The kernel (restore_rows_kernel) runs 256 threads per CTA; blockIdx.x picks
a piece of 512 16-byte vectors of a row (each thread moves vectors tid and
tid + 256 of the piece) and blockIdx.y strides over the slots with step
gridDim.y = min(slots, 65535).  The model checks that every slot is visited
exactly once, that the pieces cover each row's vectors exactly once, and
that every read lies in the compact buffer and every write in the output
buffer, for a well-formed request; malformed ones are skipped.
"""
import numpy as np
import pytest

import oracle
import workloads as W

THREADS, PIECE = 256, 512


def _launch_model(cu, B, k_max, R_cap, row_bytes, src_ld, dst_ld, src_len, dst_len):
    vecs = row_bytes // 16
    slots = B * (k_max + 1)
    gx, gy = (vecs + PIECE - 1) // PIECE, min(slots, 65535)
    assert gx >= 1 and 1 <= gy <= 65535
    # slot striding: blockIdx.y = by visits s = by, by + gy, ...
    visits = np.zeros(slots, np.int64)
    for by in range(gy):
        visits[by::gy] += 1
    assert (visits == 1).all()
    # pieces: vectors bx*PIECE + tid and + THREADS, kept below vecs
    cover = np.zeros(vecs, np.int64)
    for bx in range(gx):
        for va in (bx * PIECE + np.arange(THREADS), bx * PIECE + THREADS + np.arange(THREADS)):
            cover[va[va < vecs]] += 1
    assert (cover == 1).all()
    # per slot: the row it reads, when its request is well formed
    s = np.arange(slots)
    b, j = s // (k_max + 1), s % (k_max + 1)
    cu = np.asarray(cu, np.int64)
    lo, hi = cu[b], cu[b + 1]
    n = hi - lo
    ok = (cu[0] == 0) & (lo >= 0) & (n >= 1) & (n - 1 <= k_max) & (hi <= R_cap)
    live = ok & (j < n)
    src_row = (lo + j)[live]
    last = (vecs - 1) * 16 + 16
    assert (src_row >= 0).all() and (src_row * src_ld + last <= src_len).all()
    assert (s[live] * dst_ld + last <= dst_len).all()
    return live, int((~ok).any())


def _check_against_oracle(cu, B, k_max, R_cap, width, src_ld, dst_ld):
    rng = np.random.default_rng(0)
    src_len = (R_cap - 1) * src_ld + width                  # tight buffer ends
    slots = B * (k_max + 1)
    dst_len = (slots - 1) * dst_ld + width
    live, bad = _launch_model(cu, B, k_max, R_cap, width, src_ld, dst_ld, src_len, dst_len)
    comp = rng.integers(0, 256, size=(R_cap, width), dtype=np.uint8)
    before = rng.integers(0, 256, size=(slots, width), dtype=np.uint8)
    ref, st = oracle.restore_rows(comp, cu, B, k_max, before)
    # the slots the model writes are exactly those the oracle changes
    changed = (ref != before).any(axis=1)
    np.testing.assert_array_equal(changed, live)
    assert bool(st & oracle.BAD_ROWS) == bool(bad)


def test_allocation_shape():
    db = W.mtp_adaptive(seed=W.data_seed(4, 5), planted_draft=True)
    al = oracle.draft_confidence(db.draft_logits, db.dtype, db.V, db.B, db.k, threshold=0.3)
    k1 = db.k + 1
    _check_against_oracle(al.cu_rows, db.B, db.k, db.B * k1, 10240, 10240, 10240)


def test_ragged_padded_rows_with_a_malformed_request():
    rng = np.random.default_rng(12)
    B, k_max = 23, 5
    kb = rng.integers(0, k_max + 1, size=B)
    kb[7] = k_max + 2
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum(kb + 1)
    _check_against_oracle(cu, B, k_max, int(cu[-1]) + 3, 8224, 8240, 8224)


@pytest.mark.parametrize("B,k_max,width", [(9000, 7, 16), (128, 4, 10240)])
def test_many_slots_and_the_benchmark_shape(B, k_max, width):
    rng = np.random.default_rng(13)
    kb = rng.integers(0, k_max + 1, size=B) if width == 16 else np.full(B, k_max)
    cu = np.zeros(B + 1, np.int64)
    cu[1:] = np.cumsum(kb + 1)
    live, bad = _launch_model(cu, B, k_max, int(cu[-1]), width, width, width,
                              (int(cu[-1]) - 1) * width + width,
                              (B * (k_max + 1) - 1) * width + width)
    assert bad == 0 and live.sum() == int(cu[-1])
