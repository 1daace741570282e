"""GPU parity (through the C ABI) of the fused row reduction, greedy,
margin-loosened greedy and relaxed top-K verification and the
prefix-acceptance counters against the CPU oracle.  Integers bit-exact; LSE within 1e-5 relative (fp32 vs fp64)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests._gpu import (assert_requests_equal, host, need_gpu, run_greedy, run_margin,
                        run_relaxed, t, torch)

pytestmark = pytest.mark.gpu

LSE_RTOL = 1e-5


def check_greedy(sv, vb, lse=True):
    ref = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    got = host(run_greedy(sv, vb, rows=True))
    assert_requests_equal(got, ref)
    R = vb.R
    np.testing.assert_array_equal(got["row_argmax"][:R], ref.rows["row_argmax"])
    np.testing.assert_array_equal(got["row_token"][:R], ref.rows["row_argmax"])
    np.testing.assert_array_equal(got["row_max"][:R], ref.rows["row_max"].astype(np.float32))
    if lse:
        np.testing.assert_allclose(got["row_lse"][:R], ref.rows["row_lse"], rtol=LSE_RTOL, atol=0)
    assert got["status"][0] == ref.status
    return got, ref


def test_tiny_greedy_workload():
    sv = need_gpu()
    check_greedy(sv, W.tiny_greedy())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V,ld", [(152064, 152064), (151552, 151557), (1000, 1003), (7, 9),
                                  (33, 33), (300_001, 300_001)])
def test_greedy_ragged_shapes(dtype, V, ld):
    """Ragged k_b (including 0), odd leading dimensions (rows not 16-byte
    aligned: head and tail elements outside the bulk copies), exact ties at
    the maximum on every row."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=V + ld, B=6, k_max=5, V=V, dtype=dtype, ld=ld, tie_top=True)
    check_greedy(sv, vb)


def test_greedy_planted_full_size_workload():
    """Qwen2.5-14B-shaped greedy verify: B=128, k=4, V=152064 bf16, the
    launch configuration the benchmark times."""
    sv = need_gpu()
    vb = W.planted_greedy()
    got, ref = check_greedy(sv, vb)
    assert (got["row_argmax"][:vb.R] == vb.extra["planted"]).all()


def test_greedy_more_rows_than_a_grid_dimension_holds():
    """More than 65535 packed rows: the row-major stream grid is then one
    dimensional (rows x chunks in x) instead of chunks x rows."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=70, B=14000, k_max=8, V=64, dtype="f32")
    assert vb.R > 65535
    check_greedy(sv, vb)


def test_greedy_neg_inf_rows_and_k_max_31():
    sv = need_gpu()
    vb = W.ragged_batch(seed=3, B=3, k_max=31, V=4099, dtype="f32", k_values=np.array([31, 0, 17]))
    vals = vb.logits
    vals[0, :] = -np.inf                        # whole row -inf: argmax 0, lse -inf
    vals[5, ::2] = -np.inf                      # partly -inf
    check_greedy(sv, vb)


def test_greedy_invalid_requests_set_status():
    sv = need_gpu()
    vb = W.ragged_batch(seed=4, B=3, k_max=2, V=64, dtype="f32", k_values=np.array([2, 2, 2]))
    vb.cu_rows[:] = [0, 1, 1, 9]                # request 1 empty, request 2 has k=7 > k_max
    ref = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    got = host(run_greedy(sv, vb))
    assert got["status"][0] & 0x10 and ref.status & 0x10
    assert_requests_equal(got, ref)


@pytest.mark.parametrize("B", [33, 40, 159, 160])
def test_owner_search_request_counts(B):
    """Row owners for request counts around the one-round search of all
    offsets (33 to 159 requests) and the round-by-round search above it,
    with ragged lengths."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=B, B=B, k_max=4, V=3000, dtype="bf16")
    check_greedy(sv, vb)


def test_owner_search_invalid_requests():
    """40 requests (one round of offset loads) with an empty request and an
    over-long one: non-decreasing offsets, invalid ranges."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=41, B=40, k_max=2, V=500, dtype="f32", k_values=np.full(40, 2))
    n = np.full(40, 3)
    n[5], n[9] = 0, 6                                       # empty; k = 5 > k_max
    vb.cu_rows[:] = np.concatenate([[0], np.cumsum(n)])
    ref = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    got = host(run_greedy(sv, vb))
    assert got["status"][0] & 0x10 and ref.status & 0x10
    assert_requests_equal(got, ref)


def test_greedy_without_row_outputs_and_repeat_calls():
    """Optional row outputs may be NULL; the workspace tickets return to zero
    so one workspace serves back-to-back calls."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=8, B=9, k_max=6, V=20000, dtype="bf16")
    ref = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    ws = sv.new_workspace(vb.logits.shape[0], vb.B, vb.V, "bf16")
    for _ in range(3):
        got = host(run_greedy(sv, vb, rows=False, workspace=ws))
        assert_requests_equal(got, ref)
    assert int(ws.sum().item()) >= 0
    R = vb.logits.shape[0]
    off = 2 * ((R * 4 + 255) // 256 * 256)                 # tok, flag
    tick = (vb.B * 4 + 255) // 256 * 256                  # request tickets
    assert ws[off:off + tick].sum().item() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_relaxed_topk_ragged(dtype):
    sv = need_gpu()
    vb = W.ragged_batch(seed=12, B=10, k_max=7, V=50_000, dtype=dtype, tie_top=True, p_top=0.4)
    K = np.array([1, 2, 3, 4, 5, 8, 50_000, 1, 4, 0], dtype=np.int32)   # last: bad K -> 1
    ref = oracle.verify_relaxed(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                vb.draft_ids, K)
    got = host(run_relaxed(sv, vb, K))
    assert_requests_equal(got, ref)
    np.testing.assert_array_equal(got["row_argmax"][:vb.R], ref.rows["row_argmax"])
    assert got["status"][0] == ref.status == 0x40


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_relaxed_more_rows_than_a_grid_dimension_holds(dtype):
    """More than 65535 packed rows of a short vocabulary: bf16 takes the row
    path (one CTA per row, a one-dimensional grid), fp32 the chunk path's
    one-dimensional row-major grid."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=73, B=14000, k_max=8, V=64, dtype=dtype, p_top=0.4)
    assert vb.R > 65535
    K = np.random.default_rng(74).integers(1, 6, size=vb.B).astype(np.int32)
    ref = oracle.verify_relaxed(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                vb.draft_ids, K)
    got = host(run_relaxed(sv, vb, K))
    assert_requests_equal(got, ref)
    np.testing.assert_array_equal(got["row_argmax"][:vb.R], ref.rows["row_argmax"])
    assert got["status"][0] == ref.status


def test_relaxed_eagle_workload_with_fused_stats():
    """EAGLE-relaxed: B=256, k=5, V=152064 bf16, planted peaks, K=4; counters
    accumulated over 20 seeded steps by the fused path and by
    spec_prefix_stats, every step's requests compared with the oracle."""
    sv = need_gpu()
    dev = "cuda"
    acc = torch.zeros(5, dtype=torch.int64, device=dev)
    ver = torch.zeros(5, dtype=torch.int64, device=dev)
    hist = torch.zeros(6, dtype=torch.int64, device=dev)
    acc2, ver2, hist2 = acc.clone(), ver.clone(), hist.clone()
    racc = rver = rhist = None
    steps = 0
    for vb in W.relaxed_steps(20):
        K = vb.extra["relaxed_k"]
        ref = oracle.verify_relaxed(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                    vb.draft_ids, K)
        res = run_relaxed(sv, vb, K, stats=(acc, ver, hist))
        sv.prefix_stats(res["accepted_len"], t(vb.cu_rows), acc2, ver2, hist2, B=vb.B,
                        k_max=vb.k_max)
        got = host(res)
        assert_requests_equal(got, ref)
        racc, rver, rhist, _ = oracle.prefix_stats(ref.accepted_len, vb.cu_rows, vb.B, vb.k_max,
                                                   racc, rver, rhist)
        steps += 1
    assert steps == 20
    torch.cuda.synchronize()
    for a, b in [(acc, racc), (ver, rver), (hist, rhist), (acc2, racc), (ver2, rver),
                 (hist2, rhist)]:
        np.testing.assert_array_equal(a.cpu().numpy(), b)
    assert rver[0] == 20 * 256 and rhist.sum() == 20 * 256


@pytest.mark.parametrize("dtype,V,ld", [("bf16", 50_000, 50_003), ("f32", 33_001, 33_001),
                                        ("bf16", 40, 40)])
def test_margin_ragged_with_positions_and_protected_ids(dtype, V, ld):
    """Per-request margins (0, small, the 5.25 preset, infinite, negative,
    NaN), a first eligible position, a count of generated tokens and a
    protected list longer than a warp, over drafts near the top values."""
    sv = need_gpu()
    base = W.ragged_batch(seed=40 + V % 7, B=12, k_max=7, V=V, dtype=dtype, ld=ld, tie_top=True)
    vb = W.near_top_drafts(base, seed=41)
    margin = np.array([0, 0.5, 1, 2, 5.25, np.inf, -1, np.nan, 3, 5.25, 1.5, 0.25], np.float32)
    gen = np.array([0, 9, 2, 0, 5, 1, 0, 3, 4, 8, 0, 6], np.int32)
    rng = np.random.default_rng(42)
    drafts = vb.draft_ids[vb.draft_ids >= 0]
    prot = np.concatenate([rng.choice(drafts, size=min(10, drafts.size), replace=False),
                           rng.integers(0, V, size=60)]).astype(np.int32)
    for kw in [dict(), dict(from_position=1, after_tokens=4), dict(from_position=3)]:
        for g, pr in [(None, None), (gen, prot)]:
            ref = oracle.verify_margin(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                       vb.draft_ids, margin, generated=g, protected_ids=pr, **kw)
            got = host(run_margin(sv, vb, margin, g, pr, **kw))
            assert_requests_equal(got, ref)
            np.testing.assert_array_equal(got["row_argmax"][:vb.R], ref.rows["row_argmax"])
            assert got["status"][0] == ref.status == 0x200


def test_margin_preset_full_size_with_fused_stats():
    """The approximate-acceptance preset: margin 5.25 for every request on
    B=128, k=4, V=152064 bf16 rows with drafts among the top 2000 values
    (gaps on both sides of the margin); the fused counters match the
    oracle's accepted lengths."""
    sv = need_gpu()
    dev = "cuda"
    vb = W.near_top_drafts(W.ragged_batch(seed=W.data_seed(2, 7), B=128, k_max=4, V=152064,
                                          k_values=np.full(128, 4)), seed=43, max_rank=2000)
    margin = np.full(vb.B, 5.25, np.float32)
    ref = oracle.verify_margin(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                               vb.draft_ids, margin)
    greedy = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                  vb.draft_ids)
    # the margin decides: more than greedy accepts, fewer than every draft
    assert greedy.accepted_len.sum() < ref.accepted_len.sum() < vb.B * vb.k_max
    acc = torch.zeros(4, dtype=torch.int64, device=dev)
    ver = torch.zeros(4, dtype=torch.int64, device=dev)
    hist = torch.zeros(5, dtype=torch.int64, device=dev)
    got = host(run_margin(sv, vb, margin, stats=(acc, ver, hist)))
    assert_requests_equal(got, ref)
    assert got["status"][0] == ref.status == 0
    racc, rver, rhist, _ = oracle.prefix_stats(ref.accepted_len, vb.cu_rows, vb.B, vb.k_max)
    for a, b in [(acc, racc), (ver, rver), (hist, rhist)]:
        np.testing.assert_array_equal(a.cpu().numpy(), b)


def test_prefix_stats_invalid_rows():
    sv = need_gpu()
    cu = np.array([0, 3, 3, 6], np.int32)           # request 1 empty
    a = np.array([1, 0, 5], np.int32)               # request 2: a = 5 > k = 2
    acc = torch.zeros(3, dtype=torch.int64, device="cuda")
    ver = torch.zeros(3, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.prefix_stats(t(a), t(cu), acc, ver, None, st, B=3, k_max=3)
    racc, rver, _, rst = oracle.prefix_stats(a, cu, 3, 3)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), racc)
    np.testing.assert_array_equal(ver.cpu().numpy(), rver)
    assert st.item() == rst == 0x10
