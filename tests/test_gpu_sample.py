"""GPU parity (through the C ABI) of the stochastic verifier: filtered
Gumbel-max sampling with Philox4x32-10 uniforms per row and the point-mass
rejection chain per request, against the CPU oracle.

Sampled tokens must match the fp64 definition on every row except where the
oracle reports a decision (a min-p / top-p threshold or the Gumbel winner)
within the fp32 error band of its boundary (tests/_gpu.py derives the bands
per row); at most floor(10^-4 R) rows of a batch may take that allowance,
which is none below 10^4 rows.  The full-size workload must agree on every
row.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests._gpu import compare_sampled, host, need_gpu, run_sample, t, torch

pytestmark = pytest.mark.gpu


def check(sv, vb, p, label="", **kw):
    ref = oracle.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                               vb.draft_ids, p)
    got = host(run_sample(sv, vb, p, rows=True, **kw))
    n_bad = compare_sampled(vb, p, got, ref, label=label)
    assert got["status"][0] == ref.status
    got["n_differ"] = n_bad
    return got, ref


def params(B, T, k, p, m, seed=0, step=0):
    rng = np.random.default_rng(seed)
    f = lambda v, dt: np.full(B, v, dtype=dt)
    return W.SampleParams(f(T, np.float32), f(k, np.int32), f(p, np.float32), f(m, np.float32),
                          rng.integers(0, 2**63, size=B, dtype=np.int64).astype(np.uint64),
                          np.arange(B, dtype=np.uint32) * 7 + 3, step)


def test_stochastic_full_size_workload():
    """Mixed-temperature batch at B=128, k=4, V=152064 bf16 -- the benchmark's
    launch configuration -- every row compared."""
    sv = need_gpu()
    vb, p = W.stochastic()
    got, _ = check(sv, vb, p, label="full-size workload")
    assert got["n_differ"] == 0


@pytest.mark.parametrize("T,k,tp,mp", [
    (1.0, 0, 1.0, 0.0),      # no filter: Gumbel over the whole vocabulary
    (0.5, 0, 1.0, 0.0),
    (1.0, 0, 0.9, 0.0),      # pure top-p (merged per-value counts, listed elements)
    (0.5, 0, 0.9, 0.0),
    (0.7, 0, 0.5, 0.0),
    (1.0, 20, 1.0, 0.0),     # top-k: chunk lists above the k-th thread maximum
    (1.0, 50, 0.9, 0.05),
    (0.5, 0, 1.0, 0.05),     # min-p only
    (1.0, 0, 0.95, 0.05),
    (1.0, 200, 1.0, 0.0),
    (1.0, 256, 1.0, 0.0),    # the largest k bounded by the thread maxima
    (1.0, 257, 1.0, 0.0),    # beyond it: ladder bound, else the whole row
    (1.0, 1000, 0.8, 0.0),
    (2.0, 5, 1.0, 1e-6),
    (1.0, 1, 1.0, 0.0),      # top-k = 1: the maximum tie group
    (0.8, 0, 1.0, 1.0),      # min-p = 1: the maximum tie group
    (1e-3, 0, 1.0, 0.0),     # tiny temperature
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_filter_combinations(T, k, tp, mp, dtype):
    sv = need_gpu()
    vb = W.ragged_batch(seed=int(T * 1000) + k, B=5, k_max=4, V=152064 if dtype == "bf16" else 40000,
                        dtype=dtype, tie_top=True, p_top=0.7)
    check(sv, vb, params(vb.B, T, k, tp, mp, seed=k))


@pytest.mark.parametrize("V,ld", [(1000, 1003), (7, 9), (33, 40), (4097, 4097)])
def test_small_and_unaligned_rows(V, ld):
    sv = need_gpu()
    for dtype in ["bf16", "f32"]:
        vb = W.ragged_batch(seed=V, B=7, k_max=6, V=V, dtype=dtype, ld=ld)
        rng = np.random.default_rng(V)
        p = W.random_sample_params(rng, vb.B, top_ks=(0, 2, 5, 20), top_ps=(1.0, 0.9, 0.5))
        check(sv, vb, p)


def test_flat_rows_overflow_candidates():
    """Many exact ties at the top (integer logits): candidate lists overflow
    and the exact selects over the whole row take over."""
    sv = need_gpu()
    rng = np.random.default_rng(1)
    vb = W.ragged_batch(seed=2, B=4, k_max=3, V=152064, dtype="bf16")
    z = rng.integers(-3, 3, size=vb.logits.shape).astype(np.float32)
    vb.logits = W.bf16_bits(z)
    vb.draft_ids[:] = np.argmax(z, axis=1)
    for (T, k, tp, mp) in [(1.0, 20, 1.0, 0.0), (1.0, 0, 1.0, 0.5), (1.0, 50, 0.9, 0.0)]:
        check(sv, vb, params(vb.B, T, k, tp, mp, seed=k))


def test_bad_parameters_fall_back():
    sv = need_gpu()
    vb = W.ragged_batch(seed=3, B=4, k_max=2, V=5000, dtype="f32", k_values=np.array([2, 2, 2, 2]))
    p = W.SampleParams(np.array([-1.0, 1.0, 1.0, 1.0], np.float32), np.array([0, -3, 0, 0], np.int32),
                       np.array([1.0, 1.0, 1.5, 1.0], np.float32),
                       np.array([0.0, 0.0, 0.0, -0.1], np.float32),
                       np.arange(4, dtype=np.uint64), np.arange(4, dtype=np.uint32))
    got, ref = check(sv, vb, p)
    assert got["status"][0] == 0xF


def test_request_id_default_and_steps():
    """request_id NULL means the request index; different steps give
    different draws; the same call is deterministic."""
    sv = need_gpu()
    vb, p = W.stochastic(seed=31, B=16, k=4, V=30000, temperatures=(1.0,), top_ks=(0,),
                         top_ps=(1.0,), min_ps=(0.0,))
    p.request_id = None
    a, _ = check(sv, vb, p)
    b, _ = check(sv, vb, p)
    np.testing.assert_array_equal(a["row_token"], b["row_token"])
    p.step = 9
    c, _ = check(sv, vb, p)
    assert (c["row_token"][:vb.R] != a["row_token"][:vb.R]).mean() > 0.5


def test_sampler_frequencies_match_filtered_distribution():
    """Chi-square of GPU-sampled tokens over many steps against the filtered
    softmax computed independently of both implementations."""
    import scipy.special
    import scipy.stats
    sv = need_gpu()
    V = 64
    rng = np.random.default_rng(5)
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    B, steps = 256, 40
    logits = np.tile(z, (B, 1))
    cu = np.arange(B + 1, dtype=np.int32)
    vb = W.VerifyBatch(logits, "f32", V, B, 0, cu, np.full(B, -1, np.int32))
    T, k, tp = 0.8, 10, 0.9
    # reference distribution: top-10 then nucleus 0.9 over softmax(z/T)
    order = np.argsort(-z.astype(np.float64), kind="stable")
    keep = np.zeros(V, bool)
    keep[order[:k]] = True
    w = np.where(keep, scipy.special.softmax(z.astype(np.float64) / T), 0)
    w /= w.sum()
    cum = 0.0
    F = np.zeros(V, bool)
    for i in order[:k]:
        if cum < tp:
            F[i] = True
        cum += w[i]
    pF = np.where(F, w, 0)
    pF /= pF.sum()
    counts = np.zeros(V)
    for s in range(steps):
        p = params(B, T, k, tp, 0.0, seed=s, step=s)
        got = host(run_sample(sv, vb, p, rows=False))
        counts += np.bincount(got["next_token"], minlength=V)
    n = B * steps
    assert counts[~F].sum() == 0
    assert scipy.stats.chisquare(counts[F], n * pF[F]).pvalue > 1e-4


def shifted(vb, shift):
    """Add a constant to every logit (re-rounded to the batch's dtype)."""
    if shift == 0.0:
        return vb
    if vb.dtype == "bf16":
        vb.logits = W.bf16_bits(W.bf16_bits_to_f32(vb.logits) + np.float32(shift))
    else:
        vb.logits = (vb.logits + np.float32(shift)).astype(np.float32)
    return vb


@pytest.mark.parametrize("T,tp,sigma,shift", [
    (0.5, 0.9, 3.0, 0.0),     # small nucleus: settled from the candidate lists
    (1.0, 0.9, 3.0, 0.0),     # diffuse nucleus: settled from the counted values
    (2.0, 0.7, 3.0, 0.0),
    (1.0, 0.9, 0.3, 0.0),     # nearly flat rows: the lists overflow, exact row selects
    (1e-6, 0.9, 3.0, 20.0),   # grid origin beyond 2^21: exact row selects
    (1.0, 0.99, 3.0, -40.0),  # all logits negative
    (0.25, 0.5, 8.0, 0.0),    # nucleus of one or two values
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pure_top_p_paths(T, tp, sigma, shift, dtype):
    sv = need_gpu()
    V = 152064 if dtype == "bf16" else 60000
    vb = W.ragged_batch(seed=int(T * 100) + int(sigma * 10), B=6, k_max=3, V=V, dtype=dtype,
                        sigma=sigma)
    check(sv, shifted(vb, shift), params(vb.B, T, 0, tp, 0.0, seed=7))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pure_top_p_rows_not_vector_aligned(dtype):
    """Diffuse nuclei in rows whose start is not 16-byte aligned: the second
    pass over the row covers the unaligned head and tail by plain loads."""
    sv = need_gpu()
    V = 152064 if dtype == "bf16" else 60000
    vb = W.ragged_batch(seed=43, B=5, k_max=3, V=V, dtype=dtype, ld=V + 3)
    check(sv, vb, params(vb.B, 1.0, 0, 0.9, 0.0, seed=5))


def test_many_diffuse_rows():
    """Every row's nucleus is diffuse (80 requests): most rows are settled
    from the counted values, and any they cannot settle take exact selects
    over the whole row in the same finish CTA."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=47, B=80, k_max=4, V=152064, dtype="bf16")
    check(sv, vb, params(vb.B, 1.0, 0, 0.9, 0.0, seed=9))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unfiltered_rows_not_block_aligned(dtype):
    """Rows whose aligned body does not start on a Philox block (odd leading
    dimension): per-element noise instead of whole-vector blocks."""
    sv = need_gpu()
    V = 152064 if dtype == "bf16" else 60000
    vb = W.ragged_batch(seed=41, B=5, k_max=3, V=V, dtype=dtype, ld=V + 3)
    for T in (0.5, 1.0):
        check(sv, vb, params(vb.B, T, 0, 1.0, 0.0, seed=3))


def test_back_to_back_calls_share_a_workspace():
    """Three different batches of one shape queued back to back on one stream
    with one workspace and no synchronisation between them: the records
    kernel of a call waits for the previous call's finish before it
    rewrites the row records, so every call matches the oracle on its own
    inputs."""
    sv = need_gpu()
    cases = []
    for i, (T, k, tp, mp) in enumerate([(1.0, 50, 1.0, 0.0), (0.5, 0, 0.9, 0.0), (0.0, 0, 1.0, 0.0)]):
        vb = W.ragged_batch(seed=60 + i, B=24, k_max=4, V=152064, dtype="bf16",
                            k_values=np.array([4, 0, 3, 1, 2, 4] * 4))
        cases.append((vb, params(vb.B, T, k, tp, mp, seed=70 + i, step=i)))
    R = max(vb.logits.shape[0] for vb, _ in cases)
    B = max(vb.B for vb, _ in cases)
    ws = sv.new_workspace(R, B, 152064, "bf16", sampling=True)
    outs = []
    for vb, p in cases:
        assert vb.logits.shape[0] == R and vb.B == B
        outs.append(run_sample(sv, vb, p, rows=True, workspace=ws))
    for (vb, p), res in zip(cases, outs):
        ref = oracle.verify_sample(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows,
                                   vb.draft_ids, p)
        got = host(res)
        assert compare_sampled(vb, p, got, ref, label="back to back") == 0
        assert got["status"][0] == ref.status


@pytest.mark.parametrize("dtype,V", [("bf16", 1_048_000), ("f32", 524_000)])
def test_longest_rows(dtype, V):
    """Rows near the 2 MiB limit (64 chunks): bf16 top-p-alone rows span more
    chunks than the finish stages counts for and take the exact whole-row
    selects; the other filters settle from the chunk summaries as usual."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=V % 1000, B=2, k_max=2, V=V, dtype=dtype, k_values=np.array([2, 1]))
    for T, k, tp, mp in [(1.0, 0, 0.9, 0.0), (0.7, 50, 1.0, 0.05), (0.7, 0, 1.0, 0.0), (0.0, 0, 1.0, 0.0)]:
        check(sv, vb, params(vb.B, T, k, tp, mp, seed=int(T * 10) + k), label="V=%d %s" % (V, dtype))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_more_rows_than_a_grid_dimension_holds(dtype):
    """More than 65535 packed rows of a short vocabulary, mixed filters: the
    records kernel's and the chunk-major stream grid's row index past 2^16,
    and 14000 request tickets."""
    sv = need_gpu()
    vb = W.ragged_batch(seed=71, B=14000, k_max=8, V=64, dtype=dtype)
    assert vb.R > 65535
    rng = np.random.default_rng(72)
    p = W.random_sample_params(rng, vb.B, top_ks=(0, 5, 20), top_ps=(1.0, 0.9), min_ps=(0.0, 0.05))
    got, _ = check(sv, vb, p, label="R=%d %s" % (vb.R, dtype))
    assert got["n_differ"] == 0
