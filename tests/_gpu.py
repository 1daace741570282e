"""Helpers for the GPU parity tests: move seeded inputs to the device, call
the CUDA library through its C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_ragged_gb300 as sv
    sv.build()
    return sv


def t(a, dev="cuda"):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint64:
        a = a.view(np.int64)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(dev)


def logits_tensor(x: np.ndarray, dtype: str, dev="cuda"):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)


def run_greedy(sv, vb: W.VerifyBatch, **kw):
    return sv.verify_greedy(logits_tensor(vb.logits, vb.dtype), t(vb.cu_rows), t(vb.draft_ids),
                            V=vb.V, B=vb.B, k_max=vb.k_max, R_cap=vb.logits.shape[0], **kw)


def run_relaxed(sv, vb: W.VerifyBatch, K, **kw):
    return sv.verify_relaxed_topk(logits_tensor(vb.logits, vb.dtype), t(vb.cu_rows),
                                  t(vb.draft_ids), t(np.asarray(K, np.int32)), V=vb.V, B=vb.B,
                                  k_max=vb.k_max, R_cap=vb.logits.shape[0], **kw)


def run_active(sv, vb: W.VerifyBatch, draft_ids, vocab_ids, **kw):
    return sv.verify_greedy_active(logits_tensor(vb.logits, vb.dtype), t(vb.cu_rows),
                                   t(np.asarray(draft_ids, np.int32)),
                                   t(np.asarray(vocab_ids, np.int32)), V=vb.V, B=vb.B,
                                   k_max=vb.k_max, R_cap=vb.logits.shape[0], **kw)


def run_margin(sv, vb: W.VerifyBatch, margin, generated=None, protected_ids=None, **kw):
    return sv.verify_greedy_margin(
        logits_tensor(vb.logits, vb.dtype), t(vb.cu_rows), t(vb.draft_ids),
        t(np.asarray(margin, np.float32)),
        t(np.asarray(generated, np.int32)) if generated is not None else None,
        t(np.asarray(protected_ids, np.int32)) if protected_ids is not None else None,
        V=vb.V, B=vb.B, k_max=vb.k_max, R_cap=vb.logits.shape[0], **kw)


def run_sample(sv, vb: W.VerifyBatch, p: W.SampleParams, **kw):
    return sv.verify_sample(logits_tensor(vb.logits, vb.dtype), t(vb.cu_rows), t(vb.draft_ids),
                            t(p.temperature), t(p.top_k), t(p.top_p), t(p.min_p), t(p.seed),
                            t(p.request_id) if p.request_id is not None else None, p.step,
                            V=vb.V, B=vb.B, k_max=vb.k_max, R_cap=vb.logits.shape[0], **kw)


def host(res: dict) -> dict:
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def assert_requests_equal(got: dict, ref, mask=None):
    """Bit-exact request outputs (optionally only for requests in mask)."""
    sel = slice(None) if mask is None else mask
    np.testing.assert_array_equal(got["accepted_len"][sel], ref.accepted_len[sel])
    np.testing.assert_array_equal(got["out_tokens"][sel], ref.out_tokens[sel])
    np.testing.assert_array_equal(got["next_token"][sel], ref.next_token[sel])


# ---------------------------------------------------------------------------
# Sampled tokens.  The kernels take the filter decisions and the Gumbel
# argmax in fp32; the oracle takes them in fp64.  A row may come out
# differently only where one of those decisions lies within the fp32 error
# of its boundary.  The bands below bound that error per row, from the
# operations the kernels perform (U = 2^-24, the fp32 unit roundoff):
#
#   min-p   th = M + T*logf(min_p): logf within 1 ulp (2U), the product and
#           the sum rounded once each, so |th - th_exact| <= T|ln min_p| 3U
#           + |th| U.  In ratio space (the oracle's margin is the relative
#           distance of exp((z - M)/T) from min_p) that is at most
#           (|ln min_p| 3U + |th| U / T), with 1% slack for exp(x) - 1 > x.
#   top-p   every weight exp((z - M)/T) is ex2.approx (relative error below
#           4U) of an argument (z - M) * log2(e)/T carrying 3U relative
#           (1/T, log2(e)/T and the product rounded) plus |M| log2(e)/T U
#           when M is folded into an fma constant; the sums add at most
#           kSumDepth terms in sequence.  With A = the mass-weighted mean of
#           |z - M| log2(e)/T over the row, every partial mass is within
#           e_w = ln2 U (3A + |M| log2(e)/T) + 4U + kSumDepth U of exact, and
#           the decision "mass above < top_p W" can flip only if the
#           oracle's margin |above - top_p W| / W is below 2 e_w.
#   Gumbel  score = z * (1/T) + g(u): the product carries 2U |z/T|, the sum
#           U |score|, the noise g = -log(-log u) an absolute error below
#           2^-20 (hardware log2, within 2^-22 absolute / relative).  Two
#           scores can swap only if their fp64 gap is below
#           2 (3U S + 2^-20), S = max|z|/T + 17.
U32 = 2.0 ** -24
kSumDepth = 64      # longest run of sequential fp32 additions of a mass


def sample_bands(vb, p, rows_T=None):
    """Per packed row: (filter band, Gumbel band) inside which an fp32
    implementation may decide differently from the fp64 definition."""
    R = vb.R
    owner = np.repeat(np.arange(vb.B), np.diff(vb.cu_rows))[:R]
    T = p.temperature.astype(np.float64)[owner]
    tp = p.top_p.astype(np.float64)[owner]
    mp = p.min_p.astype(np.float64)[owner]
    z = vb.logits[:R, :vb.V]
    z = W.bf16_bits_to_f32(z) if vb.dtype == "bf16" else z
    z = z.astype(np.float64)
    band_f = np.zeros(R)
    band_g = np.zeros(R)
    for r in range(R):
        if not T[r] > 0:
            continue
        zr = z[r]
        M = zr.max()
        if not np.isfinite(M):
            continue
        sc = np.log2(np.e) / T[r]
        bf = 0.0
        if mp[r] > 0:
            th = M + T[r] * np.log(mp[r])
            bf = max(bf, 1.01 * (abs(np.log(mp[r])) * 3 * U32 + abs(th) * U32 / T[r]))
        if tp[r] < 1:
            arg = (zr - M) * sc
            w = np.exp2(arg)
            A = float((w * np.abs(arg)).sum() / w.sum())
            e_w = np.log(2) * U32 * (3 * A + abs(M) * sc) + 4 * U32 + kSumDepth * U32
            bf = max(bf, 2 * e_w)
        band_f[r] = bf
        S = np.abs(zr[np.isfinite(zr)]).max() / T[r] + 17.0
        band_g[r] = 2 * (3 * U32 * S + 2.0 ** -20)
    return band_f, band_g


def compare_sampled(vb, p, got: dict, ref, max_frac: float = 1e-4, label: str = ""):
    """Row tokens against the oracle.  A row may differ only inside its
    bands (sample_bands); at most floor(max_frac * R) rows may differ at
    all.  Prints the count of differing rows and of rows whose decisions lie
    inside a band, and returns the number of differing rows."""
    R = vb.R
    g = got["row_token"][:R]
    o = ref.rows["row_token"]
    band_f, band_g = sample_bands(vb, p)
    near_f = ref.rows["margin_filter"] < band_f
    near_g = ref.rows["margin_gumbel"] < band_g
    bad = (g != o)
    print("sampled-token check %s: %d rows, %d differ (%d differ inside a filter band, %d inside "
          "a Gumbel band); %d / %d rows have a decision inside a band"
          % (label, R, bad.sum(), (bad & near_f).sum(), (bad & near_g & ~near_f).sum(),
             near_f.sum(), near_g.sum()))
    assert not (bad & ~(near_f | near_g)).any(), (
        "sampled tokens differ away from float ties at rows %s" % np.nonzero(bad & ~(near_f | near_g))[0][:10])
    assert bad.sum() <= int(max_frac * R), "too many boundary disagreements: %d" % bad.sum()
    # requests whose rows all agree must agree exactly
    ok_req = np.array([not bad[vb.cu_rows[b]:vb.cu_rows[b + 1]].any() for b in range(vb.B)])
    assert_requests_equal(got, ref, ok_req)
    return int(bad.sum())
