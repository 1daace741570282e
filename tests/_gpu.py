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


# a sampled token may differ from the fp64 definition only where a float
# threshold decision or the Gumbel winner is within rounding of a tie
FILTER_MARGIN = 1e-4
GUMBEL_MARGIN = 1e-4


def compare_sampled(vb, got: dict, ref, max_frac: float = 1e-4):
    R = vb.R
    g = got["row_token"][:R]
    o = ref.rows["row_token"]
    near = (ref.rows["margin_filter"] < FILTER_MARGIN) | (ref.rows["margin_gumbel"] < GUMBEL_MARGIN)
    bad = (g != o)
    assert not (bad & ~near).any(), (
        "sampled tokens differ away from float ties at rows %s" % np.nonzero(bad & ~near)[0][:10])
    assert bad.sum() <= max(1, int(max_frac * R)), "too many boundary disagreements: %d" % bad.sum()
    # requests whose rows all agree must agree exactly
    ok_req = np.array([not bad[vb.cu_rows[b]:vb.cu_rows[b + 1]].any() for b in range(vb.B)])
    assert_requests_equal(got, ref, ok_req)
    return int(bad.sum())
