"""spec_verify_greedy_noalloc: greedy verification for callers that cannot
allocate device memory (a plugin inside an engine that owns the whole device
pool, a serving loop that forbids allocation once it runs).  The library's
built-in scratch array stands in for the workspace, so the caller passes only
inputs and outputs.

The GPU test compares it with the oracle's greedy verification and with
spec_verify_greedy, which takes a caller-owned workspace, on two calls in a
row with different batches (the shared scratch keeps the previous call's
contents).  The binding refuses logits that are not on the current device
(the scratch array used is the current device's); that check runs on CPU.  This file is collected after the
other GPU files, so that a run stopping at the first failure has run them
first."""
import ctypes as C

import numpy as np
import pytest

import oracle
import workloads as W

LSE_RTOL = 1e-5


def test_oversized_batch_is_rejected_before_any_launch():
    """A batch whose workspace exceeds the built-in scratch returns
    SPEC_ERR_WORKSPACE; nothing is launched, so no device is needed."""
    import speculative_decoding_verification_ragged_gb300 as sv
    from speculative_decoding_verification_ragged_gb300.binding import Batch, Outputs
    sv.build()
    L = sv.load_library()
    fake = C.c_void_p(0x1000)
    outs = Outputs(fake, fake, fake, None, None, None, None, None, None, None, None)
    big = Batch(fake, 1, 152064, 152064, 4000, 4, 20000, fake, fake)
    assert L.spec_workspace_bytes(20000, 4000, 152064, 1, 0) > 4 * 1024 * 1024
    assert L.spec_verify_greedy_noalloc(C.byref(big), C.byref(outs), None) == 4
    bad = Batch(fake, 1, 0, 152064, 4, 4, 20, fake, fake)
    assert L.spec_verify_greedy_noalloc(C.byref(bad), C.byref(outs), None) == 1


class _FakeLogits:
    """Stands in for a tensor on another GPU: only .device is read before
    the check refuses it."""
    def __init__(self, dev):
        self.device = dev


def test_binding_refuses_logits_off_the_current_device(monkeypatch):
    torch = pytest.importorskip("torch")
    import speculative_decoding_verification_ragged_gb300 as sv
    from speculative_decoding_verification_ragged_gb300.binding import SpecError
    kw = dict(V=10, B=1, k_max=0)
    with pytest.raises(SpecError, match="CUDA tensor"):
        sv.verify_greedy_noalloc(torch.zeros(1, 10), None, None, **kw)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(SpecError, match="current device is cuda:0"):
        sv.verify_greedy_noalloc(_FakeLogits(torch.device("cuda", 1)), None, None, **kw)


def _compare_oracle(got, vb):
    ref = oracle.verify_greedy(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, vb.draft_ids)
    R = vb.R
    np.testing.assert_array_equal(got["accepted_len"].cpu().numpy(), ref.accepted_len)
    np.testing.assert_array_equal(got["out_tokens"].cpu().numpy(), ref.out_tokens)
    np.testing.assert_array_equal(got["next_token"].cpu().numpy(), ref.next_token)
    np.testing.assert_array_equal(got["row_argmax"][:R].cpu().numpy(), ref.rows["row_argmax"])
    np.testing.assert_array_equal(got["row_max"][:R].cpu().numpy(), ref.rows["row_max"].astype(np.float32))
    np.testing.assert_allclose(got["row_lse"][:R].cpu().numpy(), ref.rows["row_lse"], rtol=LSE_RTOL, atol=0)
    assert got["status"].cpu().numpy()[0] == ref.status


def _compare(got, ref, R):
    for key in ["accepted_len", "out_tokens", "next_token", "status"]:
        np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key].cpu().numpy(), err_msg=key)
    for key in ["row_argmax", "row_token", "row_max"]:
        np.testing.assert_array_equal(got[key][:R].cpu().numpy(), ref[key][:R].cpu().numpy(),
                                      err_msg=key)
    np.testing.assert_allclose(got["row_lse"][:R].cpu().numpy(), ref["row_lse"][:R].cpu().numpy(),
                               rtol=LSE_RTOL, atol=0)


@pytest.mark.gpu
def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    from tests._gpu import need_gpu, t, torch
    sv = need_gpu()
    batches = [W.planted_greedy(),
               W.ragged_batch(seed=77, B=9, k_max=6, V=30011, dtype="f32", ld=30013,
                              tie_top=True)]
    for vb in batches:
        if vb.dtype == "bf16":
            logits = torch.from_numpy(vb.logits.view(np.int16)).view(torch.bfloat16).cuda()
        else:
            logits = torch.from_numpy(vb.logits).cuda()
        cu, dr = t(vb.cu_rows), t(vb.draft_ids)
        kw = dict(V=vb.V, B=vb.B, k_max=vb.k_max, R_cap=vb.logits.shape[0])
        ref = sv.verify_greedy(logits, cu, dr, **kw)
        got = sv.verify_greedy_noalloc(logits, cu, dr, **kw)
        torch.cuda.synchronize()
        _compare_oracle(got, vb)
        _compare(got, ref, vb.R)
