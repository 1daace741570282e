"""CPU-side checks of the C ABI library: it loads without a GPU and exports
every function the headers in include/ declare; argument errors are rejected
on the host before anything is launched."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
    return sorted(set(re.findall(r"SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_ragged_gb300 as sv
    sv.build()
    return sv


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ["spec_verify_greedy", "spec_verify_sample", "spec_verify_relaxed_topk",
              "spec_draft_confidence", "spec_prefix_stats"]:
        assert n in names


def test_library_exports_every_declared_symbol(sv):
    L = sv.load_library()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert sorted(sv.EXPORTS) == declared_functions()
    assert L.spec_abi_version() == 100


def test_package_exposes_a_binding_per_entry_point(sv):
    for name in sv.EXPORTS:
        if name.startswith("spec_verify_") or name in ("spec_draft_confidence", "spec_prefix_stats"):
            assert callable(getattr(sv, name[len("spec_"):])), name


def test_workspace_bytes(sv):
    L = sv.load_library()
    # 640 rows of V = 152064 bf16: 10 chunks of 32 KiB per row
    base = 2 * 2560 + 512 + 640 * 64 + 640 * 10 * 32
    assert L.spec_workspace_bytes(640, 128, 152064, 1, 0) == base
    assert L.spec_workspace_bytes(640, 128, 152064, 1, 1) == base + 640 * 10 * 512 * 8
    assert L.spec_workspace_bytes(640, 128, 152064, 0, 0) == 2 * 2560 + 512 + 640 * 64 + 640 * 19 * 32
    assert L.spec_workspace_bytes(0, 128, 100, 1, 0) == 0
    assert L.spec_workspace_bytes(10, 0, 100, 1, 1) == 0
    assert L.spec_workspace_bytes(10, 1, 100, 9, 1) == 0
    assert L.spec_draft_workspace_bytes(16, 7, 151552, 1) == (
        2 * 512 + 256 + 112 * 64 + ((112 * 10 * 32 + 255) // 256) * 256)


def test_host_argument_errors_launch_nothing(sv):
    """Invalid arguments return an error code before any CUDA call, so these
    run without a device."""
    from speculative_decoding_verification_ragged_gb300.binding import Batch, Outputs, Sampling
    L = sv.load_library()
    fake = C.c_void_p(0x1000)
    good = dict(logits=fake, dtype=1, V=100, ld=100, B=2, k_max=3, R_cap=8, cu_rows=fake,
                draft_ids=fake)
    outs = Outputs(fake, fake, fake, None, None, None, None, None, None, None, None)
    ws = C.c_void_p(0x2000)
    n = L.spec_workspace_bytes(8, 2, 100, 1, 0)

    def call(**over):
        b = Batch(**{**good, **over})
        return L.spec_verify_greedy(C.byref(b), C.byref(outs), ws, n, None)

    assert call(V=0) == 1
    assert call(ld=99) == 1
    assert call(B=0) == 1
    assert call(k_max=32) == 2
    assert call(dtype=7) == 2
    assert call(cu_rows=None) == 1
    assert call(V=10_000_000, ld=10_000_000) == 2
    assert call(V=2_000_000, ld=2_000_000) == 2       # 4 MB bf16 row: beyond 2 MiB
    assert call(logits=C.c_void_p(0x1001)) == 1      # bf16 pointer not 2-byte aligned
    b = Batch(**good)
    assert L.spec_verify_greedy(C.byref(b), C.byref(outs), ws, n - 1, None) == 4
    assert L.spec_verify_greedy(C.byref(b), C.byref(outs), None, n, None) == 4
    assert L.spec_verify_greedy(None, C.byref(outs), ws, n, None) == 1
    s = Sampling(fake, None, fake, fake, fake, None, 0)
    assert L.spec_verify_sample(C.byref(b), C.byref(s), C.byref(outs), ws, n, None) == 1
    assert L.spec_verify_relaxed_topk(C.byref(b), None, C.byref(outs), ws, n, None) == 1
    assert L.spec_verify_greedy_active(C.byref(b), None, C.byref(outs), ws, n, None) == 1
    assert L.spec_verify_greedy_active(C.byref(b), fake, C.byref(outs), ws, n - 1, None) == 4
    from speculative_decoding_verification_ragged_gb300.binding import Margin
    for m, rc in [(Margin(None, None, None, 0, 0, 0), 1), (Margin(fake, None, None, -1, 0, 0), 1),
                  (Margin(fake, None, None, 3, 0, 0), 1)]:
        assert L.spec_verify_greedy_margin(C.byref(b), C.byref(m), C.byref(outs), ws, n, None) == rc
    m = Margin(fake, None, fake, 3, 1, 4)
    assert L.spec_verify_greedy_margin(C.byref(b), C.byref(m), C.byref(outs), ws, n - 1, None) == 4
    assert L.spec_verify_greedy_margin(C.byref(b), None, C.byref(outs), ws, n, None) == 1
    assert L.spec_prefix_stats(fake, fake, 4, 40, fake, fake, None, None, None) == 2
    # restore: every case below fails its host checks, so nothing launches
    rr, big = L.spec_restore_rows, C.c_void_p(0x10000)
    assert rr(None, 64, 8, fake, 2, 3, 64, big, 64, None, None) == 1
    assert rr(big, 64, 8, fake, 0, 3, 64, big, 64, None, None) == 1
    assert rr(big, 32, 8, fake, 2, 3, 64, big, 64, None, None) == 1      # stride < row
    assert rr(big, 64, 8, fake, 2, 32, 64, big, 64, None, None) == 2     # k_max > 31
    assert rr(big, 64, 8, fake, 2, 3, 56, big, 64, None, None) == 2      # row not 16-byte
    assert rr(big, 72, 8, fake, 2, 3, 64, big, 72, None, None) == 2      # stride not 16-byte
    assert rr(C.c_void_p(0x10008), 64, 8, fake, 2, 3, 64, big, 64, None, None) == 2
    assert rr(big, 64, 8, fake, 1 << 28, 31, 64, big, 64, None, None) == 2   # too many slots
    assert L.spec_prefix_stats(fake, fake, 0, 4, fake, fake, None, None, None) == 1
    assert L.spec_result_string(4) == b"SPEC_ERR_WORKSPACE"


def test_binding_rejects_bad_tensors_before_any_call(sv):
    """The Python binding checks devices, dtypes and shapes of the new entry
    points' tensors before calling the library (CPU tensors never reach it)."""
    import torch
    from speculative_decoding_verification_ragged_gb300 import SpecError
    x = torch.zeros(10, 8)
    cu = torch.tensor([0, 5, 10], dtype=torch.int32)
    d = torch.zeros(10, dtype=torch.int32)
    with pytest.raises(SpecError):
        sv.verify_greedy_margin(x, cu, d, torch.zeros(2), V=8, B=2, k_max=4,
                                workspace=torch.zeros(1, dtype=torch.uint8))
    with pytest.raises(SpecError):                    # map shorter than the active columns
        sv.verify_greedy_active(x, cu, d, torch.zeros(7, dtype=torch.int32), V=8, B=2, k_max=4,
                                workspace=torch.zeros(1, dtype=torch.uint8))
    with pytest.raises(SpecError):                    # one dtype for both buffers
        sv.restore_rows(torch.zeros(4, 8), cu, torch.zeros(8, 8, dtype=torch.float64), B=2, k_max=3)
    with pytest.raises(SpecError):                    # out too short for B * (k_max + 1) slots
        sv.restore_rows(torch.zeros(4, 8), cu, torch.zeros(7, 8), B=2, k_max=3)
    with pytest.raises(SpecError):                    # row widths differ
        sv.restore_rows(torch.zeros(4, 8), cu, torch.zeros(8, 4), B=2, k_max=3)
    with pytest.raises(SpecError):                    # host tensors
        sv.restore_rows(torch.zeros(4, 8), cu, torch.zeros(8, 8), B=2, k_max=3)
