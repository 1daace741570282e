"""Thin ctypes binding of libspecverify (include/spec_verify.h).

Argument marshalling only: every step of verification runs in the CUDA
kernels of libspecverify.so.  PyTorch supplies device memory and the current
stream.  There is no CPU fallback: if the library is missing or no CUDA
device is present, the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np
import torch

from . import _build

_LIB_PATH = _build.OUT

SPEC_F32, SPEC_BF16 = 0, 1
RESULT_NAMES = {0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARG", 2: "SPEC_ERR_UNSUPPORTED",
                3: "SPEC_ERR_CUDA", 4: "SPEC_ERR_WORKSPACE"}

STATUS_BAD_TEMPERATURE = 0x1
STATUS_BAD_TOP_K = 0x2
STATUS_BAD_TOP_P = 0x4
STATUS_BAD_MIN_P = 0x8
STATUS_BAD_ROWS = 0x10
STATUS_BAD_SELECTED = 0x20
STATUS_BAD_RELAXED_K = 0x40
STATUS_BAD_BUDGET = 0x80
STATUS_TIMEOUT = 0x100
STATUS_BAD_MARGIN = 0x200

EXPORTS = ["spec_workspace_bytes", "spec_draft_workspace_bytes", "spec_verify_greedy",
           "spec_verify_greedy_noalloc", "spec_verify_relaxed_topk",
           "spec_verify_greedy_margin", "spec_verify_greedy_active", "spec_verify_sample",
           "spec_draft_confidence", "spec_prefix_stats", "spec_restore_rows",
           "spec_result_string", "spec_last_cuda_error", "spec_abi_version",
           "spec_step_state_bytes", "spec_step_init", "spec_step_update", "spec_step_query",
           "spec_step_cost_sps", "spec_step_cost_additive"]


class SpecError(RuntimeError):
    pass


class Batch(C.Structure):
    _fields_ = [("logits", C.c_void_p), ("dtype", C.c_int32), ("V", C.c_int32),
                ("ld", C.c_int64), ("B", C.c_int32), ("k_max", C.c_int32),
                ("R_cap", C.c_int32), ("cu_rows", C.c_void_p), ("draft_ids", C.c_void_p)]


class Outputs(C.Structure):
    _fields_ = [("accepted_len", C.c_void_p), ("out_tokens", C.c_void_p),
                ("next_token", C.c_void_p), ("row_max", C.c_void_p), ("row_lse", C.c_void_p),
                ("row_argmax", C.c_void_p), ("row_token", C.c_void_p), ("status", C.c_void_p),
                ("acc", C.c_void_p), ("ver", C.c_void_p), ("hist", C.c_void_p)]


class Sampling(C.Structure):
    _fields_ = [("temperature", C.c_void_p), ("top_k", C.c_void_p), ("top_p", C.c_void_p),
                ("min_p", C.c_void_p), ("seed", C.c_void_p), ("request_id", C.c_void_p),
                ("step", C.c_uint32)]


class Margin(C.Structure):
    _fields_ = [("margin", C.c_void_p), ("generated", C.c_void_p),
                ("protected_ids", C.c_void_p), ("n_protected", C.c_int32),
                ("from_position", C.c_int32), ("after_tokens", C.c_int32)]


class StepPolicy(C.Structure):
    _fields_ = [("k_min", C.c_int32), ("k_max", C.c_int32), ("k_init", C.c_int32),
                ("window_size", C.c_int32), ("update_interval", C.c_int32),
                ("switch_min_gain", C.c_double)]


class Draft(C.Structure):
    _fields_ = [("draft_logits", C.c_void_p), ("dtype", C.c_int32), ("V", C.c_int32),
                ("ld", C.c_int64), ("B", C.c_int32), ("k", C.c_int32),
                ("selected", C.c_void_p), ("threshold", C.c_float), ("max_rows", C.c_int32)]


class Allocation(C.Structure):
    _fields_ = [("conf", C.c_void_p), ("draft_token", C.c_void_p), ("k_alloc", C.c_void_p),
                ("cu_rows", C.c_void_p), ("row_owner", C.c_void_p), ("row_pos", C.c_void_p),
                ("packed_draft", C.c_void_p), ("total_rows", C.c_void_p),
                ("status", C.c_void_p)]


_lib = None


def load_library(path: Optional[str] = None) -> C.CDLL:
    """Load libspecverify.so (no device needed).  Raises if it was not built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise SpecError("libspecverify.so is not built (%s); run the package build first" % p)
    L = C.CDLL(p)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    L.spec_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.spec_draft_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.spec_draft_workspace_bytes.restype = C.c_size_t
    L.spec_workspace_bytes.restype = C.c_size_t
    L.spec_verify_greedy.argtypes = [C.POINTER(Batch), C.POINTER(Outputs), vp, C.c_size_t, vp]
    L.spec_verify_greedy_noalloc.argtypes = [C.POINTER(Batch), C.POINTER(Outputs), vp]
    L.spec_verify_relaxed_topk.argtypes = [C.POINTER(Batch), vp, C.POINTER(Outputs), vp,
                                           C.c_size_t, vp]
    L.spec_verify_greedy_active.argtypes = [C.POINTER(Batch), vp, C.POINTER(Outputs), vp,
                                            C.c_size_t, vp]
    L.spec_verify_greedy_margin.argtypes = [C.POINTER(Batch), C.POINTER(Margin),
                                            C.POINTER(Outputs), vp, C.c_size_t, vp]
    L.spec_verify_sample.argtypes = [C.POINTER(Batch), C.POINTER(Sampling), C.POINTER(Outputs),
                                     vp, C.c_size_t, vp]
    L.spec_draft_confidence.argtypes = [C.POINTER(Draft), C.POINTER(Allocation), vp, C.c_size_t,
                                        vp]
    L.spec_prefix_stats.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp]
    L.spec_restore_rows.argtypes = [vp, i64, i32, vp, i32, i32, i64, vp, i64, vp, vp]
    L.spec_restore_rows.restype = C.c_int
    for f in ["spec_verify_greedy", "spec_verify_greedy_noalloc", "spec_verify_relaxed_topk",
              "spec_verify_greedy_margin", "spec_verify_greedy_active", "spec_verify_sample",
              "spec_draft_confidence", "spec_prefix_stats", "spec_abi_version"]:
        getattr(L, f).restype = C.c_int
    L.spec_step_state_bytes.restype = C.c_size_t
    L.spec_step_state_bytes.argtypes = []
    L.spec_step_init.argtypes = [vp, C.c_size_t, C.POINTER(StepPolicy)]
    L.spec_step_update.argtypes = [vp, vp, vp, vp, i32, vp]
    L.spec_step_query.argtypes = [vp, vp, vp, vp]
    L.spec_step_cost_sps.argtypes = [i32, i32, vp, vp, i32, vp]
    L.spec_step_cost_additive.argtypes = [i32, i32, C.c_double, vp, vp, i32, vp, vp, i32, vp]
    for f in ["spec_step_init", "spec_step_update", "spec_step_query", "spec_step_cost_sps",
              "spec_step_cost_additive"]:
        getattr(L, f).restype = C.c_int
    L.spec_result_string.argtypes = [C.c_int]
    L.spec_result_string.restype = C.c_char_p
    L.spec_last_cuda_error.restype = C.c_char_p
    if path is None:
        _lib = L
    return L


def _check(rc: int):
    if rc != 0:
        L = load_library()
        msg = RESULT_NAMES.get(rc, str(rc))
        if rc == 3:
            msg += ": " + L.spec_last_cuda_error().decode()
        raise SpecError(msg)


def _dev(t: Optional[torch.Tensor], what: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise SpecError("%s must be a CUDA tensor" % what)
    if dtype is not None and t.dtype != dtype:
        raise SpecError("%s must have dtype %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise SpecError("%s must be contiguous" % what)
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _logits_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16 or t.dtype == torch.int16 or t.dtype == torch.uint16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise SpecError("logits must be float32 or bfloat16, got %s" % t.dtype)


def workspace_bytes(R_cap: int, B: int, V: int, dtype=SPEC_BF16, sampling: bool = False) -> int:
    return int(load_library().spec_workspace_bytes(int(R_cap), int(B), int(V), int(dtype),
                                                   int(bool(sampling))))


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return SPEC_F32 if dtype in (torch.float32, "f32") else SPEC_BF16


def new_workspace(R_cap: int, B: int, V: int, dtype=SPEC_BF16, device=None,
                  sampling: bool = False) -> torch.Tensor:
    """Zero-filled workspace for the verify calls (reusable, stream-ordered);
    sampling=True sizes it for spec_verify_sample."""
    n = workspace_bytes(R_cap, B, V, _dtype_code(dtype), sampling)
    if n == 0:
        raise SpecError("invalid workspace size for R_cap=%d B=%d V=%d" % (R_cap, B, V))
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def new_draft_workspace(B: int, k: int, V: int, dtype=SPEC_BF16, device=None) -> torch.Tensor:
    n = int(load_library().spec_draft_workspace_bytes(int(B), int(k), int(V), _dtype_code(dtype)))
    if n == 0:
        raise SpecError("invalid draft workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids) -> Batch:
    if logits.dim() != 2:
        raise SpecError("logits must be 2-D [rows, ld]")
    if logits.stride(1) != 1:
        raise SpecError("logits rows must be contiguous")
    return Batch(_dev(logits, "logits"), _logits_dtype(logits), int(V), int(logits.stride(0)),
                 int(B), int(k_max), int(R_cap), _dev(cu_rows, "cu_rows", torch.int32),
                 _dev(draft_ids, "draft_ids", torch.int32))


def _outputs(B, k_max, R_cap, device, rows: bool, stats) -> tuple:
    # the request outputs and the status word in one int32 buffer
    # ("request_block"), so one copy brings them to the host
    blk = torch.zeros(B * (k_max + 3) + 1, dtype=torch.int32, device=device)
    res = {
        "accepted_len": blk[:B],
        "out_tokens": blk[B:B * (k_max + 2)].view(B, k_max + 1),
        "next_token": blk[B * (k_max + 2):B * (k_max + 3)],
        "status": blk[B * (k_max + 3):],
        "request_block": blk,
    }
    if rows:
        res["row_max"] = torch.empty(R_cap, dtype=torch.float32, device=device)
        res["row_lse"] = torch.empty(R_cap, dtype=torch.float32, device=device)
        res["row_argmax"] = torch.empty(R_cap, dtype=torch.int32, device=device)
        res["row_token"] = torch.empty(R_cap, dtype=torch.int32, device=device)
    o = Outputs(res["accepted_len"].data_ptr(), res["out_tokens"].data_ptr(),
                res["next_token"].data_ptr(),
                res["row_max"].data_ptr() if rows else None,
                res["row_lse"].data_ptr() if rows else None,
                res["row_argmax"].data_ptr() if rows else None,
                res["row_token"].data_ptr() if rows else None,
                res["status"].data_ptr(), None, None, None)
    if stats is not None:
        acc, ver, hist = stats
        o.acc = _dev(acc, "acc", torch.int64)
        o.ver = _dev(ver, "ver", torch.int64)
        o.hist = _dev(hist, "hist", torch.int64)
    return o, res


def verify_greedy(logits, cu_rows, draft_ids, *, V: int, B: int, k_max: int,
                  R_cap: Optional[int] = None, workspace=None, rows: bool = True, stats=None,
                  stream=None) -> dict:
    """spec_verify_greedy: fused max/LSE/argmax per row, then greedy prefix
    acceptance per request.  Returns a dict of device tensors: accepted_len,
    out_tokens, next_token and status are views of one int32 block
    ("request_block", in that order), so one copy brings them to the host;
    with rows=True also row_max, row_lse, row_argmax and row_token."""
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    ws = workspace if workspace is not None else new_workspace(
        R_cap, B, V, _logits_dtype(logits), logits.device)
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    _check(L.spec_verify_greedy(C.byref(b), C.byref(o), ws.data_ptr(), ws.numel(), _stream(stream)))
    return res


def verify_greedy_noalloc(logits, cu_rows, draft_ids, *, V: int, B: int, k_max: int,
                          R_cap: Optional[int] = None, rows: bool = True, stats=None,
                          stream=None) -> dict:
    """spec_verify_greedy_noalloc: greedy verification for callers that cannot
    allocate device memory; the library's built-in scratch array stands in
    for the workspace.  Calls that overlap on the GPU race on that array.
    The array used is the current device's, so logits must be on it."""
    if logits.device.type != "cuda":
        raise SpecError("verify_greedy_noalloc: logits must be a CUDA tensor, got %s" % logits.device)
    cur = torch.cuda.current_device()
    if logits.device.index != cur:
        raise SpecError("verify_greedy_noalloc: logits are on %s but the current device is "
                        "cuda:%d (the built-in scratch array is the current device's)"
                        % (logits.device, cur))
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    _check(L.spec_verify_greedy_noalloc(C.byref(b), C.byref(o), _stream(stream)))
    return res


def verify_relaxed_topk(logits, cu_rows, draft_ids, relaxed_k, *, V: int, B: int, k_max: int,
                        R_cap: Optional[int] = None, workspace=None, rows: bool = True,
                        stats=None, stream=None) -> dict:
    """spec_verify_relaxed_topk: accept d iff #{z > z_d} < K_b, strict prefix."""
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    ws = workspace if workspace is not None else new_workspace(
        R_cap, B, V, _logits_dtype(logits), logits.device)
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    _check(L.spec_verify_relaxed_topk(C.byref(b), _dev(relaxed_k, "relaxed_k", torch.int32),
                                      C.byref(o), ws.data_ptr(), ws.numel(), _stream(stream)))
    return res


def verify_greedy_active(logits, cu_rows, draft_ids, vocab_ids, *, V: int, B: int, k_max: int,
                         R_cap: Optional[int] = None, workspace=None, rows: bool = True,
                         stats=None, stream=None) -> dict:
    """spec_verify_greedy_active: greedy verification over V active columns,
    column i standing for full token id vocab_ids[i]; drafts and outputs are
    full ids."""
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    ws = workspace if workspace is not None else new_workspace(
        R_cap, B, V, _logits_dtype(logits), logits.device)
    if vocab_ids is None or vocab_ids.numel() < V:
        raise SpecError("vocab_ids needs one full id per active column")
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    _check(L.spec_verify_greedy_active(C.byref(b), _dev(vocab_ids, "vocab_ids", torch.int32),
                                       C.byref(o), ws.data_ptr(), ws.numel(), _stream(stream)))
    return res


def verify_greedy_margin(logits, cu_rows, draft_ids, margin, generated=None, protected_ids=None,
                         from_position: int = 0, after_tokens: int = 0, *, V: int, B: int,
                         k_max: int, R_cap: Optional[int] = None, workspace=None,
                         rows: bool = True, stats=None, stream=None) -> dict:
    """spec_verify_greedy_margin: greedy acceptance that also passes a draft
    within margin[b] of the row maximum at eligible positions, never for a
    protected token id; strict prefix."""
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    ws = workspace if workspace is not None else new_workspace(
        R_cap, B, V, _logits_dtype(logits), logits.device)
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    n_prot = 0 if protected_ids is None else int(protected_ids.numel())
    m = Margin(_dev(margin, "margin", torch.float32),
               _dev(generated, "generated", torch.int32),
               _dev(protected_ids, "protected_ids", torch.int32) if n_prot else None,
               n_prot, int(from_position), int(after_tokens))
    _check(L.spec_verify_greedy_margin(C.byref(b), C.byref(m), C.byref(o), ws.data_ptr(),
                                       ws.numel(), _stream(stream)))
    return res


def verify_sample(logits, cu_rows, draft_ids, temperature, top_k, top_p, min_p, seed,
                  request_id=None, step: int = 0, *, V: int, B: int, k_max: int,
                  R_cap: Optional[int] = None, workspace=None, rows: bool = True, stats=None,
                  stream=None) -> dict:
    """spec_verify_sample: filtered Gumbel-max sampling per row (Philox4x32-10
    uniforms) and the point-mass rejection chain per request.  `seed` is an
    int64 tensor holding the 64-bit seeds' bit patterns."""
    L = load_library()
    R_cap = R_cap or B * (k_max + 1)
    ws = workspace if workspace is not None else new_workspace(
        R_cap, B, V, _logits_dtype(logits), logits.device, sampling=True)
    b = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
    s = Sampling(_dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
                 _dev(top_p, "top_p", torch.float32), _dev(min_p, "min_p", torch.float32),
                 _dev(seed, "seed", torch.int64),
                 _dev(request_id, "request_id", torch.int32) if request_id is not None else None,
                 int(step) & 0xFFFFFFFF)
    o, res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
    _check(L.spec_verify_sample(C.byref(b), C.byref(s), C.byref(o), ws.data_ptr(), ws.numel(),
                                _stream(stream)))
    return res


def draft_confidence(draft_logits, *, V: int, B: int, k: int, selected=None,
                     threshold: float = 0.3, max_rows: int = 0, workspace=None,
                     stream=None) -> dict:
    """spec_draft_confidence: conf = exp(z[s] - logsumexp(z)) per draft row,
    then device-side prefix allocation and packing."""
    L = load_library()
    dev = draft_logits.device
    if draft_logits.dim() != 2 or draft_logits.stride(1) != 1:
        raise SpecError("draft_logits must be 2-D with contiguous rows")
    d = Draft(_dev(draft_logits, "draft_logits"), _logits_dtype(draft_logits), int(V),
              int(draft_logits.stride(0)), int(B), int(k),
              _dev(selected, "selected", torch.int32) if selected is not None else None,
              float(threshold), int(max_rows))
    cap = B * (k + 1)
    res = {
        "conf": torch.empty(B * k, dtype=torch.float32, device=dev),
        "draft_token": torch.empty(B * k, dtype=torch.int32, device=dev),
        "k_alloc": torch.empty(B, dtype=torch.int32, device=dev),
        "cu_rows": torch.empty(B + 1, dtype=torch.int32, device=dev),
        "row_owner": torch.empty(cap, dtype=torch.int32, device=dev),
        "row_pos": torch.empty(cap, dtype=torch.int32, device=dev),
        "packed_draft": torch.empty(cap, dtype=torch.int32, device=dev),
        "total_rows": torch.empty(1, dtype=torch.int32, device=dev),
        "status": torch.zeros(1, dtype=torch.int32, device=dev),
    }
    a = Allocation(*[res[n].data_ptr() for n in ["conf", "draft_token", "k_alloc", "cu_rows",
                                                  "row_owner", "row_pos", "packed_draft",
                                                  "total_rows", "status"]])
    ws = workspace if workspace is not None else new_draft_workspace(
        B, k, V, _logits_dtype(draft_logits), dev)
    _check(L.spec_draft_confidence(C.byref(d), C.byref(a), ws.data_ptr(), ws.numel(),
                                   _stream(stream)))
    return res


def restore_rows(compact: torch.Tensor, cu_rows, out: torch.Tensor, *, B: int, k_max: int,
                 status=None, stream=None) -> torch.Tensor:
    """spec_restore_rows: compact row cu_rows[b] + j goes to row
    b * (k_max + 1) + j of `out` for j <= k_b; other rows of `out` are left
    as they are.  compact [R_cap, H] and out [B * (k_max + 1), H] are 2-D
    device tensors of one dtype whose rows are 16-byte multiples."""
    L = load_library()
    if compact.dim() != 2 or out.dim() != 2 or compact.dtype != out.dtype:
        raise SpecError("compact and out must be 2-D tensors of one dtype")
    if compact.shape[1] != out.shape[1] or out.shape[0] < B * (k_max + 1):
        raise SpecError("out needs B * (k_max + 1) rows of the compact row width")
    if compact.stride(1) != 1 or out.stride(1) != 1:
        raise SpecError("rows must be contiguous")
    for x, what in [(compact, "compact"), (out, "out")]:
        if not x.is_cuda:
            raise SpecError("%s must be a CUDA tensor" % what)
    es = compact.element_size()
    _check(L.spec_restore_rows(compact.data_ptr(), compact.stride(0) * es, compact.shape[0],
                               _dev(cu_rows, "cu_rows", torch.int32), B, k_max,
                               compact.shape[1] * es, out.data_ptr(), out.stride(0) * es,
                               _dev(status, "status", torch.int32), _stream(stream)))
    return out


def prefix_stats(accepted_len, cu_rows, acc, ver, hist=None, status=None, *, B: int, k_max: int,
                 stream=None):
    """spec_prefix_stats: accumulate per-position prefix-acceptance counters
    (int64 tensors acc[k_max], ver[k_max], hist[k_max+1]) in place."""
    L = load_library()
    _check(L.spec_prefix_stats(_dev(accepted_len, "accepted_len", torch.int32),
                               _dev(cu_rows, "cu_rows", torch.int32), int(B), int(k_max),
                               _dev(acc, "acc", torch.int64), _dev(ver, "ver", torch.int64),
                               _dev(hist, "hist", torch.int64) if hist is not None else None,
                               _dev(status, "status", torch.int32) if status is not None else None,
                               _stream(stream)))


class PreparedSample:
    """A spec_verify_sample call with every argument marshalled once; each
    __call__ swaps only the logits pointer and the step word, so a loop of
    calls costs one ctypes call per launch (for benchmarking and serving
    loops).  The tensors passed here must stay alive while it is used."""

    def __init__(self, logits, cu_rows, draft_ids, temperature, top_k, top_p, min_p, seed,
                 request_id=None, *, V: int, B: int, k_max: int, R_cap: Optional[int] = None,
                 workspace=None, rows: bool = True, stats=None, stream=None):
        self.L = load_library()
        R_cap = R_cap or B * (k_max + 1)
        self.ws = workspace if workspace is not None else new_workspace(
            R_cap, B, V, _logits_dtype(logits), logits.device, sampling=True)
        self.batch = _batch(logits, V, B, k_max, R_cap, cu_rows, draft_ids)
        self.samp = Sampling(_dev(temperature, "temperature", torch.float32),
                             _dev(top_k, "top_k", torch.int32), _dev(top_p, "top_p", torch.float32),
                             _dev(min_p, "min_p", torch.float32), _dev(seed, "seed", torch.int64),
                             _dev(request_id, "request_id", torch.int32)
                             if request_id is not None else None, 0)
        self.out, self.res = _outputs(B, k_max, R_cap, logits.device, rows, stats)
        self.stream = _stream(stream)
        self._keep = (logits, cu_rows, draft_ids, temperature, top_k, top_p, min_p, seed,
                      request_id, stats)
        self._args = (C.byref(self.batch), C.byref(self.samp), C.byref(self.out),
                      C.c_void_p(self.ws.data_ptr()), C.c_size_t(self.ws.numel()),
                      C.c_void_p(self.stream))

    def __call__(self, logits=None, step: int = 0) -> dict:
        if logits is not None:
            self.batch.logits = logits.data_ptr()
        self.samp.step = int(step) & 0xFFFFFFFF
        rc = self.L.spec_verify_sample(*self._args)
        if rc:
            _check(rc)
        return self.res


# ------------------------------------------------------------------------
# adaptive draft-step controller (host code in the library; no GPU needed)
# ------------------------------------------------------------------------

def _host(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(C.c_void_p)


class StepController:
    """spec_step_init / spec_step_update / spec_step_query: one speculative
    step count per batch from the windowed prefix acceptance of completed
    batches and the full-step cost of each candidate."""

    def __init__(self, k_min: int, k_max: int, k_init: int, window_size: int = 20,
                 update_interval: int = 5, switch_min_gain: float = 0.05):
        L = load_library()
        self.k_max = k_max
        self._state = np.zeros((L.spec_step_state_bytes() + 7) // 8, np.uint64)
        pol = StepPolicy(k_min, k_max, k_init, window_size, update_interval, switch_min_gain)
        _check(L.spec_step_init(self._state.ctypes.data_as(C.c_void_p), self._state.nbytes,
                                C.byref(pol)))

    def update(self, acc, ver, cost_ms, B: int) -> int:
        L = load_library()
        a, pa = _host(acc, np.int64)
        v, pv = _host(ver, np.int64)
        c, pc = _host(cost_ms, np.float64)
        k = C.c_int32(0)
        _check(L.spec_step_update(self._state.ctypes.data_as(C.c_void_p), pa, pv, pc, int(B),
                                  C.byref(k)))
        return int(k.value)

    def query(self):
        """(prefix_acceptance [k_max], score [k_max + 1], current k)."""
        L = load_library()
        pa = np.zeros(max(self.k_max, 1), np.float64)
        sc = np.zeros(self.k_max + 1, np.float64)
        k = C.c_int32(0)
        _check(L.spec_step_query(self._state.ctypes.data_as(C.c_void_p),
                                 pa.ctypes.data_as(C.c_void_p), sc.ctypes.data_as(C.c_void_p),
                                 C.byref(k)))
        return pa[:self.k_max], sc, int(k.value)


def step_cost_sps(B: int, k_max: int, g_rows, sps) -> np.ndarray:
    """spec_step_cost_sps: cost_ms[k] = 1000 / SPS of the first captured
    graph size >= B (k + 1), +inf when none covers it."""
    L = load_library()
    g, pg = _host(g_rows, np.int32)
    s_, ps = _host(sps, np.float64)
    if g.size != s_.size:
        raise SpecError("g_rows and sps differ in length")
    out = np.zeros(k_max + 1, np.float64)
    _check(L.spec_step_cost_sps(int(B), int(k_max), pg, ps, int(g.size),
                                out.ctypes.data_as(C.c_void_p)))
    return out


def step_cost_additive(B: int, k_max: int, bias_s: float, b_buckets, alpha_s, g_rows,
                       theta_s) -> np.ndarray:
    """spec_step_cost_additive: cost_ms[k] = 1000 (bias + alpha(Bcap) +
    theta(G_k)) over the first covering request bucket and graph size."""
    L = load_library()
    b, pb = _host(b_buckets, np.int32)
    a, pa = _host(alpha_s, np.float64)
    g, pg = _host(g_rows, np.int32)
    t, pt = _host(theta_s, np.float64)
    if b.size != a.size or g.size != t.size:
        raise SpecError("bucket and term lists differ in length")
    out = np.zeros(k_max + 1, np.float64)
    _check(L.spec_step_cost_additive(int(B), int(k_max), float(bias_s), pb, pa, int(b.size),
                                     pg, pt, int(g.size), out.ctypes.data_as(C.c_void_p)))
    return out
