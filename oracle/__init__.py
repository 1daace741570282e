"""CPU oracle for ragged speculative-decoding verification (test infrastructure).

ONLY the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product path (the CUDA library and its binding) never imports, links or runs
it; the two share no code -- only the seeded input generators in
``workloads`` feed both.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64, full sorts), built
with gcc into ``liboracle.so`` next to this file.  This module only marshals
numpy arrays.  Each wrapper names the page passage it follows; the C file's
header lists the passages and the readings taken where the pages are silent.

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, library routines, brute force over tiny
inputs and distribution tests; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# status bits of the documented contract (the oracle's own copy)
BAD_TEMPERATURE = 0x1
BAD_TOP_K = 0x2
BAD_TOP_P = 0x4
BAD_MIN_P = 0x8
BAD_ROWS = 0x10
BAD_SELECTED = 0x20
BAD_RELAXED_K = 0x40
BAD_BUDGET = 0x80
BAD_MARGIN = 0x200


def build(force: bool = False) -> str:
    """Compile spec_oracle.c with gcc (OpenMP when available)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        p = C.c_void_p
        i32, i64, u32, f64 = C.c_int32, C.c_int64, C.c_uint32, C.c_double
        L.oracle_threads.argtypes = [C.c_int]
        L.oracle_threads.restype = C.c_int
        L.oracle_philox4x32_10.argtypes = [p, p, p]
        L.oracle_philox4x32_10.restype = None
        L.oracle_uniform.argtypes = [u32]
        L.oracle_uniform.restype = f64
        L.oracle_token_uniform.argtypes = [C.c_uint64, u32, u32, u32, u32]
        L.oracle_token_uniform.restype = f64
        L.oracle_row_reduce.argtypes = [p, C.c_int, i64, i32, i32, p, p, p]
        L.oracle_row_reduce.restype = None
        L.oracle_verify_greedy.argtypes = [p, C.c_int, i64, i32, i32, i32, p, p, p, p, p, p, p, p]
        L.oracle_verify_greedy.restype = u32
        L.oracle_filter_row.argtypes = [p, i32, f64, i32, f64, f64, p, p]
        L.oracle_filter_row.restype = None
        L.oracle_sample_row.argtypes = [p, i32, f64, i32, f64, f64, C.c_uint64, u32, u32, u32,
                                        p, p, p]
        L.oracle_sample_row.restype = i32
        L.oracle_verify_sample.argtypes = [p, C.c_int, i64, i32, i32, i32, p, p,
                                           p, p, p, p, p, p, u32,
                                           p, p, p, p, p, p]
        L.oracle_verify_sample.restype = u32
        L.oracle_verify_relaxed.argtypes = [p, C.c_int, i64, i32, i32, i32, p, p, p,
                                            p, p, p, p, p]
        L.oracle_verify_relaxed.restype = u32
        L.oracle_verify_greedy_active.argtypes = [p, C.c_int, i64, i32, i32, i32, p, p, p,
                                                  p, p, p, p, p]
        L.oracle_verify_greedy_active.restype = u32
        L.oracle_verify_margin.argtypes = [p, C.c_int, i64, i32, i32, i32, p, p, p, p, i32, i32,
                                           p, i32, p, p, p, p, p]
        L.oracle_verify_margin.restype = u32
        L.oracle_draft_confidence.argtypes = [p, C.c_int, i64, i32, i32, i32, p, f64, i32,
                                              p, p, p, p, p, p, p, p]
        L.oracle_draft_confidence.restype = u32
        L.oracle_prefix_stats.argtypes = [p, p, i32, i32, p, p, p]
        L.oracle_prefix_stats.restype = u32
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits(x: np.ndarray, dtype: str):
    if dtype == "bf16":
        return _c(x, np.uint16), 1
    if dtype == "f32":
        return _c(x, np.float32), 0
    raise ValueError(dtype)


def threads(n: int = 0) -> int:
    """Set (n > 0) and return the number of OpenMP threads the oracle uses."""
    return int(lib().oracle_threads(int(n)))


# ----------------------------------------------------------------------------
# Philox4x32-10 and uniforms (Salmon et al., SC'11)
# ----------------------------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(x: int) -> float:
    return float(lib().oracle_uniform(int(x) & 0xFFFFFFFF))


def token_uniform(seed: int, rid: int, pos: int, step: int, i: int) -> float:
    return float(lib().oracle_token_uniform(int(seed) & (2**64 - 1), rid, pos, step, i))


# ----------------------------------------------------------------------------
# A1 fused row reduction
# ----------------------------------------------------------------------------

def row_reduce(logits: np.ndarray, dtype: str, V: Optional[int] = None, R: Optional[int] = None):
    """Per row: max, log-sum-exp, first argmax (xLLM "自适应投机推理",
    §"基于 MTP logits 的自适应 target 验证": logsumexp; vSpec README
    §"EAGLE 功能": greedy top-1)."""
    x, dt = _logits(logits, dtype)
    V = x.shape[1] if V is None else V
    R = x.shape[0] if R is None else R
    mx = np.zeros(max(R, 1)); lse = np.zeros(max(R, 1)); am = np.zeros(max(R, 1), np.int32)
    lib().oracle_row_reduce(_ptr(x), dt, x.shape[1], V, R, _ptr(mx), _ptr(lse), _ptr(am))
    return mx[:R], lse[:R], am[:R]


@dataclass
class VerifyResult:
    accepted_len: np.ndarray
    out_tokens: np.ndarray
    next_token: np.ndarray
    status: int
    rows: dict


def _outs(B, k_max):
    return (np.zeros(max(B, 1), np.int32), np.zeros((max(B, 1), k_max + 1), np.int32),
            np.zeros(max(B, 1), np.int32))


# ----------------------------------------------------------------------------
# A2 greedy verification
# ----------------------------------------------------------------------------

def verify_greedy(logits, dtype, V, B, k_max, cu_rows, draft_ids) -> VerifyResult:
    """Longest draft prefix equal to the target's first argmax, then the
    target token (vSpec README §"EAGLE 功能": strict greedy top-1)."""
    x, dt = _logits(logits, dtype)
    cu = _c(cu_rows, np.int32); d = _c(draft_ids, np.int32)
    R = max(int(cu[B]), 1)
    acc, out, nxt = _outs(B, k_max)
    mx = np.zeros(R); lse = np.zeros(R); am = np.zeros(R, np.int32)
    st = lib().oracle_verify_greedy(_ptr(x), dt, x.shape[1], V, B, k_max, _ptr(cu), _ptr(d),
                                    _ptr(acc), _ptr(out), _ptr(nxt), _ptr(mx), _ptr(lse), _ptr(am))
    Rr = max(int(cu[B]), 0)
    return VerifyResult(acc[:B], out[:B], nxt[:B], int(st),
                        dict(row_max=mx[:Rr], row_lse=lse[:Rr], row_argmax=am[:Rr]))


# ----------------------------------------------------------------------------
# A3 filters / sampler and A4 chain
# ----------------------------------------------------------------------------

def filter_row(z: np.ndarray, T: float, top_k: int, top_p: float, min_p: float):
    """Survivor mask of the temperature/top-k/min-p/top-p filters for T > 0
    (xLLM "自适应投机推理" §"启动示例": ordinary sampler semantics).
    Returns (mask, margin)."""
    zz = _c(z, np.float64)
    keep = np.zeros(max(zz.size, 1), np.uint8)
    mg = np.zeros(1)
    lib().oracle_filter_row(_ptr(zz), zz.size, float(T), int(top_k), float(top_p), float(min_p),
                            _ptr(keep), _ptr(mg))
    return keep[:zz.size].astype(bool), float(mg[0])


def sample_row(z: np.ndarray, T: float, top_k: int, top_p: float, min_p: float,
               seed: int, rid: int, pos: int, step: int):
    """Sampled token of one row (Gumbel-max over survivors).
    Returns (token, mask, margin_filter, margin_gumbel)."""
    zz = _c(z, np.float64)
    keep = np.zeros(max(zz.size, 1), np.uint8)
    mf = np.zeros(1); mg = np.zeros(1)
    y = lib().oracle_sample_row(_ptr(zz), zz.size, float(T), int(top_k), float(top_p),
                                float(min_p), int(seed) & (2**64 - 1), rid, pos, step,
                                _ptr(keep), _ptr(mf), _ptr(mg))
    return int(y), keep[:zz.size].astype(bool), float(mf[0]), float(mg[0])


def verify_sample(logits, dtype, V, B, k_max, cu_rows, draft_ids, params) -> VerifyResult:
    """Stochastic verification with a point-mass draft (xLLM
    "自适应投机推理" §"启动示例"): sample every packed row with its owner's
    parameters; accept while sample == draft; the first mismatching sample is
    the replacement, else the last row's sample is the bonus."""
    x, dt = _logits(logits, dtype)
    cu = _c(cu_rows, np.int32); d = _c(draft_ids, np.int32)
    R = max(int(cu[B]), 1)
    acc, out, nxt = _outs(B, k_max)
    tok = np.zeros(R, np.int32); mf = np.zeros(R); mg = np.zeros(R)
    t = _c(params.temperature, np.float32); tk = _c(params.top_k, np.int32)
    tp = _c(params.top_p, np.float32); mp = _c(params.min_p, np.float32)
    sd = _c(params.seed, np.uint64)
    rid = None if params.request_id is None else _c(params.request_id, np.uint32)
    st = lib().oracle_verify_sample(_ptr(x), dt, x.shape[1], V, B, k_max, _ptr(cu), _ptr(d),
                                    _ptr(t), _ptr(tk), _ptr(tp), _ptr(mp), _ptr(sd), _ptr(rid),
                                    int(params.step), _ptr(acc), _ptr(out), _ptr(nxt),
                                    _ptr(tok), _ptr(mf), _ptr(mg))
    Rr = max(int(cu[B]), 0)
    return VerifyResult(acc[:B], out[:B], nxt[:B], int(st),
                        dict(row_token=tok[:Rr], margin_filter=mf[:Rr], margin_gumbel=mg[:Rr]))


# ----------------------------------------------------------------------------
# A5 relaxed top-K
# ----------------------------------------------------------------------------

def verify_relaxed(logits, dtype, V, B, k_max, cu_rows, draft_ids, relaxed_k) -> VerifyResult:
    """Relaxed top-K acceptance with strict prefix (vSpec README §"支持范围",
    §"EAGLE 功能"): accept d iff #{i : z_i > z_d} < K; stop at the first
    failure; emit the target's first argmax of the stopping row."""
    x, dt = _logits(logits, dtype)
    cu = _c(cu_rows, np.int32); d = _c(draft_ids, np.int32); K = _c(relaxed_k, np.int32)
    R = max(int(cu[B]), 1)
    acc, out, nxt = _outs(B, k_max)
    am = np.zeros(R, np.int32); rk = np.zeros(R, np.int32)
    st = lib().oracle_verify_relaxed(_ptr(x), dt, x.shape[1], V, B, k_max, _ptr(cu), _ptr(d),
                                     _ptr(K), _ptr(acc), _ptr(out), _ptr(nxt), _ptr(am), _ptr(rk))
    Rr = max(int(cu[B]), 0)
    return VerifyResult(acc[:B], out[:B], nxt[:B], int(st),
                        dict(row_argmax=am[:Rr], row_rank=rk[:Rr]))


# ----------------------------------------------------------------------------
# Compact rows back to request slots
# ----------------------------------------------------------------------------

def restore_rows(compact: np.ndarray, cu_rows, B: int, k_max: int, out: np.ndarray):
    """Restore of compact per-row outputs to request slots by device offsets
    (xLLM "自适应投机推理" §"基于 MTP logits 的自适应 target 验证": compact
    target outputs, e.g. hidden states, are restored by the device offsets
    before the draft context is updated).  Row cu_rows[b] + j of `compact`
    goes to slot b * (k_max + 1) + j of `out` for j = 0 .. k_b; other slots
    are left as they are.  A request whose offsets are malformed (cu_rows[0]
    != 0, a negative start, k_b outside [0, k_max], or rows beyond the
    compact buffer) is skipped and reported.  Returns (out copy, status)."""
    cu = _c(cu_rows, np.int64)
    res = out.copy()
    status = 0
    R_cap = compact.shape[0]
    for b in range(B):
        lo, hi = int(cu[b]), int(cu[b + 1])
        n = hi - lo
        if cu[0] != 0 or lo < 0 or n < 1 or n - 1 > k_max or hi > R_cap:
            status |= BAD_ROWS
            continue
        for j in range(n):
            res[b * (k_max + 1) + j] = compact[lo + j]
    return res, status


# ----------------------------------------------------------------------------
# Greedy verification over an active vocabulary
# ----------------------------------------------------------------------------

def verify_greedy_active(logits, dtype, V, B, k_max, cu_rows, draft_ids,
                         vocab_ids) -> VerifyResult:
    """Greedy verification when the target scores only V active columns,
    column i standing for full token id vocab_ids[i] (vSpec README
    §"EAGLE 功能", §"代码所有权": active-vocabulary LM head with a full
    token-id map).  Row token = vocab_ids[first argmax column]; drafts are
    full ids, accepted while equal to it."""
    x, dt = _logits(logits, dtype)
    cu = _c(cu_rows, np.int32); d = _c(draft_ids, np.int32); m = _c(vocab_ids, np.int32)
    if m.size < V:
        raise ValueError("vocab_ids needs one full id per active column")
    R = max(int(cu[B]), 1)
    acc, out, nxt = _outs(B, k_max)
    col = np.zeros(R, np.int32); tok = np.zeros(R, np.int32)
    st = lib().oracle_verify_greedy_active(_ptr(x), dt, x.shape[1], V, B, k_max, _ptr(cu),
                                           _ptr(d), _ptr(m), _ptr(acc), _ptr(out), _ptr(nxt),
                                           _ptr(col), _ptr(tok))
    Rr = max(int(cu[B]), 0)
    return VerifyResult(acc[:B], out[:B], nxt[:B], int(st),
                        dict(row_argmax=col[:Rr], row_token=tok[:Rr]))


# ----------------------------------------------------------------------------
# Confidence-margin acceptance
# ----------------------------------------------------------------------------

def verify_margin(logits, dtype, V, B, k_max, cu_rows, draft_ids, margin, generated=None,
                  from_position: int = 0, after_tokens: int = 0,
                  protected_ids=None) -> VerifyResult:
    """Greedy acceptance loosened by a logit margin (vSpec README §"启动"
    approximate-acceptance preset, §"通用参数": --confidence-accept-margin,
    --confidence-accept-from-position / --confidence-accept-after-tokens,
    --confidence-protected-token-ids).  Draft d at position j of request b
    passes when it is the first argmax, or when j >= from_position,
    generated[b] + j >= after_tokens, d is not protected and the fp32 gap
    max - z[d] <= margin[b].  Strict prefix; the emitted token is the
    stopping row's first argmax."""
    x, dt = _logits(logits, dtype)
    cu = _c(cu_rows, np.int32); d = _c(draft_ids, np.int32)
    mg = _c(margin, np.float32)
    gen = None if generated is None else _c(generated, np.int32)
    prot = np.zeros(1, np.int32) if protected_ids is None else _c(protected_ids, np.int32)
    n_prot = 0 if protected_ids is None else int(prot.size)
    R = max(int(cu[B]), 1)
    acc, out, nxt = _outs(B, k_max)
    am = np.zeros(R, np.int32); ok = np.zeros(R, np.int32)
    st = lib().oracle_verify_margin(_ptr(x), dt, x.shape[1], V, B, k_max, _ptr(cu), _ptr(d),
                                    _ptr(mg), _ptr(gen), int(from_position), int(after_tokens),
                                    _ptr(prot), n_prot, _ptr(acc), _ptr(out), _ptr(nxt),
                                    _ptr(am), _ptr(ok))
    Rr = max(int(cu[B]), 0)
    return VerifyResult(acc[:B], out[:B], nxt[:B], int(st),
                        dict(row_argmax=am[:Rr], row_ok=ok[:Rr]))


# ----------------------------------------------------------------------------
# A6 + A7 confidence and prefix allocation
# ----------------------------------------------------------------------------

@dataclass
class Allocation:
    conf: np.ndarray
    k_alloc: np.ndarray
    cu_rows: np.ndarray
    row_owner: np.ndarray
    row_pos: np.ndarray
    packed_draft: np.ndarray
    total_rows: int
    margin: float
    status: int


def draft_confidence(draft_logits, dtype, V, B, k, selected=None, threshold=0.3,
                     max_rows=0) -> Allocation:
    """conf = exp(selected_logit - logsumexp(draft_logits)) per draft
    position, then device-side prefix allocation and packing (xLLM
    "自适应投机推理" §"基于 MTP logits 的自适应 target 验证")."""
    x, dt = _logits(draft_logits, dtype)
    sel = None if selected is None else _c(selected, np.int32)
    Q = max(B * k, 1); cap = max(B * (k + 1), 1)
    conf = np.zeros(Q); ka = np.zeros(max(B, 1), np.int32); cu = np.zeros(B + 1, np.int32)
    own = np.zeros(cap, np.int32); pos = np.zeros(cap, np.int32); pk = np.zeros(cap, np.int32)
    tot = np.zeros(1, np.int32); mg = np.zeros(1)
    st = lib().oracle_draft_confidence(_ptr(x), dt, x.shape[1], V, B, k, _ptr(sel),
                                       float(threshold), int(max_rows), _ptr(conf), _ptr(ka),
                                       _ptr(cu), _ptr(own), _ptr(pos), _ptr(pk), _ptr(tot),
                                       _ptr(mg))
    n = B * (k + 1)
    return Allocation(conf[:B * k], ka[:B], cu, own[:n], pos[:n], pk[:n], int(tot[0]),
                      float(mg[0]), int(st))


# ----------------------------------------------------------------------------
# A8 prefix-acceptance counters
# ----------------------------------------------------------------------------

def prefix_stats(accepted_len, cu_rows, B, k_max, acc=None, ver=None, hist=None):
    """acc[j] += #{a_b > j}, ver[j] += #{k_b > j}, hist[a_b] += 1 (xLLM
    "自适应投机推理" §"自适应 draft 步长（MTP）": per-position prefix
    acceptance feeding B*(1+sum(prefix_acceptance[:k]))/cost_ms)."""
    acc = np.zeros(max(k_max, 1), np.int64) if acc is None else acc
    ver = np.zeros(max(k_max, 1), np.int64) if ver is None else ver
    hist = np.zeros(k_max + 1, np.int64) if hist is None else hist
    a = _c(accepted_len, np.int32); cu = _c(cu_rows, np.int32)
    st = lib().oracle_prefix_stats(_ptr(a), _ptr(cu), B, k_max, _ptr(acc), _ptr(ver), _ptr(hist))
    return acc, ver, hist, int(st)
