"""Seeded synthetic inputs for ragged draft-token verification.

This module builds the inputs that both the CPU oracle and the CUDA path are
fed: packed target-logit rows, draft tokens, ragged row offsets and
per-request sampling parameters.  It performs no step of the verification
method itself; the only computations here construct inputs (planting a peak,
choosing which draft tokens copy a row's top token).

Shapes follow the workloads the source pages describe (Qwen-class vocabulary,
batch 16-256, 4-7 draft tokens):

* xLLM docs "自适应投机推理", §"基于 MTP logits 的自适应 target 验证" and
  §"启动示例": ragged packed verify rows, one owner request per row, mixed
  temperature batches, top-k / top-p / min-p per request.
* vllm-hust-vSpec README, §"支持范围" / §"EAGLE 功能": Qwen2.5-14B target
  (vocabulary 152064), B128, gamma 4, relaxed top-K acceptance.

The page workloads run real models on datasets that are not available here;
these synthetic logits stand in for them: seeded N(0, sigma) rows of the
pages' shapes, with the planted peaks, draft rules and parameter mixes each
generator below states.

Logits are produced in fp32 and, for bf16 rows, rounded to bf16 with
round-to-nearest-even; the bf16 *bit patterns* (uint16) are what both sides
read, so the oracle and the kernels see exactly the same values.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "VerifyBatch", "SampleParams", "DraftBatch",
    "bf16_bits", "bf16_bits_to_f32", "data_seed",
    "tiny_greedy", "planted_greedy", "stochastic", "mtp_adaptive",
    "relaxed_planted", "ragged_batch", "random_sample_params",
]

QWEN_VOCAB = 152064      # Qwen2.5 vocabulary (target of the vSpec presets)
GLM_MTP_VOCAB = 151552   # vocabulary of the MTP/DSpark-shaped workload


def data_seed(cfg: int, step: int = 0) -> int:
    """Data seed convention: 1000 * workload-number + step."""
    return 1000 * cfg + step


# ----------------------------------------------------------------------------
# bf16 encoding (input encoding only)
# ----------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs are finite (the generators never produce NaN), so no NaN quieting.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# containers
# ----------------------------------------------------------------------------

@dataclass
class VerifyBatch:
    """A ragged batch of packed verify rows.

    logits     [R_alloc, ld]  float32, or uint16 bf16 bit patterns
    dtype      "f32" | "bf16"
    V          vocabulary size (<= ld)
    B, k_max   requests, maximum draft tokens per request
    cu_rows    [B+1] int32, request b owns rows cu_rows[b] .. cu_rows[b+1]-1
               (k_b + 1 rows: k_b draft positions then the bonus row)
    draft_ids  [R_alloc] int32, draft token checked by row r, -1 on bonus rows
    """
    logits: np.ndarray
    dtype: str
    V: int
    B: int
    k_max: int
    cu_rows: np.ndarray
    draft_ids: np.ndarray
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return int(self.cu_rows[-1])

    @property
    def ld(self) -> int:
        return int(self.logits.shape[1])

    def values_f32(self) -> np.ndarray:
        """Logits as fp32 values (exact for bf16)."""
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self.logits)
        return self.logits


@dataclass
class SampleParams:
    """Per-request sampling parameters of the stochastic verifier."""
    temperature: np.ndarray   # [B] float32, 0 = greedy
    top_k: np.ndarray         # [B] int32, 0 = off
    top_p: np.ndarray         # [B] float32, 1 = off
    min_p: np.ndarray         # [B] float32, 0 = off
    seed: np.ndarray          # [B] uint64
    request_id: np.ndarray    # [B] uint32
    step: int = 0


@dataclass
class DraftBatch:
    """Draft-model logits for the adaptive-verify workload.

    draft_logits [B*k, ld] (row b*k + j = draft position j of request b)
    target_logits [B*(k+1), ld]: room for every packed verify row; after
    prefix allocation the first R rows are the packed target rows.
    """
    draft_logits: np.ndarray
    target_logits: np.ndarray
    dtype: str
    V: int
    B: int
    k: int


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _normal_rows(rng: np.random.Generator, rows: int, V: int, sigma: float,
                 ld: Optional[int] = None) -> np.ndarray:
    ld = V if ld is None else ld
    z = np.zeros((rows, ld), dtype=np.float32)
    z[:, :V] = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma)
    return z


def _plant_peaks(rng: np.random.Generator, z: np.ndarray, V: int, gap: float) -> np.ndarray:
    """Set one seeded token per row to (largest other value) + gap, in fp32.

    Returns the planted token of every row.  Done before the bf16 cast; with
    gap >= 1 the planted token stays the unique largest value after rounding.
    """
    rows = z.shape[0]
    tok = rng.integers(0, V, size=rows).astype(np.int32)
    idx = np.arange(rows)
    z[idx, tok] = -np.inf
    top = z[:, :V].max(axis=1)
    z[idx, tok] = top + np.float32(gap)
    return tok


def _encode(z: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits(z)
    if dtype == "f32":
        return np.ascontiguousarray(z, dtype=np.float32)
    raise ValueError(dtype)


def _first_top(values: np.ndarray, V: int) -> np.ndarray:
    """Index of the first largest value of each row (input construction:
    picks the token a greedy draft that agrees with the target would propose)."""
    return np.argmax(values[:, :V], axis=1).astype(np.int32)


def _uniform_cu_rows(B: int, k: int) -> np.ndarray:
    return (np.arange(B + 1, dtype=np.int64) * (k + 1)).astype(np.int32)


def _drafts_from(cu_rows: np.ndarray, proposal: np.ndarray) -> np.ndarray:
    """draft_ids[r] = proposal[r] on draft rows, -1 on each request's last row."""
    d = proposal.astype(np.int32).copy()
    d[cu_rows[1:] - 1] = -1
    return d


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

def tiny_greedy(seed: int = data_seed(1), B: int = 4, k: int = 4, V: int = 1024,
                sigma: float = 2.0, p_match: float = 0.7) -> VerifyBatch:
    """Tiny greedy verify: fp32 logits ~ N(0, sigma); the draft token at each
    position is the row's top token with probability p_match, else a uniform
    random token."""
    rng = np.random.default_rng(seed)
    R = B * (k + 1)
    z = _normal_rows(rng, R, V, sigma)
    cu = _uniform_cu_rows(B, k)
    top = _first_top(z, V)
    rand = rng.integers(0, V, size=R).astype(np.int32)
    use_top = rng.random(R) < p_match
    return VerifyBatch(_encode(z, "f32"), "f32", V, B, k, cu,
                       _drafts_from(cu, np.where(use_top, top, rand)))


def planted_greedy(seed: int = data_seed(2), B: int = 128, k: int = 4, V: int = QWEN_VOCAB,
                   sigma: float = 3.0, gap: float = 8.0,
                   p_pos=(0.8, 0.65, 0.5, 0.4), dtype: str = "bf16") -> VerifyBatch:
    """Greedy verify with a planted peak per row.

    Logits ~ N(0, sigma) in fp32; one seeded token per row is set to the row's
    largest other value + gap, then the row is rounded to bf16.  The draft at
    position j equals the planted token with probability p_pos[j] (the last
    entry repeats for longer drafts), else a uniform token different from it.
    """
    rng = np.random.default_rng(seed)
    R = B * (k + 1)
    z = _normal_rows(rng, R, V, sigma)
    planted = _plant_peaks(rng, z, V, gap)
    cu = _uniform_cu_rows(B, k)
    pos = np.tile(np.arange(k + 1), B)
    probs = np.array([p_pos[min(j, len(p_pos) - 1)] for j in range(k + 1)])[pos]
    other = (planted + rng.integers(1, V, size=R)) % V
    prop = np.where(rng.random(R) < probs, planted, other).astype(np.int32)
    vb = VerifyBatch(_encode(z, dtype), dtype, V, B, k, cu, _drafts_from(cu, prop))
    vb.extra["planted"] = planted
    return vb


def random_sample_params(rng: np.random.Generator, B: int,
                         temperatures=(0.0, 0.5, 1.0), top_ks=(0, 20, 50),
                         top_ps=(1.0, 0.9), min_ps=(0.0, 0.05), step: int = 0) -> SampleParams:
    """Per-request parameters drawn independently and uniformly from the given
    value sets; one 64-bit sampling seed per request."""
    t = rng.choice(np.asarray(temperatures, dtype=np.float32), size=B).astype(np.float32)
    tk = rng.choice(np.asarray(top_ks, dtype=np.int32), size=B).astype(np.int32)
    tp = rng.choice(np.asarray(top_ps, dtype=np.float32), size=B).astype(np.float32)
    mp = rng.choice(np.asarray(min_ps, dtype=np.float32), size=B).astype(np.float32)
    seed = rng.integers(0, 2**63, size=B, dtype=np.int64).astype(np.uint64) \
        ^ (rng.integers(0, 2, size=B, dtype=np.int64).astype(np.uint64) << np.uint64(63))
    rid = np.arange(B, dtype=np.uint32)
    return SampleParams(t, tk, tp, mp, seed, rid, step)


def stochastic(seed: int = data_seed(3), B: int = 128, k: int = 4, V: int = QWEN_VOCAB,
               sigma: float = 3.0, p_top: float = 0.8, dtype: str = "bf16",
               **param_sets):
    """Stochastic (mixed-temperature) verify.

    Logits ~ N(0, sigma), no planting.  Point-mass (deterministic) draft: the
    draft at each position is the row's first top token with probability
    p_top, else a uniform random token.  Per-request temperature, top-k,
    top-p, min-p are drawn uniformly from {0,0.5,1}, {0,20,50}, {1,0.9},
    {0,0.05}; each request gets its own 64-bit seed.
    Returns (VerifyBatch, SampleParams).
    """
    rng = np.random.default_rng(seed)
    R = B * (k + 1)
    z = _normal_rows(rng, R, V, sigma)
    enc = _encode(z, dtype)
    vals = bf16_bits_to_f32(enc) if dtype == "bf16" else enc
    top = _first_top(vals, V)
    rand = rng.integers(0, V, size=R).astype(np.int32)
    prop = np.where(rng.random(R) < p_top, top, rand)
    cu = _uniform_cu_rows(B, k)
    params = random_sample_params(rng, B, **param_sets)
    return VerifyBatch(enc, dtype, V, B, k, cu, _drafts_from(cu, prop)), params


def mtp_adaptive(seed: int = data_seed(4), B: int = 16, k: int = 7, V: int = GLM_MTP_VOCAB,
                 sigma: float = 3.0, planted_draft: bool = False,
                 dtype: str = "bf16") -> DraftBatch:
    """MTP/DSpark-shaped adaptive verify: draft logits [B*k, V] and target
    logits [B*(k+1), V], both ~ N(0, sigma).  With planted_draft, each draft
    row gets a peak at (largest other value) + delta, delta ~ U(0, 8), so the
    draft confidences spread over (0, 1)."""
    rng = np.random.default_rng(seed)
    d = _normal_rows(rng, B * k, V, sigma)
    if planted_draft:
        rows = B * k
        tok = rng.integers(0, V, size=rows)
        idx = np.arange(rows)
        d[idx, tok] = -np.inf
        top = d[:, :V].max(axis=1)
        d[idx, tok] = top + rng.uniform(0.0, 8.0, size=rows).astype(np.float32)
    t = _normal_rows(rng, B * (k + 1), V, sigma)
    return DraftBatch(_encode(d, dtype), _encode(t, dtype), dtype, V, B, k)


def relaxed_planted(seed: int = data_seed(5), B: int = 256, k: int = 5, V: int = QWEN_VOCAB,
                    sigma: float = 3.0, gap: float = 8.0, p_planted: float = 0.7,
                    p_near: float = 0.5, relaxed_k: int = 4, dtype: str = "bf16") -> VerifyBatch:
    """EAGLE-relaxed workload: N(0, sigma) logits with a planted peak per row.
    Draft at each position: the planted token with probability p_planted;
    otherwise, with probability p_near, a uniform pick among the row's 2nd..4th
    largest tokens; otherwise a uniform token.  extra["relaxed_k"] holds the
    per-request K (relaxed top-K acceptance)."""
    rng = np.random.default_rng(seed)
    R = B * (k + 1)
    z = _normal_rows(rng, R, V, sigma)
    planted = _plant_peaks(rng, z, V, gap)
    enc = _encode(z, dtype)
    vals = bf16_bits_to_f32(enc) if dtype == "bf16" else enc
    # 2nd..4th largest tokens of each row (input construction only)
    part = np.argpartition(-vals[:, :V], 4, axis=1)[:, :4]
    order = np.argsort(-np.take_along_axis(vals[:, :V], part, axis=1), axis=1, kind="stable")
    ranked = np.take_along_axis(part, order, axis=1)          # [R, 4], rank 1..4
    near = ranked[np.arange(R), rng.integers(1, 4, size=R)]
    rand = rng.integers(0, V, size=R)
    u = rng.random(R)
    prop = np.where(u < p_planted, planted,
                    np.where(rng.random(R) < p_near, near, rand)).astype(np.int32)
    cu = _uniform_cu_rows(B, k)
    vb = VerifyBatch(enc, dtype, V, B, k, cu, _drafts_from(cu, prop))
    vb.extra["relaxed_k"] = np.full(B, relaxed_k, dtype=np.int32)
    vb.extra["planted"] = planted
    return vb


def relaxed_steps(n_steps: int = 20, seed: int = data_seed(5), B: int = 256, k: int = 5,
                  V: int = QWEN_VOCAB, sigma: float = 3.0, gap: float = 8.0,
                  p_planted: float = 0.7, p_near: float = 0.5, relaxed_k: int = 4):
    """Seeded steps of the EAGLE-relaxed workload (bf16), one VerifyBatch per
    step.  The N(0, sigma) rows are drawn once (seed); step s (its own
    generator, seeded by (seed, s)) permutes them, plants a peak per row at
    (largest other value) + gap and draws the drafts as relaxed_planted
    does, from the row's planted token, its 2nd..4th largest tokens or a
    uniform token.  Each step costs a copy instead of a fresh draw of
    R x V normals."""
    R = B * (k + 1)
    base = _normal_rows(np.random.default_rng(seed), R, V, sigma)
    # per base row: largest and second largest fp32 value (the planted value
    # is the largest *other* value + gap) and the five largest bf16 values'
    # tokens, by value then index (the near drafts after planting)
    part = np.argpartition(-base[:, :V], 1, axis=1)[:, :2]
    pv = np.take_along_axis(base, part, axis=1)
    first = np.where(pv[:, 0] >= pv[:, 1], 0, 1)
    top_tok = part[np.arange(R), first]
    top1 = pv[np.arange(R), first]
    top2 = pv[np.arange(R), 1 - first]
    enc = _encode(base, "bf16")
    vals = bf16_bits_to_f32(enc)
    p5 = np.argpartition(-vals[:, :V], 5, axis=1)[:, :5]
    key = np.take_along_axis(vals, p5, axis=1)
    o5 = np.lexsort((p5, -key), axis=1)
    top5 = np.take_along_axis(p5, o5, axis=1)
    del vals
    cu = _uniform_cu_rows(B, k)
    rows = np.arange(R)
    for s in range(n_steps):
        rng = np.random.default_rng([seed, s])
        perm = rng.permutation(R)
        e = enc[perm]
        tok = rng.integers(0, V, size=R).astype(np.int32)
        other = np.where(tok == top_tok[perm], top2[perm], top1[perm])
        e[rows, tok] = bf16_bits((other + np.float32(gap)).astype(np.float32)[:, None])[:, 0]
        # ranks 2..4 after planting: the base row's largest tokens other than tok
        cand = top5[perm]
        keep = cand != tok[:, None]
        ranked = np.array([c[m][:3] for c, m in zip(cand, keep)])
        near = ranked[rows, rng.integers(0, 3, size=R)]
        rand = rng.integers(0, V, size=R)
        u = rng.random(R)
        prop = np.where(u < p_planted, tok,
                        np.where(rng.random(R) < p_near, near, rand)).astype(np.int32)
        vb = VerifyBatch(e, "bf16", V, B, k, cu, _drafts_from(cu, prop))
        vb.extra["relaxed_k"] = np.full(B, relaxed_k, dtype=np.int32)
        vb.extra["planted"] = tok
        yield vb


def ragged_batch(seed: int, B: int, k_max: int, V: int, dtype: str = "bf16",
                 sigma: float = 3.0, p_top: float = 0.6, ld: Optional[int] = None,
                 k_values: Optional[np.ndarray] = None, plant_gap: Optional[float] = None,
                 tie_top: bool = False) -> VerifyBatch:
    """Ragged packed batch: request b has k_b in [0, k_max] draft tokens
    (uniform, or given), rows laid out back to back with leading dimension ld.
    With tie_top, each row's largest value is copied to a second, later
    position so that exact top ties occur on every row."""
    rng = np.random.default_rng(seed)
    kb = (rng.integers(0, k_max + 1, size=B) if k_values is None
          else np.asarray(k_values)).astype(np.int32)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(kb + 1)
    R = int(cu[-1])
    z = _normal_rows(rng, max(R, 1), V, sigma, ld)
    if plant_gap is not None:
        _plant_peaks(rng, z, V, plant_gap)
    if tie_top and V > 1:
        for r in range(R):
            i = int(np.argmax(z[r, :V]))
            j = int(rng.integers(0, V))
            if j != i:
                z[r, j] = z[r, i]
    enc = _encode(z, dtype)
    vals = bf16_bits_to_f32(enc) if dtype == "bf16" else enc
    top = _first_top(vals, V)
    rand = rng.integers(0, V, size=max(R, 1)).astype(np.int32)
    prop = np.where(rng.random(max(R, 1)) < p_top, top, rand)
    d = prop.astype(np.int32)
    if R:
        d[cu[1:] - 1] = -1
    return VerifyBatch(enc, dtype, V, B, k_max, cu, d)


def near_top_drafts(vb: VerifyBatch, seed: int, p_top: float = 0.4,
                    max_rank: int = 10) -> VerifyBatch:
    """The same rows with each draft replaced by the token at a random rank
    among its row's largest values: rank 0 (the first top value) with
    probability p_top, else a rank uniform in [1, max_rank] (value order,
    lower index first on equal values).  Drafts then sit at small, varied
    distances below the row maximum, the range a confidence margin decides."""
    rng = np.random.default_rng(seed)
    vals = bf16_bits_to_f32(vb.logits) if vb.dtype == "bf16" else vb.logits
    d = vb.draft_ids.copy()
    for b in range(vb.B):
        for r in range(int(vb.cu_rows[b]), int(vb.cu_rows[b + 1]) - 1):
            q = 0 if rng.random() < p_top else int(rng.integers(1, max_rank + 1))
            q = min(q, vb.V - 1)
            v = vals[r, :vb.V]
            cut = np.partition(v, vb.V - 1 - q)[vb.V - 1 - q]      # the (q+1)-th largest
            idx = np.nonzero(v >= cut)[0]
            d[r] = idx[np.argsort(-v[idx], kind="stable")][q]
    return VerifyBatch(vb.logits, vb.dtype, vb.V, vb.B, vb.k_max, vb.cu_rows, d)
