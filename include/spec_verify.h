/*
 * spec_verify.h -- C ABI of libspecverify: batched draft-token verification
 * over vocabulary-wide target logits, for GB300 (sm_103a).
 *
 * What it computes (web pages this library implements; section names as
 * printed on the pages):
 *   - xLLM docs "自适应投机推理" (adaptive speculative inference),
 *       §"启动示例": the ragged rejection sampler -- every packed verify row
 *       is sampled with its owner request's parameters (found through the
 *       packed-row owners); with a deterministic (point-mass) draft this is
 *       rejection sampling: accept while the sample equals the draft, the
 *       first mismatching sample is the replacement token, and when every
 *       draft matches the last row's sample is the bonus token; temperature 0
 *       is greedy, and top-k / top-p / min-p follow the ordinary sampler.
 *       §"基于 MTP logits 的自适应 target 验证": the draft confidence
 *       exp(selected_logit - logsumexp(draft_logits)), kept on the device for
 *       prefix allocation and packing with device offsets, and the restore
 *       of the compact target rows' outputs by those offsets.
 *       §"自适应 draft 步长（MTP）": per-position prefix acceptance feeding the
 *       controller objective B * (1 + sum(prefix_acceptance[:k])) / cost_ms.
 *   - "vllm-hust-vSpec" README, §"EAGLE 功能" and §"支持范围": strict greedy
 *       top-1 acceptance, and relaxed top-K acceptance with a strict prefix;
 *       acceptance without a per-request device-to-host sync; the active
 *       vocabulary with a full token-id map (also §"代码所有权").
 *       §"启动" and §"通用参数": greedy acceptance loosened by a confidence
 *       margin, from a position or after a token count, never for protected
 *       token ids.
 *   The host-side adaptive step controller that consumes the counters is
 *   declared in spec_step.h.
 *
 * Conventions (all entry points):
 *   - Every pointer argument is DEVICE memory owned by the caller unless the
 *     comment says "host".  The library never allocates memory.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *     and performs no host synchronisation and no device-to-host copy.
 *   - The return value is a spec_result code.  Host-checkable argument
 *     errors return SPEC_ERR_INVALID_ARG / SPEC_ERR_UNSUPPORTED with NOTHING
 *     launched and no output touched.  SPEC_ERR_CUDA reports a launch error
 *     (text from spec_last_cuda_error()).
 *   - Problems only visible in device data (bad per-request parameters,
 *     malformed row offsets, out-of-range selected tokens, a wait that gave
 *     up) never trap: they OR bits (SPEC_STATUS_*) into the optional device
 *     word `status` and the affected request or row takes the documented
 *     fallback.
 *   - Logits are row-major with leading dimension `ld >= V` elements, dtype
 *     SPEC_F32 or SPEC_BF16 (bf16 stored as raw 16-bit patterns), base
 *     pointer aligned to the element size.  Values must be finite or -inf;
 *     NaN and +inf are outside the contract (results unspecified).
 *   - Ragged packing: request b owns the k_b + 1 consecutive rows
 *     cu_rows[b] .. cu_rows[b+1]-1: draft positions j = 0..k_b-1, then the
 *     bonus row j = k_b.  cu_rows must be non-decreasing with cu_rows[0] = 0
 *     and 0 <= k_b <= k_max; a request that breaks this gets
 *     SPEC_STATUS_BAD_ROWS, accepted_len = 0, next_token = -1 and an all -1
 *     out_tokens row.  draft_ids[r] is the draft token checked by row r
 *     (ignored on bonus rows); ids outside [0, V) are mismatches, not errors.
 *   - Argmax ties resolve to the lowest index; -0.0 equals +0.0.
 *   - Calls that share a workspace must be ordered on one stream.
 *   - Launch order: each call's kernels follow one another by programmatic
 *     dependent launch.  spec_verify_sample's first kernel is itself a
 *     programmatic dependent of whatever kernel precedes it on the stream:
 *     its blocks may become resident early, but they read nothing and
 *     release nothing before that kernel has completed, so inputs written by
 *     it are seen.  A call's last kernel lets the next kernel on the stream
 *     launch early in the same way; a kernel that reads this call's outputs
 *     must wait (griddepcontrol.wait) if it is itself launched as a
 *     programmatic dependent.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *spec_stream;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, ld < V ...    */
    SPEC_ERR_UNSUPPORTED = 2,   /* dtype, k_max > 31, row longer than 2 MiB          */
    SPEC_ERR_CUDA = 3,          /* launch failed; see spec_last_cuda_error()       */
    SPEC_ERR_WORKSPACE = 4      /* workspace null or smaller than required         */
} spec_result;

/* device status bits (OR-ed into *status when status != NULL) */
#define SPEC_STATUS_BAD_TEMPERATURE 0x1u   /* T < 0, NaN or inf: request sampled greedily      */
#define SPEC_STATUS_BAD_TOP_K       0x2u   /* top_k < 0: top-k off                             */
#define SPEC_STATUS_BAD_TOP_P       0x4u   /* top_p outside (0, 1]: top-p off                  */
#define SPEC_STATUS_BAD_MIN_P       0x8u   /* min_p outside [0, 1]: min-p off                  */
#define SPEC_STATUS_BAD_ROWS        0x10u  /* malformed cu_rows for a request (see above)      */
#define SPEC_STATUS_BAD_SELECTED    0x20u  /* selected token outside [0, V): confidence 0      */
#define SPEC_STATUS_BAD_RELAXED_K   0x40u  /* relaxed K < 1: treated as 1                      */
#define SPEC_STATUS_BAD_BUDGET      0x80u  /* max_rows < B: budget ignored                     */
#define SPEC_STATUS_TIMEOUT         0x100u /* an on-chip copy wait gave up; results invalid    */
#define SPEC_STATUS_BAD_MARGIN      0x200u /* confidence margin NaN: request verified strictly */

/* A ragged batch of packed verify rows (all pointers device memory). */
typedef struct {
    const void *logits;        /* [R_cap, ld] target logits                            */
    int32_t dtype;             /* spec_dtype                                           */
    int32_t V;                 /* vocabulary size, 1 <= V <= ld                        */
    int64_t ld;                /* leading dimension in elements                       */
    int32_t B;                 /* requests, >= 1                                       */
    int32_t k_max;             /* max draft tokens per request, 0..31                  */
    int32_t R_cap;             /* HOST-known upper bound on R = cu_rows[B]; rows beyond
                                  R are ignored.  Normally B * (k_max + 1).            */
    const int32_t *cu_rows;    /* [B+1] row offsets                                     */
    const int32_t *draft_ids;  /* [R_cap] draft token per packed row                   */
} spec_batch;

/* Outputs (device).  The first three are required; the rest may be NULL. */
typedef struct {
    int32_t *accepted_len;     /* [B] accepted draft tokens a_b in [0, k_b]            */
    int32_t *out_tokens;       /* [B, k_max+1] accepted drafts, then the target token,
                                  then -1 padding                                      */
    int32_t *next_token;       /* [B] the target token (replacement or bonus)          */
    float *row_max;            /* [R_cap] max logit of each row                        */
    float *row_lse;            /* [R_cap] log-sum-exp of each row (fp32)               */
    int32_t *row_argmax;       /* [R_cap] first argmax of each row                     */
    int32_t *row_token;        /* [R_cap] target token of each row (argmax or sample)  */
    uint32_t *status;          /* [1] SPEC_STATUS_* bits, OR-ed                        */
    int64_t *acc;              /* [k_max] += #{b : a_b > j}   (fused prefix stats)     */
    int64_t *ver;              /* [k_max] += #{b : k_b > j}                            */
    int64_t *hist;             /* [k_max+1] += 1 at a_b                                */
} spec_outputs;

/* Per-request sampling parameters (device arrays of length B). */
typedef struct {
    const float *temperature;  /* T >= 0; 0 = greedy (first argmax)                    */
    const int32_t *top_k;      /* 0 or >= V = off; else keep values >= k-th largest    */
    const float *top_p;        /* (0, 1]; 1 = off                                      */
    const float *min_p;        /* [0, 1]; 0 = off; keep exp((z - max)/T) >= min_p      */
    const uint64_t *seed;      /* Philox4x32-10 key per request                        */
    const uint32_t *request_id;/* counter word; NULL = the request index b             */
    uint32_t step;             /* counter word supplied by the caller (decode step)    */
} spec_sampling;

/*
 * Workspace for the verify calls: per-row and per-chunk scratch (a row is
 * processed as ceil(V * element bytes / 32 KiB) chunks) and per-request
 * tickets; for spec_verify_sample (sampling != 0) also the sampler's
 * per-chunk candidate lists and mass bins (4.5 KiB per chunk).  Size from
 * spec_workspace_bytes(R_cap, B, V, dtype, sampling).  It must be
 * ZERO-FILLED once before its first use; every completed call leaves the
 * ticket words at zero again, so one zeroed workspace serves any number of
 * stream-ordered calls.  Returns 0 for invalid sizes.
 */
SPEC_API size_t spec_workspace_bytes(int32_t R_cap, int32_t B, int32_t V, int32_t dtype,
                                     int32_t sampling);

/*
 * A1 + A2: greedy verification (vSpec README §"EAGLE 功能": strict greedy
 * top-1).  Per row: max, log-sum-exp (fp32), first argmax in one pass over
 * the logits.  Per request: a_b = the longest prefix with
 * draft_ids[r] == argmax(row r); out_tokens = drafts[0..a_b-1] followed by
 * argmax(row cu_rows[b] + a_b) (the correction, or the bonus when a_b = k_b).
 */
SPEC_API int spec_verify_greedy(const spec_batch *batch, const spec_outputs *out,
                       void *workspace, size_t workspace_bytes, spec_stream stream);

/*
 * spec_verify_greedy for callers that cannot allocate device memory.  This
 * entry point has no counterpart in the method; it is a convenience of this
 * library.  Some callers cannot call cudaMalloc at the point where they
 * verify: a plugin running inside an engine that owns the whole device
 * memory pool, or a serving loop that forbids allocation (and its latency or
 * failure) once it is running.  They pass inputs and outputs only; the
 * workspace is a scratch array of SPEC_NOALLOC_SCRATCH_BYTES compiled into
 * the library, which every GPU that loads the library holds until the
 * process exits.
 *
 * Same inputs, outputs and results as spec_verify_greedy.  A batch whose
 * workspace (spec_workspace_bytes(R_cap, B, V, dtype, 0)) exceeds
 * SPEC_NOALLOC_SCRATCH_BYTES returns SPEC_ERR_WORKSPACE before any launch
 * (about 250 KiB suffice for 640 rows of a 152064-token vocabulary).
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress), so the address is never stale after a device
 * reset or under a non-primary context.  The array used is the current
 * device's: the inputs and outputs must be on that device (the Python
 * binding refuses a mismatch).  Every call shares the one array: calls that
 * can overlap on the GPU (two streams, two host threads) race and must be
 * ordered by the caller.  Each call clears the array's ticket words itself
 * on its stream before its kernels run.  Nothing is allocated or freed.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
SPEC_API int spec_verify_greedy_noalloc(const spec_batch *batch, const spec_outputs *out,
                                        spec_stream stream);

/*
 * A5: relaxed top-K acceptance with a strict prefix (vSpec README
 * §"支持范围", §"EAGLE 功能").  Draft d of row r is accepted iff d is in
 * [0, V) and #{i : z_r[i] > z_r[d]} < relaxed_k[b] (ties with the K-th value
 * accepted); acceptance stops at the first failure; the token emitted after
 * the prefix is that row's first argmax.  relaxed_k[b] = 1 is top-1 by value.
 * relaxed_k: device [B].
 */
SPEC_API int spec_verify_relaxed_topk(const spec_batch *batch, const int32_t *relaxed_k,
                             const spec_outputs *out, void *workspace,
                             size_t workspace_bytes, spec_stream stream);

/*
 * Greedy verification over an active vocabulary (vSpec README §"EAGLE 功能",
 * §"代码所有权": an active-vocabulary target LM head with a full token-id
 * map).  The logits have batch->V columns; column i stands for the full
 * token id vocab_ids[i].  A row's token is vocab_ids[first argmax column];
 * draft_ids hold FULL token ids and are accepted while they equal the row's
 * token; out_tokens and next_token are full ids.  Optional row outputs:
 * row_argmax is the column, row_token the full id.  The page's active
 * vocabulary presumes pure greedy decoding, so there is no sampling variant.
 * vocab_ids: device [batch->V], read only; ids are copied as given (a full
 * id outside the model's vocabulary is the caller's error).  Returns
 * SPEC_ERR_INVALID_ARG before any launch for a NULL map.  Workspace as for
 * spec_verify_greedy (with V = the active column count).
 */
SPEC_API int spec_verify_greedy_active(const spec_batch *batch, const int32_t *vocab_ids,
                                       const spec_outputs *out, void *workspace,
                                       size_t workspace_bytes, spec_stream stream);

/*
 * Greedy verification loosened by a confidence margin (vSpec README §"启动"
 * approximate-acceptance preset; §"通用参数": --confidence-accept-margin,
 * --confidence-accept-from-position / --confidence-accept-after-tokens,
 * --confidence-protected-token-ids).  The result is no longer guaranteed to
 * equal target-only greedy decoding.  Draft d at position j of request b
 * (row r = cu_rows[b] + j, j < k_b) is accepted iff d is in [0, V) and
 *   d == argmax(row r)  (first argmax: the strict rule always applies), or
 *   j >= from_position, generated[b] + j >= after_tokens, d is not in
 *   protected_ids, and max(row r) - z_r[d] <= margin[b] with the difference
 *   rounded to fp32 (both values are exact in fp32).
 * Acceptance stops at the first failure; the token emitted after the prefix
 * is that row's first argmax.  A negative margin keeps request b strict; a
 * NaN margin does too and sets SPEC_STATUS_BAD_MARGIN.
 * Inputs (device memory, owned by the caller, read only):
 *   margin         [B] f32 logit margins; required.
 *   generated      [B] i32 tokens request b produced before this step, or
 *                  NULL (all 0).
 *   protected_ids  [n_protected] i32 token ids the margin never accepts, in
 *                  any order; NULL when n_protected = 0.  Each draft row
 *                  scans the list once (n_protected / 32 loads per lane).
 * Returns SPEC_ERR_INVALID_ARG before any launch for a NULL margin,
 * n_protected < 0, or n_protected > 0 with a NULL list.  Workspace as for
 * spec_verify_greedy.
 */
typedef struct {
    const float *margin;
    const int32_t *generated;
    const int32_t *protected_ids;
    int32_t n_protected;
    int32_t from_position;
    int32_t after_tokens;
} spec_margin;

SPEC_API int spec_verify_greedy_margin(const spec_batch *batch, const spec_margin *margin,
                                       const spec_outputs *out, void *workspace,
                                       size_t workspace_bytes, spec_stream stream);

/*
 * A1 + A3 + A4: stochastic verification with a point-mass draft (xLLM
 * "自适应投机推理" §"启动示例").  For row r of request b with T_b > 0:
 *   survivors F = {i : z_i >= top-k threshold} ∩ {i : exp((z_i-max)/T) >= min_p},
 *   then top-p over them: keep i iff the mass (weights exp((z-max)/T)) of
 *   survivors with a strictly larger logit is < top_p * (their total mass);
 *   ties are kept or cut as whole groups.
 *   y_r = argmax_{i in F} ( z_i / T - log(-log u_i) ), lowest index on ties,
 *   u_i = (2*(x>>9)+1) * 2^-24 with x = word (i & 3) of
 *   Philox4x32-10(counter = (i >> 2, j, request_id_b, step),
 *                 key = (low 32 bits of seed_b, high 32 bits)),
 *   j = position of row r within its request.
 * T_b = 0 gives y_r = first argmax.  Then accept while y == draft; the first
 * mismatching y is the replacement, else the last row's y is the bonus.
 * Rows are decided in fp32; results equal the fp64 definition except where a
 * top-p / min-p decision or the Gumbel winner is within float rounding of a
 * tie.
 */
SPEC_API int spec_verify_sample(const spec_batch *batch, const spec_sampling *params,
                       const spec_outputs *out, void *workspace, size_t workspace_bytes,
                       spec_stream stream);

/* Draft-side inputs of the adaptive target verification. */
typedef struct {
    const void *draft_logits;  /* [B*k, ld] draft logits; row b*k + j = position j      */
    int32_t dtype;             /* spec_dtype                                           */
    int32_t V;
    int64_t ld;
    int32_t B;                 /* requests, >= 1                                       */
    int32_t k;                 /* draft width, 1..31                                   */
    const int32_t *selected;   /* [B*k] selected draft token, NULL = draft argmax      */
    float threshold;           /* cumulative-confidence threshold tau                  */
    int32_t max_rows;          /* global row budget G (0 = none); needs G >= B         */
} spec_draft;

/* Outputs of spec_draft_confidence (device). */
typedef struct {
    float *conf;               /* [B*k] exp(z[s] - logsumexp(z))                       */
    int32_t *draft_token;      /* [B*k] the selected token s of each draft position    */
    int32_t *k_alloc;          /* [B] allocated draft positions k_b                    */
    int32_t *cu_rows;          /* [B+1] packed row offsets                             */
    int32_t *row_owner;        /* [B*(k+1)] owner request of packed row r, -1 beyond R */
    int32_t *row_pos;          /* [B*(k+1)] position j of packed row r, -1 beyond R    */
    int32_t *packed_draft;     /* [B*(k+1)] draft token of packed row r (-1 on bonus
                                  rows and beyond R); may be NULL                      */
    int32_t *total_rows;       /* [1] R = cu_rows[B]                                   */
    uint32_t *status;          /* [1] SPEC_STATUS_* bits; may be NULL                  */
} spec_allocation;

/*
 * A6 + A7 (xLLM "自适应投机推理" §"基于 MTP logits 的自适应 target 验证"):
 * conf[b*k+j] = exp(z[s] - logsumexp(z)) over draft row b*k+j, s = selected
 * token (default: the first argmax).  Cumulative confidence
 * c_{b,j} = prod_{i<=j} conf[b*k+i] (fp32, in order); k_b = #{j : c_{b,j} >= tau}
 * (a prefix, since c is non-increasing).  With max_rows = G > 0 and
 * sum(k_b + 1) > G, only the best G - B positions are kept, ordered by
 * (c desc, b asc, j asc).  Then cu_rows = exclusive scan of (k_b + 1) and the
 * per-row owner / position / draft token of the packed layout.  Three kernel
 * launches (the draft rows' streaming pass, the per-row finish, the
 * allocation), the last two chained by programmatic dependent launch;
 * nothing is read back to the host.  The workspace comes from
 * spec_draft_workspace_bytes.  A batch with 8 B k + 16 B + 4 bytes above
 * 200 KiB (the allocation stages it on chip) returns SPEC_ERR_UNSUPPORTED.
 */
SPEC_API int spec_draft_confidence(const spec_draft *draft, const spec_allocation *out,
                                   void *workspace, size_t workspace_bytes, spec_stream stream);

/* Workspace bytes of spec_draft_confidence (zero-filled once before first
 * use, like the verify workspace); 0 for invalid sizes. */
SPEC_API size_t spec_draft_workspace_bytes(int32_t B, int32_t k, int32_t V, int32_t dtype);

/*
 * Restore of compact rows to request slots (xLLM "自适应投机推理"
 * §"基于 MTP logits 的自适应 target 验证": the outputs of the compact
 * target rows, such as hidden states, are restored by the device offsets
 * before the draft context is updated).  For each request b whose offsets
 * are well formed (cu_rows as for the verify calls, and cu_rows[B] <= R_cap),
 * slot b * (k_max + 1) + j of `out` receives the first row_bytes bytes of
 * compact row cu_rows[b] + j, for j = 0 .. k_b.  Other slots are untouched.
 * A malformed request is skipped and sets SPEC_STATUS_BAD_ROWS.
 *   compact  device [R_cap rows, compact_ld bytes each], read only.
 *   out      device [B * (k_max + 1) rows, out_ld bytes each]; must not
 *            overlap `compact`.
 *   cu_rows  device [B + 1], e.g. spec_draft_confidence's output.
 *   status   device [1] or NULL.
 * Rows are opaque bytes, so any element type works.  Returns
 * SPEC_ERR_INVALID_ARG for NULL pointers, B < 1, R_cap < 1, k_max < 0,
 * row_bytes < 1 or a stride below row_bytes; SPEC_ERR_UNSUPPORTED for
 * k_max > 31, row_bytes > 2^30, B * (k_max + 1) > 2^31 - 1, or when
 * row_bytes, either stride or either base address is not a multiple of 16.
 * One kernel launch; HBM-bound (each restored row read and written once).
 */
SPEC_API int spec_restore_rows(const void *compact, int64_t compact_ld, int32_t R_cap,
                               const int32_t *cu_rows, int32_t B, int32_t k_max,
                               int64_t row_bytes, void *out, int64_t out_ld, uint32_t *status,
                               spec_stream stream);

/*
 * A8 (xLLM "自适应投机推理" §"自适应 draft 步长（MTP）"): accumulate
 * acc[j] += #{b : a_b > j}, ver[j] += #{b : k_b > j} for j < k_max and
 * hist[a_b] += 1 (hist may be NULL).  prefix_acceptance[j] = acc[j] / ver[j].
 * Requests with malformed rows or a_b outside [0, k_b] are skipped and set
 * SPEC_STATUS_BAD_ROWS.  One kernel launch.
 */
SPEC_API int spec_prefix_stats(const int32_t *accepted_len, const int32_t *cu_rows, int32_t B,
                      int32_t k_max, int64_t *acc, int64_t *ver, int64_t *hist,
                      uint32_t *status, spec_stream stream);

/* Human-readable name of a spec_result code (static string). */
SPEC_API const char *spec_result_string(int code);

/* Text of the last CUDA error seen by this library in the calling thread. */
SPEC_API const char *spec_last_cuda_error(void);

/* ABI version of this header (major * 100 + minor). */
SPEC_API int spec_abi_version(void);

#define SPEC_ABI_VERSION 100

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
