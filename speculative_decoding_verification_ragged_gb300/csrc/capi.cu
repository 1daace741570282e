// capi.cu -- the extern "C" entry points of libspecverify: host-side argument
// checks (nothing is launched when they fail), workspace layout, dispatch.
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "internal.h"

using namespace specv;

namespace {

thread_local char g_cuda_error[256] = "no error";

int cuda_fail(cudaError_t e)
{
    std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return SPEC_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t elt_bytes(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

struct WsLayout {
    int32_t *tok, *flag;
    uint32_t *ticket;
    void *info, *part, *cand;
};

// tok [R_cap] | flag [R_cap] | ticket [B] | info [R_cap * 64 B] |
// part [R_cap * nchunk * 32 B] | cand (sampler only); 256-byte aligned
size_t ws_bytes(int32_t R_cap, int32_t B, int32_t V, int elt, bool sampling)
{
    const size_t R = static_cast<size_t>(R_cap);
    const size_t rc = R * static_cast<size_t>(chunks_per_row(V, elt));
    size_t n = 2 * align256(R * 4) + align256(static_cast<size_t>(B) * 4) + align256(R * 64) +
               align256(rc * 32);
    if (sampling) n += align256(rc * kWsCandCap * 8);
    return n;
}

WsLayout ws_layout(void *ws, int32_t R_cap, int32_t B, int32_t V, int elt, bool sampling)
{
    uint8_t *p = static_cast<uint8_t *>(ws);
    const size_t R = static_cast<size_t>(R_cap);
    const size_t rc = R * static_cast<size_t>(chunks_per_row(V, elt));
    WsLayout l = {};
    l.tok = reinterpret_cast<int32_t *>(p);
    p += align256(R * 4);
    l.flag = reinterpret_cast<int32_t *>(p);
    p += align256(R * 4);
    l.ticket = reinterpret_cast<uint32_t *>(p);
    p += align256(static_cast<size_t>(B) * 4);
    l.info = p;
    p += align256(R * 64);
    l.part = p;
    p += align256(rc * 32);
    if (sampling) l.cand = p;
    return l;
}

// checks shared by the three verify entry points
int check_batch(const spec_batch *b, const spec_outputs *o)
{
    if (!b || !o) return SPEC_ERR_INVALID_ARG;
    if (!b->logits || !b->cu_rows || !b->draft_ids) return SPEC_ERR_INVALID_ARG;
    if (!o->accepted_len || !o->out_tokens || !o->next_token) return SPEC_ERR_INVALID_ARG;
    if (b->dtype != SPEC_F32 && b->dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (b->V < 1 || b->ld < b->V || b->B < 1 || b->R_cap < 1) return SPEC_ERR_INVALID_ARG;
    if (b->k_max < 0) return SPEC_ERR_INVALID_ARG;
    if (b->k_max > 31) return SPEC_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(b->logits) % elt_bytes(b->dtype)) return SPEC_ERR_INVALID_ARG;
    if (static_cast<size_t>(b->V) * elt_bytes(b->dtype) > max_row_bytes()) return SPEC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(b->R_cap) * b->ld > (int64_t(1) << 40)) return SPEC_ERR_UNSUPPORTED;
    // one CTA per (row, chunk): the grid stays below 2^31
    if (static_cast<int64_t>(b->R_cap) * chunks_per_row(b->V, static_cast<int>(elt_bytes(b->dtype))) >
        INT32_MAX)
        return SPEC_ERR_UNSUPPORTED;
    if ((o->acc == nullptr) != (o->ver == nullptr)) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

VerifyParams base_params(const spec_batch *b, const spec_outputs *o, void *ws, bool sampling)
{
    VerifyParams p;
    std::memset(&p, 0, sizeof p);
    p.logits = b->logits;
    p.ld = b->ld;
    p.V = b->V;
    p.B = b->B;
    p.k_max = b->k_max;
    p.R_cap = b->R_cap;
    p.cu_rows = b->cu_rows;
    p.draft_ids = b->draft_ids;
    p.accepted_len = o->accepted_len;
    p.out_tokens = o->out_tokens;
    p.next_token = o->next_token;
    p.row_max = o->row_max;
    p.row_lse = o->row_lse;
    p.row_argmax = o->row_argmax;
    p.row_token = o->row_token;
    p.status = o->status;
    p.acc = o->acc;
    p.ver = o->ver;
    p.hist = o->hist;
    const int elt = static_cast<int>(elt_bytes(b->dtype));
    const WsLayout l = ws_layout(ws, b->R_cap, b->B, b->V, elt, sampling);
    p.ws_tok = l.tok;
    p.ws_flag = l.flag;
    p.ws_ticket = l.ticket;
    p.ws_info = l.info;
    p.ws_part = l.part;
    p.ws_cand = l.cand;
    p.nchunk = chunks_per_row(b->V, elt);
    p.n_rows = b->R_cap;
    return p;
}

int run_verify(int mode, const spec_batch *b, VerifyParams &p, cudaStream_t s)
{
    const cudaError_t e = launch_verify(mode, b->dtype, p, s);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

// Built-in scratch of spec_verify_greedy_noalloc: a device array of the
// library (zero at load).
static __device__ __align__(256) uint8_t g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context (the host-side
// name of the array is not a device address; only this lookup gives one).
// Looked up on every call, never cached: after a device reset, or under a
// context other than the device's primary one, the module is loaded again
// and the array can move.
int noalloc_scratch(void **ptr)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    *ptr = p;
    return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int32_t R_cap, int32_t B, int32_t V, int32_t dtype, int32_t sampling)
{
    if (R_cap < 1 || B < 1 || V < 1 || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return 0;
    if (static_cast<size_t>(V) * elt_bytes(dtype) > max_row_bytes()) return 0;
    return ws_bytes(R_cap, B, V, static_cast<int>(elt_bytes(dtype)), sampling != 0);
}

size_t spec_draft_workspace_bytes(int32_t B, int32_t k, int32_t V, int32_t dtype)
{
    if (B < 1 || k < 1 || V < 1 || (dtype != SPEC_F32 && dtype != SPEC_BF16)) return 0;
    if (static_cast<size_t>(V) * elt_bytes(dtype) > max_row_bytes()) return 0;
    const int64_t Q = static_cast<int64_t>(B) * k;
    if (Q > INT32_MAX) return 0;
    return ws_bytes(static_cast<int32_t>(Q), 1, V, static_cast<int>(elt_bytes(dtype)), false);
}

int spec_verify_greedy(const spec_batch *batch, const spec_outputs *out, void *workspace,
                       size_t workspace_bytes, spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    if (!workspace || workspace_bytes < ws_bytes(batch->R_cap, batch->B, batch->V,
                                                     static_cast<int>(elt_bytes(batch->dtype)), false))
        return SPEC_ERR_WORKSPACE;
    VerifyParams p = base_params(batch, out, workspace, false);
    return run_verify(MODE_GREEDY, batch, p, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_greedy_noalloc(const spec_batch *batch, const spec_outputs *out, spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    const int elt = static_cast<int>(elt_bytes(batch->dtype));
    if (ws_bytes(batch->R_cap, batch->B, batch->V, elt, false) > SPEC_NOALLOC_SCRATCH_BYTES)
        return SPEC_ERR_WORKSPACE;
    void *ws = nullptr;
    rc = noalloc_scratch(&ws);
    if (rc != SPEC_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the per-request and per-row tickets must start at zero (they are
    // adjacent in the layout); the rest is written before it is read
    const WsLayout l = ws_layout(ws, batch->R_cap, batch->B, batch->V, elt, false);
    const size_t tick = align256(static_cast<size_t>(batch->B) * 4) +
                        align256(static_cast<size_t>(batch->R_cap) * 4);
    cudaError_t e = cudaMemsetAsync(l.ticket, 0, tick, s);
    if (e != cudaSuccess) return cuda_fail(e);
    VerifyParams p = base_params(batch, out, ws, false);
    return run_verify(MODE_GREEDY, batch, p, s);
}

int spec_verify_relaxed_topk(const spec_batch *batch, const int32_t *relaxed_k,
                             const spec_outputs *out, void *workspace, size_t workspace_bytes,
                             spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    if (!relaxed_k) return SPEC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < ws_bytes(batch->R_cap, batch->B, batch->V,
                                                     static_cast<int>(elt_bytes(batch->dtype)), false))
        return SPEC_ERR_WORKSPACE;
    VerifyParams p = base_params(batch, out, workspace, false);
    p.relaxed_k = relaxed_k;
    return run_verify(MODE_RELAXED, batch, p, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_greedy_active(const spec_batch *batch, const int32_t *vocab_ids,
                              const spec_outputs *out, void *workspace, size_t workspace_bytes,
                              spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    if (!vocab_ids) return SPEC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < ws_bytes(batch->R_cap, batch->B, batch->V,
                                                     static_cast<int>(elt_bytes(batch->dtype)), false))
        return SPEC_ERR_WORKSPACE;
    VerifyParams p = base_params(batch, out, workspace, false);
    p.vocab_ids = vocab_ids;
    return run_verify(MODE_GREEDY, batch, p, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_greedy_margin(const spec_batch *batch, const spec_margin *margin,
                              const spec_outputs *out, void *workspace, size_t workspace_bytes,
                              spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    if (!margin || !margin->margin || margin->n_protected < 0 ||
        (margin->n_protected > 0 && !margin->protected_ids))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < ws_bytes(batch->R_cap, batch->B, batch->V,
                                                     static_cast<int>(elt_bytes(batch->dtype)), false))
        return SPEC_ERR_WORKSPACE;
    VerifyParams p = base_params(batch, out, workspace, false);
    p.margin = margin->margin;
    p.generated = margin->generated;
    p.protected_ids = margin->protected_ids;
    p.n_protected = margin->n_protected;
    p.from_position = margin->from_position;
    p.after_tokens = margin->after_tokens;
    return run_verify(MODE_GREEDY, batch, p, reinterpret_cast<cudaStream_t>(stream));
}

int spec_verify_sample(const spec_batch *batch, const spec_sampling *params,
                       const spec_outputs *out, void *workspace, size_t workspace_bytes,
                       spec_stream stream)
{
    int rc = check_batch(batch, out);
    if (rc != SPEC_OK) return rc;
    if (!params || !params->temperature || !params->top_k || !params->top_p || !params->min_p ||
        !params->seed)
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < ws_bytes(batch->R_cap, batch->B, batch->V,
                                                     static_cast<int>(elt_bytes(batch->dtype)), true))
        return SPEC_ERR_WORKSPACE;
    VerifyParams p = base_params(batch, out, workspace, true);
    p.temperature = params->temperature;
    p.top_k = params->top_k;
    p.top_p = params->top_p;
    p.min_p = params->min_p;
    p.seed = params->seed;
    p.request_id = params->request_id;
    p.step = params->step;
    return run_verify(MODE_SAMPLE, batch, p, reinterpret_cast<cudaStream_t>(stream));
}

int spec_draft_confidence(const spec_draft *d, const spec_allocation *o, void *workspace,
                          size_t workspace_bytes, spec_stream stream)
{
    if (!d || !o || !d->draft_logits) return SPEC_ERR_INVALID_ARG;
    if (!o->conf || !o->draft_token || !o->k_alloc || !o->cu_rows || !o->row_owner ||
        !o->row_pos || !o->total_rows)
        return SPEC_ERR_INVALID_ARG;
    if (d->dtype != SPEC_F32 && d->dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (d->V < 1 || d->ld < d->V || d->B < 1 || d->k < 1) return SPEC_ERR_INVALID_ARG;
    if (d->k > 31) return SPEC_ERR_UNSUPPORTED;
    if (!(d->threshold == d->threshold)) return SPEC_ERR_INVALID_ARG;
    if (d->max_rows < 0) return SPEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d->draft_logits) % elt_bytes(d->dtype)) return SPEC_ERR_INVALID_ARG;
    if (static_cast<size_t>(d->V) * elt_bytes(d->dtype) > max_row_bytes()) return SPEC_ERR_UNSUPPORTED;
    const int64_t Q = static_cast<int64_t>(d->B) * d->k;
    if (Q * 8 + (static_cast<int64_t>(d->B) * 4 + 1) * 4 > 200 * 1024) return SPEC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(Q) * d->ld > (int64_t(1) << 40)) return SPEC_ERR_UNSUPPORTED;
    if (Q * chunks_per_row(d->V, static_cast<int>(elt_bytes(d->dtype))) > INT32_MAX)
        return SPEC_ERR_UNSUPPORTED;

    const int elt = static_cast<int>(elt_bytes(d->dtype));
    if (!workspace || workspace_bytes < ws_bytes(static_cast<int32_t>(Q), 1, d->V, elt, false))
        return SPEC_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    VerifyParams p;
    std::memset(&p, 0, sizeof p);
    const WsLayout l = ws_layout(workspace, static_cast<int32_t>(Q), 1, d->V, elt, false);
    p.ws_tok = l.tok;
    p.ws_flag = l.flag;
    p.ws_ticket = l.ticket;
    p.ws_info = l.info;
    p.ws_part = l.part;
    p.nchunk = chunks_per_row(d->V, elt);
    p.logits = d->draft_logits;
    p.ld = d->ld;
    p.V = d->V;
    p.B = d->B;
    p.k_max = d->k;
    p.R_cap = static_cast<int32_t>(Q);
    p.n_rows = static_cast<int32_t>(Q);
    p.selected = d->selected;
    p.conf = o->conf;
    p.draft_token = o->draft_token;
    p.status = o->status;
    cudaError_t e = launch_verify(MODE_CONF, d->dtype, p, s);
    if (e != cudaSuccess) return cuda_fail(e);

    AllocParams a;
    a.conf = o->conf;
    a.draft_token = o->draft_token;
    a.B = d->B;
    a.k = d->k;
    a.threshold = d->threshold;
    a.max_rows = d->max_rows;
    a.k_alloc = o->k_alloc;
    a.cu_rows = o->cu_rows;
    a.row_owner = o->row_owner;
    a.row_pos = o->row_pos;
    a.packed_draft = o->packed_draft;
    a.total_rows = o->total_rows;
    a.status = o->status;
    e = launch_alloc(a, s);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

int spec_prefix_stats(const int32_t *accepted_len, const int32_t *cu_rows, int32_t B,
                      int32_t k_max, int64_t *acc, int64_t *ver, int64_t *hist, uint32_t *status,
                      spec_stream stream)
{
    if (!accepted_len || !cu_rows || !acc || !ver) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || k_max < 0) return SPEC_ERR_INVALID_ARG;
    if (k_max > 31) return SPEC_ERR_UNSUPPORTED;
    const cudaError_t e = launch_prefix_stats(accepted_len, cu_rows, B, k_max, acc, ver, hist,
                                              status, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

int spec_restore_rows(const void *compact, int64_t compact_ld, int32_t R_cap,
                      const int32_t *cu_rows, int32_t B, int32_t k_max, int64_t row_bytes,
                      void *out, int64_t out_ld, uint32_t *status, spec_stream stream)
{
    if (!compact || !cu_rows || !out) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || R_cap < 1 || k_max < 0 || row_bytes < 1 || compact_ld < row_bytes ||
        out_ld < row_bytes)
        return SPEC_ERR_INVALID_ARG;
    if (k_max > 31 || row_bytes > (static_cast<int64_t>(1) << 30)) return SPEC_ERR_UNSUPPORTED;
    if (row_bytes % 16 || compact_ld % 16 || out_ld % 16 ||
        reinterpret_cast<uintptr_t>(compact) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
        return SPEC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(B) * (k_max + 1) > INT32_MAX) return SPEC_ERR_UNSUPPORTED;
    const cudaError_t e = launch_restore_rows(compact, compact_ld, R_cap, cu_rows, B, k_max,
                                              row_bytes, out, out_ld, status,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

const char *spec_result_string(int code)
{
    switch (code) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    default: return "unknown spec_result";
    }
}

const char *spec_last_cuda_error(void) { return g_cuda_error; }

int spec_abi_version(void) { return SPEC_ABI_VERSION; }

}  // extern "C"
