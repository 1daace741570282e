// internal.h -- declarations shared by the translation units of libspecverify.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

enum Mode : int { MODE_GREEDY = 0, MODE_RELAXED = 1, MODE_SAMPLE = 2, MODE_CONF = 3 };

// Workspace of the row kernel, per packed row r and chunk c (a row is split
// into nchunk = ceil(V * elt / kChunkBytes) chunks, one work item each):
//   info[r]     (64 bytes) owner request and parameters of the row
//   part[r][c]  (32 bytes) chunk reduction and sampler summary
//   cand[r][c]  (kWsCandCap (value, index) pairs) candidate lists, or for
//               bf16 top-p alone the listed elements and value counts
//                                                             (sampler only)
constexpr int kWsCandCap = 512;

// Everything one verify launch needs (passed by value to the row kernel).
struct VerifyParams {
    const void *logits;
    int64_t ld;
    int32_t V, B, k_max, R_cap;
    const int32_t *cu_rows;      // [B+1]        (not used by MODE_CONF)
    const int32_t *draft_ids;    // [R_cap]
    // stochastic verification
    const float *temperature;
    const int32_t *top_k;
    const float *top_p;
    const float *min_p;
    const uint64_t *seed;
    const uint32_t *request_id;
    uint32_t step;
    // relaxed top-K
    const int32_t *relaxed_k;
    // greedy with a confidence margin (margin == nullptr: strict greedy)
    const float *margin;
    const int32_t *generated;
    const int32_t *protected_ids;
    int32_t n_protected, from_position, after_tokens;
    // greedy over an active vocabulary: full token id of each column (or nullptr)
    const int32_t *vocab_ids;
    // draft confidence (MODE_CONF: rows are draft positions)
    const int32_t *selected;
    float *conf;
    int32_t *draft_token;
    // request outputs
    int32_t *accepted_len;
    int32_t *out_tokens;
    int32_t *next_token;
    // optional row outputs
    float *row_max;
    float *row_lse;
    int32_t *row_argmax;
    int32_t *row_token;
    uint32_t *status;
    // optional fused prefix statistics
    int64_t *acc;
    int64_t *ver;
    int64_t *hist;
    // workspace
    int32_t *ws_tok;             // [R_cap] per-row target token
    int32_t *ws_flag;            // [R_cap] per-row relaxed acceptance
    uint32_t *ws_ticket;         // [B] arrivals per request (zero between calls)
    void *ws_info;               // [R_cap] row records (64 bytes each)
    void *ws_part;               // [R_cap * nchunk] chunk partials (32 bytes each)
    void *ws_cand;               // [R_cap * nchunk * kWsCandCap] (value, index) pairs
    int32_t nchunk;              // chunks per row
    int32_t n_rows;              // rows of the work (R_cap; draft rows for the confidence)
};

struct AllocParams {
    const float *conf;
    const int32_t *draft_token;
    int32_t B, k;
    float threshold;
    int32_t max_rows;
    int32_t *k_alloc;
    int32_t *cu_rows;
    int32_t *row_owner;
    int32_t *row_pos;
    int32_t *packed_draft;
    int32_t *total_rows;
    uint32_t *status;
};

// Host launchers (return cudaError_t of the launch).
cudaError_t launch_verify(int mode, int dtype, const VerifyParams &p, cudaStream_t stream);
// the row path of relaxed top-K (bf16, large batches; called by launch_verify)
cudaError_t launch_relaxed_rows(const VerifyParams &p, cudaStream_t stream);
cudaError_t launch_alloc(const AllocParams &p, cudaStream_t stream);
cudaError_t launch_restore_rows(const void *src, int64_t src_ld, int32_t R_cap,
                                const int32_t *cu_rows, int32_t B, int32_t k_max,
                                int64_t row_bytes, void *dst, int64_t dst_ld, uint32_t *status,
                                cudaStream_t stream);
cudaError_t launch_prefix_stats(const int32_t *accepted_len, const int32_t *cu_rows, int32_t B,
                                int32_t k_max, int64_t *acc, int64_t *ver, int64_t *hist,
                                uint32_t *status, cudaStream_t stream);

// Largest row (bytes) the verify path accepts.
size_t max_row_bytes();

// chunks per row for a vocabulary of V elements of `elt` bytes
int chunks_per_row(int32_t V, int elt);

// workspace bytes of the row kernel (sampling adds the candidate lists)
size_t row_workspace_bytes(int32_t R_cap, int32_t B, int32_t V, int elt, bool sampling);

}  // namespace specv
