// rows.cu -- the row path of relaxed top-K verification for large bf16
// batches: one CTA per packed row, resident kRowCtas to an SM, streams its
// row through kRowStages shared-memory buffers of kRowPiece bytes with 1-D
// TMA bulk copies (the row is read from HBM once) and keeps every per-row
// quantity in each thread's registers across the pieces, so a piece costs
// no CTA barrier: the maximum, its first index, sum exp(z - max) (rescaled
// when the maximum rises) and the count of logits above the draft's.  A
// piece's buffer is refilled by the last thread to finish with it.  The CTA
// then reduces the row maximum, first argmax, LSE and count, writes the row
// results, and the CTA finishing a request's last row (atomic ticket) runs
// the request chain.  The row record (owner request, position, K, the
// draft's logit) is computed by warp 0 while the first copies are in
// flight; extra CTAs write the outputs of requests without a valid row
// range.  With one CTA per row there is no chunk summary round trip and no
// finish kernel, which pays once the batch fills the SMs several times over.
//
// Definitions: "vllm-hust-vSpec" README §"EAGLE 功能" (relaxed top-K
// acceptance with a strict prefix), xLLM docs "自适应投机推理" §"启动示例"
// (packed-row owners, replacement / bonus token).
#include "rowkit.cuh"

namespace specv {

constexpr int kRowPiece = 32 * 1024;    // bytes of a row staged at a time
constexpr int kRowStages = 2;           // piece buffers per CTA
constexpr int kRowCtas = 3;             // resident CTAs per SM
static_assert(kRowPiece / 16 / kThreads == 8, "eight 16-byte vectors per thread and piece");

// per-CTA shared state, after the piece buffers
struct __align__(16) RowShared {
    Shared sh;
    uint64_t full[kRowStages];
    int32_t cnt[kRowStages];
    int32_t R;
};

__device__ __forceinline__ int64_t lmin64(int64_t a, int64_t b) { return a < b ? a : b; }

__global__ void __launch_bounds__(kThreads, kRowCtas) relaxed_rows_kernel(const VerifyParams p, int row_blocks)
{
    constexpr int MODE = MODE_RELAXED;
    using E = Elt<uint16_t>;
    constexpr int VEC = 8;
    extern __shared__ __align__(128) uint8_t smem[];
    RowShared &rs = *reinterpret_cast<RowShared *>(smem + kRowStages * kRowPiece);
    Shared &sh = rs.sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (static_cast<int>(blockIdx.x) >= row_blocks) {
        bad_request_outputs(p, (blockIdx.x - row_blocks) * kThreads + tid);
        return;
    }
    const int r = blockIdx.x;
    const uint16_t *row = reinterpret_cast<const uint16_t *>(p.logits) + static_cast<int64_t>(r) * p.ld;
    const int V = p.V;
    // the aligned body [a0, a1) in pieces of kRowPiece bytes; head and tail
    // elements (n_extra of them) by plain loads
    const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
    const int a0 = min(mis ? static_cast<int>((16u - mis) / 2) : 0, V);
    const int nvec = (V - a0) / VEC;
    const int a1 = a0 + nvec * VEC;
    const int n_head = a0, n_extra = a0 + (V - a1);
    const int64_t body_bytes = static_cast<int64_t>(nvec) * 16;
    const int np = static_cast<int>((body_bytes + kRowPiece - 1) / kRowPiece);
    constexpr int PE = kRowPiece / 2;                   // elements of a piece
    auto issue = [&](int q) {
        const int s = q % kRowStages;
        const uint32_t bytes = static_cast<uint32_t>(lmin64(kRowPiece, body_bytes - static_cast<int64_t>(q) * kRowPiece));
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&rs.full[s], bytes);
        bulk_g2s(smem + s * kRowPiece, row + a0 + static_cast<int64_t>(q) * PE, bytes, &rs.full[s]);
    };
    if (tid == 0) {
        for (int s = 0; s < kRowStages; ++s) {
            mbar_init(&rs.full[s], 1);
            rs.cnt[s] = 0;
        }
        fence_mbar_init();
        sh.timeout = 0;
        // the logits buffer holds R_cap rows: the first copies go out first
        for (int q = 0; q < min(kRowStages, np); ++q) issue(q);
        rs.R = min(__ldg(p.cu_rows + p.B), p.R_cap);
    }
    if (warp == 0) {
        const RowInfo inf = row_record<uint16_t, MODE>(p, r);
        if (lane == 0) sh.info = inf;
    }
    __syncthreads();
    const RowInfo &info = sh.info;
    if (r >= rs.R || !info.valid) {
        // no outputs for this row: the copies in flight land before leaving
        if (tid == 0)
            for (int q = 0; q < min(kRowStages, np); ++q) mbar_wait(&rs.full[q], 0);
        return;
    }
    const bool need_sum = p.row_lse != nullptr;
    const float zd = info.zd;

    // per-thread running state
    float tmax = -INFINITY, tsum = 0.f;
    int32_t targ = INT_MAX, tcnt = 0;
    uint32_t phase = 0u;
    for (int q = 0; q < np; ++q) {
        const int s = q % kRowStages;
        // every thread waits for the piece itself (no CTA barrier); a wait
        // that times out reports it and the thread skips the piece's data
        const bool ok = mbar_wait(&rs.full[s], (phase >> s) & 1u);
        if (!ok) {
            set_status(p.status, SPEC_STATUS_TIMEOUT);
            sh.timeout = 1;
        }
        phase ^= 1u << s;
        const uint4 *body = reinterpret_cast<const uint4 *>(smem + s * kRowPiece);
        const int nv = ok ? static_cast<int>(lmin64(kRowPiece, body_bytes - static_cast<int64_t>(q) * kRowPiece) / 16) : 0;
        const int base = a0 + q * PE;

        // the piece maximum and its first vector (selects only), then the
        // sum against the running maximum and the count above the draft
        float pm = -INFINITY;
        int pj = -1;
#pragma unroll 4
        for (int i = tid; i < nv; i += kThreads) {
            const float vm = E::vmax(body[i]);
            pj = (vm > pm) ? i : pj;
            pm = fmaxf(pm, vm);
        }
        if (pj >= 0) {
            float x[VEC];
            E::unpack(body[pj], x);
            int first = VEC - 1;
#pragma unroll
            for (int e = VEC - 1; e >= 0; --e)
                if (x[e] == pm) first = e;
            if (pm > tmax) {
                if (need_sum && tmax > -INFINITY) tsum *= ex2((tmax - pm) * kLog2e);
                tmax = pm;
                targ = base + pj * VEC + first;
            }
        }
        const float c0 = -tmax * kLog2e;
        uint64_t acc = f2_pack(0.f, 0.f);
        const uint64_t l2 = f2_pack(kLog2e, kLog2e), c2 = f2_pack(c0, c0);
#pragma unroll 4
        for (int i = tid; i < nv; i += kThreads) {
            const uint4 v = body[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = bf_lo(w[j]), hi = bf_hi(w[j]);
                if (need_sum) {
                    float e0, e1;
                    f2_unpack(f2_fma(f2_pack(lo, hi), l2, c2), e0, e1);
                    acc = f2_add(acc, f2_pack(ex2(e0), ex2(e1)));
                }
                tcnt += ((lo > zd) ? 1 : 0) + ((hi > zd) ? 1 : 0);
            }
        }
        float s0, s1;
        f2_unpack(acc, s0, s1);
        if (tmax > -INFINITY) tsum += s0 + s1;

        // the last thread done with the piece refills its buffer (its reads
        // precede its count: block-scope fence)
        __threadfence_block();
        if (atomicAdd(&rs.cnt[s], 1) == kThreads - 1) {
            rs.cnt[s] = 0;
            if (q + kRowStages < np && !sh.timeout) issue(q + kRowStages);
        }
    }
    __syncthreads();
    if (sh.timeout) {
        // the row cannot be settled (TIMEOUT is reported); copies still in
        // flight land before the CTA leaves (bounded waits)
        if (tid == 0)
            for (int s = 0; s < kRowStages; ++s) mbar_wait(&rs.full[s], (phase >> s) & 1u);
        return;
    }

    // ---- head / tail elements (plain loads)
    if (tid < n_extra) {
        const int32_t ie = (tid < n_head) ? tid : a1 + (tid - n_head);
        const float xe = E::load(row, ie);
        if (xe > tmax || (xe == tmax && ie < targ)) {
            if (need_sum && tmax > -INFINITY && xe > tmax) tsum *= ex2((tmax - xe) * kLog2e);
            if (xe > tmax) tmax = xe;
            targ = ie;
        }
        if (need_sum && tmax > -INFINITY) tsum += ex2((xe - tmax) * kLog2e);
        tcnt += (xe > zd) ? 1 : 0;
    }

    // ---- the row's maximum, first argmax, sum and count (CTA reduction)
    chunk_reduce<MODE>(tmax, targ, tsum, tcnt, need_sum, sh);
    const float M = sh.part.m;
    const int32_t AMAX = (M == -INFINITY) ? 0 : sh.part.amax;
    const float S = sh.part.s;
    const int32_t flag = (info.draft >= 0 && info.draft < V && sh.part.aux < info.K) ? 1 : 0;

    // ---- row results and the request chain
    if (tid == 0) {
        if (p.row_max) p.row_max[r] = M;
        if (p.row_lse) p.row_lse[r] = (S > 0.f) ? M + logf(S) : -INFINITY;
        if (p.row_argmax) p.row_argmax[r] = AMAX;
        if (p.row_token) p.row_token[r] = AMAX;
        p.ws_tok[r] = AMAX;
        p.ws_flag[r] = flag;
    }
    if (warp == 0) {
        uint32_t t = 0;
        if (lane == 0) {
            fence_acq_rel_gpu();
            t = atomicAdd(p.ws_ticket + info.b, 1u);
            if (t == static_cast<uint32_t>(info.k_b)) fence_acq_rel_gpu();
        }
        t = __shfl_sync(0xFFFFFFFFu, t, 0);
        if (t == static_cast<uint32_t>(info.k_b))
            chain_request<MODE>(p, info.b, info.k_b, r - info.pos, static_cast<uint32_t>(info.bad));
    }
}

cudaError_t launch_relaxed_rows(const VerifyParams &p, cudaStream_t stream)
{
    const size_t smem = static_cast<size_t>(kRowStages) * kRowPiece + sizeof(RowShared);
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(relaxed_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(relaxed_rows_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    const int row_blocks = p.R_cap;
    const int req_blocks = (p.B + kThreads - 1) / kThreads;
    relaxed_rows_kernel<<<row_blocks + req_blocks, kThreads, smem, stream>>>(p, row_blocks);
    return cudaGetLastError();
}

}  // namespace specv
