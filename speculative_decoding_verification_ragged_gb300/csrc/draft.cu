// draft.cu -- prefix-budget allocation / packing, the restore of compact
// rows to request slots, and prefix-acceptance counters (xLLM docs
// "自适应投机推理": §"基于 MTP logits 的自适应 target 验证" -- confidence kept
// on device, prefix allocation and packing with device offsets, compact
// target outputs restored by those offsets; §"自适应 draft 步长（MTP）" --
// per-position prefix acceptance).  The draft confidences themselves come from the row kernel
// in verify.cu (MODE_CONF).
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace specv {

constexpr int kAllocThreads = 256;

// block-wide sum of an int64 over kAllocThreads threads
__device__ long long block_sum(long long v, long long *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < kAllocThreads / 32; ++w) t += scratch[w];
    __syncthreads();
    return t;
}

// Exclusive scan of v[0..n) in place (kAllocThreads threads, tiles of one
// value per thread); returns the total.
__device__ int block_exclusive_scan(int *v, int n, int *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int carry = 0;
    for (int base = 0; base < n; base += kAllocThreads) {
        const int i = base + threadIdx.x;
        const int x = (i < n) ? v[i] : 0;
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) scratch[warp] = incl;
        __syncthreads();
        int off = carry;
        for (int w = 0; w < warp; ++w) off += scratch[w];
        int tile = 0;
        for (int w = 0; w < kAllocThreads / 32; ++w) tile += scratch[w];
        if (i < n) v[i] = off + incl - x;
        __syncthreads();
        carry += tile;
    }
    return carry;
}

__global__ void __launch_bounds__(kAllocThreads) alloc_kernel(const AllocParams p)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    // launched while the confidence kernels run: their results are complete
    // and visible past this wait
    griddep_wait();
    const int B = p.B, k = p.k, Q = B * k;
    float *cum = reinterpret_cast<float *>(smem_raw);        // [Q]
    int *tok = reinterpret_cast<int *>(cum + Q);             // [Q]
    int *ka = tok + Q;                                       // [B]
    int *gt = ka + B;                                        // [B]
    int *eq = gt + B;                                        // [B]
    int *cu = eq + B;                                        // [B+1]
    __shared__ long long lsum[kAllocThreads / 32];
    __shared__ int iscr[kAllocThreads / 32];
    const int tid = threadIdx.x;

    // the confidences and draft tokens staged in shared memory, every load
    // in flight at once
    for (int q = tid; q < Q; q += kAllocThreads) {
        cum[q] = p.conf[q];
        tok[q] = p.draft_token[q];
    }
    __syncthreads();
    // cumulative confidence per request (in order, fp32) and threshold count
    for (int b = tid; b < B; b += kAllocThreads) {
        float c = 1.f;
        int cnt = 0;
        for (int j = 0; j < k; ++j) {
            c *= cum[b * k + j];
            cum[b * k + j] = c;
            cnt += (c >= p.threshold) ? 1 : 0;
        }
        ka[b] = cnt;
    }
    __syncthreads();

    long long want = 0;
    for (int b = tid; b < B; b += kAllocThreads) want += ka[b] + 1;
    want = block_sum(want, lsum);

    if (p.max_rows > 0 && want > p.max_rows) {
        if (p.max_rows < B) {
            if (tid == 0) set_status(p.status, SPEC_STATUS_BAD_BUDGET);
        } else {
            const long long keep = static_cast<long long>(p.max_rows) - B;
            // key of the keep-th largest eligible cumulative confidence, by a
            // bitwise search for the largest key with count(key' >= key) >= keep
            uint32_t key = 0u;
            if (keep > 0) {
                for (int bit = 31; bit >= 0; --bit) {
                    const uint32_t cand = key | (1u << bit);
                    long long cnt = 0;
                    for (int q = tid; q < Q; q += kAllocThreads) {
                        const int b = q / k, j = q - b * k;
                        if (j < ka[b] && fkey(cum[q]) >= cand) ++cnt;
                    }
                    cnt = block_sum(cnt, lsum);
                    if (cnt >= keep) key = cand;
                }
            }
            // entries above the key are kept; ties at the key go in (b, j) order
            for (int b = tid; b < B; b += kAllocThreads) {
                int g = 0, e = 0;
                for (int j = 0; j < ka[b]; ++j) {
                    const uint32_t kq = fkey(cum[b * k + j]);
                    if (keep > 0 && kq > key) ++g;
                    else if (keep > 0 && kq == key) ++e;
                }
                gt[b] = g;
                eq[b] = e;
            }
            __syncthreads();
            long long ngt = 0;
            for (int b = tid; b < B; b += kAllocThreads) ngt += gt[b];
            ngt = block_sum(ngt, lsum);
            block_exclusive_scan(eq, B, iscr);   // eq[b] := ties of requests before b
            __syncthreads();
            const long long rem = keep - ngt;
            for (int b = tid; b < B; b += kAllocThreads) {
                int e = 0;
                for (int j = 0; j < ka[b]; ++j)
                    if (keep > 0 && fkey(cum[b * k + j]) == key) ++e;
                long long take = rem - eq[b];
                take = take < 0 ? 0 : (take > e ? e : take);
                ka[b] = (keep > 0) ? gt[b] + static_cast<int>(take) : 0;
            }
            __syncthreads();
        }
    }

    // packing: row offsets, owner / position / draft token of every row
    for (int b = tid; b < B; b += kAllocThreads) cu[b] = ka[b] + 1;
    __syncthreads();
    const int R = block_exclusive_scan(cu, B, iscr);
    __syncthreads();
    const int cap = B * (k + 1);
    for (int r = R + tid; r < cap; r += kAllocThreads) {
        p.row_owner[r] = -1;
        p.row_pos[r] = -1;
        if (p.packed_draft) p.packed_draft[r] = -1;
    }
    for (int b = tid; b < B; b += kAllocThreads) {
        p.k_alloc[b] = ka[b];
        p.cu_rows[b] = cu[b];
        for (int j = 0; j <= ka[b]; ++j) {
            const int r = cu[b] + j;
            p.row_owner[r] = b;
            p.row_pos[r] = j;
            if (p.packed_draft) p.packed_draft[r] = (j < ka[b]) ? tok[b * k + j] : -1;
        }
    }
    if (tid == 0) {
        p.cu_rows[B] = R;
        p.total_rows[0] = R;
    }
}

cudaError_t launch_alloc(const AllocParams &p, cudaStream_t stream)
{
    const size_t smem = static_cast<size_t>(p.B) * p.k * (sizeof(float) + sizeof(int)) +
                        (static_cast<size_t>(p.B) * 4 + 1) * sizeof(int);
    // the shared-memory limit is raised once per device (to the most any
    // accepted batch needs: the entry point bounds it by 200 KiB)
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(alloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    // programmatic dependent launch after the confidence kernels (the
    // kernel waits for them before reading)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kAllocThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, alloc_kernel, p);
}

// ------------------------------------------ compact rows to request slots --

// xLLM "自适应投机推理" §"基于 MTP logits 的自适应 target 验证": outputs of the
// compact target rows (hidden states, per-row results) are restored to their
// request slots by the device offsets.  Slot s = (b, j) takes compact row
// cu_rows[b] + j when j <= k_b; other slots are left untouched.  Rows are
// opaque bytes in 16-byte vectors (alignment checked on the host).
// blockIdx.x selects an 8 KiB piece of the row and blockIdx.y strides over
// the slots; a thread moves two vectors, both loads issued before the
// stores.  HBM-bound: each restored row is read once and written once.
constexpr int kRestoreThreads = 256;
constexpr int kRestoreVecs = 2 * kRestoreThreads;

__global__ void __launch_bounds__(kRestoreThreads) restore_rows_kernel(
    const uint8_t *__restrict__ src, int64_t src_ld, int32_t R_cap,
    const int32_t *__restrict__ cu_rows, int32_t B, int32_t k_max, int64_t vecs,
    uint8_t *__restrict__ dst, int64_t dst_ld, uint32_t *status)
{
    const int32_t k1 = k_max + 1;
    const int32_t slots = B * k1;
    const int32_t c0 = __ldg(cu_rows);
    const int64_t va = static_cast<int64_t>(blockIdx.x) * kRestoreVecs + threadIdx.x;
    const int64_t vb = va + kRestoreThreads;
    for (int32_t s = blockIdx.y; s < slots; s += gridDim.y) {
        const int32_t b = s / k1, j = s - b * k1;
        const int64_t lo = __ldg(cu_rows + b), hi = __ldg(cu_rows + b + 1);
        const int64_t n = hi - lo;
        const bool ok = c0 == 0 && lo >= 0 && n >= 1 && n - 1 <= k_max && hi <= R_cap;
        if (!ok) {
            if (j == 0 && blockIdx.x == 0 && threadIdx.x == 0) set_status(status, SPEC_STATUS_BAD_ROWS);
            continue;
        }
        if (j >= n) continue;
        const uint4 *in = reinterpret_cast<const uint4 *>(src + (lo + j) * src_ld);
        uint4 *out = reinterpret_cast<uint4 *>(dst + static_cast<int64_t>(s) * dst_ld);
        uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
        if (va < vecs) xa = __ldcs(in + va);
        if (vb < vecs) xb = __ldcs(in + vb);
        if (va < vecs) __stcs(out + va, xa);
        if (vb < vecs) __stcs(out + vb, xb);
    }
}

cudaError_t launch_restore_rows(const void *src, int64_t src_ld, int32_t R_cap,
                                const int32_t *cu_rows, int32_t B, int32_t k_max,
                                int64_t row_bytes, void *dst, int64_t dst_ld, uint32_t *status,
                                cudaStream_t stream)
{
    const int64_t vecs = row_bytes / 16;
    const int64_t slots = static_cast<int64_t>(B) * (k_max + 1);
    const dim3 grid(static_cast<unsigned>((vecs + kRestoreVecs - 1) / kRestoreVecs),
                    static_cast<unsigned>(slots < 65535 ? slots : 65535));
    restore_rows_kernel<<<grid, kRestoreThreads, 0, stream>>>(
        static_cast<const uint8_t *>(src), src_ld, R_cap, cu_rows, B, k_max, vecs,
        static_cast<uint8_t *>(dst), dst_ld, status);
    return cudaGetLastError();
}

// ------------------------------------------------- prefix statistics -----

__global__ void __launch_bounds__(1024) prefix_stats_kernel(const int32_t *accepted_len,
                                                            const int32_t *cu_rows, int32_t B,
                                                            int32_t k_max, int64_t *acc,
                                                            int64_t *ver, int64_t *hist,
                                                            uint32_t *status)
{
    __shared__ unsigned int cacc[32], cver[32], chist[33];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid < 33) { chist[tid] = 0u; if (tid < 32) { cacc[tid] = 0u; cver[tid] = 0u; } }
    if (tid == 0) bad = 0;
    __syncthreads();
    const int32_t c0 = __ldg(cu_rows);
    for (int b = blockIdx.x * blockDim.x + tid; b < B; b += gridDim.x * blockDim.x) {
        const int32_t n = __ldg(cu_rows + b + 1) - __ldg(cu_rows + b);
        const int32_t k = n - 1, a = __ldg(accepted_len + b);
        if (c0 != 0 || n < 1 || k > k_max || a < 0 || a > k) { bad = 1; continue; }
        for (int j = 0; j < k_max; ++j) {
            if (a > j) atomicAdd(&cacc[j], 1u);
            if (k > j) atomicAdd(&cver[j], 1u);
        }
        atomicAdd(&chist[a], 1u);
    }
    __syncthreads();
    if (tid < k_max) {
        if (cacc[tid]) atomicAdd(reinterpret_cast<unsigned long long *>(acc + tid), cacc[tid]);
        if (cver[tid]) atomicAdd(reinterpret_cast<unsigned long long *>(ver + tid), cver[tid]);
    }
    if (hist && tid <= k_max && chist[tid])
        atomicAdd(reinterpret_cast<unsigned long long *>(hist + tid), chist[tid]);
    if (tid == 0 && bad) set_status(status, SPEC_STATUS_BAD_ROWS);
}

cudaError_t launch_prefix_stats(const int32_t *accepted_len, const int32_t *cu_rows, int32_t B,
                                int32_t k_max, int64_t *acc, int64_t *ver, int64_t *hist,
                                uint32_t *status, cudaStream_t stream)
{
    int grid = (B + 1023) / 1024;
    grid = grid < 1 ? 1 : (grid > 152 ? 152 : grid);
    prefix_stats_kernel<<<grid, 1024, 0, stream>>>(accepted_len, cu_rows, B, k_max, acc, ver,
                                                  hist, status);
    return cudaGetLastError();
}

}  // namespace specv
