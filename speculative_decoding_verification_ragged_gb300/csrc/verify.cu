// verify.cu -- the kernels of every verification entry point: fused max /
// LSE / argmax over ragged packed logits; greedy acceptance (strict,
// loosened by a confidence margin, or over an active vocabulary); relaxed
// top-K acceptance; the filtered Gumbel-max sampler with the point-mass
// rejection chain; and the draft confidence.
//
// Two kernels per call (three for the sampler), chained with programmatic
// dependent launch:
//
//   records (sampler only), one warp per packed row: the row record (see
//     below), before the stream kernel.
//
//   stream, one CTA per (row, chunk of kChunkBytes): thread 0 issues one 1-D
//     TMA bulk copy of the chunk's 16-byte-aligned body into shared memory
//     (the row is read from HBM exactly once; unaligned head / tail
//     elements use plain loads); many short CTAs per SM keep the copies in
//     flight and hide each other's latencies.  While the copy is in flight,
//     warp 0 computes the row record (the sampler's CTAs of later chunks
//     copy it from the records kernel): the owner request (32-way
//     search of cu_rows), the row's position and validity and the owner's
//     parameters; with a confidence margin also whether the margin applies
//     (position, generated-token count, a warp scan of the protected ids)
//     and the draft's logit (NaN if not).  Outside the sampler the row's
//     first chunk stores the record for the finish.  Pass 1 takes two loops
//     over the thread's 16-byte vectors: the maximum and the first vector holding
//     it (selects only), then sum exp(z - max) against it (packed f32x2
//     arithmetic for bf16) and, for relaxed top-K, the count of logits above
//     the draft's; warp reductions (redux.sync) and a CTA reduction give the
//     chunk summary.  Sampler rows (T > 0) add, by filter:
//       no filter   - the chunk's Gumbel-max winner (vectors that cannot beat
//                     a lower bound from the thread maxima are skipped, and so
//                     are the logarithms of elements whose uniform cannot
//                     reach the running best);
//       top-k/min-p - a record of the 256 thread slices: each one's maximum,
//                     second largest element and the maximum's offset (bf16
//                     values as 16 bits); the survivors form an upper set
//                     {z >= th}, and the finish bounds th from below with the
//                     maxima (at least k thread maxima, hence k elements,
//                     reach the k-th largest maximum) and reads back only the
//                     slices whose second largest element reaches the bound;
//       top-p alone - bf16: counts of the kTopBins bf16 values at and below
//                     the chunk maximum, the chunk's mass at temperature T,
//                     and the elements whose Gumbel score reaches that of the
//                     chunk's first maximum; fp32: the record above and the
//                     chunk's mass.
//     The logits are copied with an L2 evict-first hint: they are read once,
//     and the summaries the finish reads back stay in L2.
//     Only plain stores: nothing in this kernel waits for another CTA.
//
//   finish, one CTA per row (extra CTAs write the outputs of requests
//     without a valid row range): combine the chunk summaries and settle the
//     row's token: the best chunk score (no filter); a scan of the merged
//     value counts from the top value to the nucleus boundary, then the best
//     score at or above it (bf16 top-p alone); or, for top-k / min-p (and
//     fp32 top-p alone), the row's chunk records bulk-copied on chip with
//     its first loads, the elements at or above the bound gathered from them
//     (and from the few slices read back), radix selects over them (exact
//     k-th largest value, exact top-p crossing by mass, or per-value tallies
//     for a narrow bf16 set) and Gumbel-max over the survivors.  A row the
//     summaries cannot settle (a nucleus reaching below every chunk's
//     counted values, a list overflow) takes exact selects over the whole
//     row, streamed again through the same CTA's shared memory.  The CTA
//     finishing the last row of a request (atomic ticket) runs the
//     accept-while-equal prefix scan with one warp ballot and writes the
//     request's tokens and the optional prefix-acceptance counters.
//
// Definitions: xLLM docs "自适应投机推理" §"启动示例" (ragged rejection
// sampler with packed-row owners, point-mass draft, replacement / bonus,
// temperature 0 = greedy, ordinary top-k/top-p/min-p semantics),
// §"基于 MTP logits 的自适应 target 验证" (exp(selected - logsumexp)),
// "vllm-hust-vSpec" README §"EAGLE 功能" (strict top-1 and relaxed top-K
// acceptance with a strict prefix, no per-request host sync, the active
// vocabulary with a full token-id map), §"启动" and §"通用参数" (the
// confidence margin and its position, token-count and protected-id options).
#include <algorithm>

#include "rowkit.cuh"

namespace specv {

constexpr int kTopBins = 256;       // bf16 top-p alone: values counted at and below the chunk max
constexpr int kFrontCap = 384;      // bf16 top-p alone: listed elements per chunk
// bf16 top-p alone: Philox blocks a warp may queue (two per 16-byte vector
// of its share of a chunk), and the stream kernel's queue area after Shared
constexpr int kQueuePerWarp = 2 * (kChunkBytes / 16) / kWarps;
constexpr int kQueueBytes = kWarps * kQueuePerWarp * static_cast<int>(sizeof(uint16_t));
constexpr int kFinScratch = 20 * 1024;   // finish kernel: candidates or counts (6 CTAs per SM)

static_assert(5 * (kChunkBytes + sizeof(Shared) + kQueueBytes + 1024) <= 228 * 1024,
              "five bf16 sampler stream CTAs fit an SM's shared memory");

// Element listed by a bf16 top-p-alone chunk: its Gumbel score reaches the
// score of the chunk's first maximum.  8 bytes: the score, then the bf16
// value's bits above the element's offset in its chunk.
struct __align__(8) Front {
    float s;
    uint32_t vo;
};
static_assert(kChunkBytes / 2 <= 65536, "a bf16 chunk offset fits 16 bits");
// a chunk's candidate area holds its listed elements then its value counts
// (bf16 top-p alone), or its record (other filtered rows)
static_assert(kFrontCap * sizeof(Front) + kTopBins * sizeof(uint16_t) <= kCandCap * sizeof(Cand),
              "listed elements and counts fit a chunk's candidate area");
static_assert(kThreads * (2 * sizeof(float) + sizeof(uint16_t)) <= kCandCap * sizeof(Cand),
              "thread maxima, second values and offsets fit");
// the finish stages gathered candidates, then the survivors' tallies
static_assert(kListCap * sizeof(Cand) + kTally * (sizeof(uint32_t) + sizeof(uint64_t)) <= kFinScratch,
              "gathered candidates and tallies fit the finish scratch");
// bf16 top-p alone stages every chunk's counts (longer rows take the exact path)
constexpr int kCountChunks = static_cast<int>(kFinScratch / (kTopBins * sizeof(uint16_t)));

// Record of a top-k / min-p (and fp32 top-p alone) chunk, at the start of
// its candidate area: per thread slot its maximum, its second largest
// element (both in the input type: bf16 bits for bf16 rows) and the
// maximum's offset in the chunk.  The finish copies every chunk's record of
// its row into shared memory with one bulk copy each.
template <typename E>
struct Rec {
    static constexpr int BYTES = kThreads * (2 * E::BYTES + 2);
    static __device__ __forceinline__ float max(const uint8_t *r, int t) { return val(r, t); }
    static __device__ __forceinline__ float sec(const uint8_t *r, int t) { return val(r, kThreads + t); }
    static __device__ __forceinline__ uint16_t off(const uint8_t *r, int t)
    {
        return reinterpret_cast<const uint16_t *>(r + 2 * kThreads * E::BYTES)[t];
    }
    static __device__ __forceinline__ void put(uint8_t *r, int t, float mx, float sc, uint16_t o)
    {
        if constexpr (E::BYTES == 2) {
            reinterpret_cast<uint16_t *>(r)[t] = static_cast<uint16_t>(__float_as_uint(mx) >> 16);
            reinterpret_cast<uint16_t *>(r)[kThreads + t] = static_cast<uint16_t>(__float_as_uint(sc) >> 16);
        } else {
            reinterpret_cast<float *>(r)[t] = mx;
            reinterpret_cast<float *>(r)[kThreads + t] = sc;
        }
        reinterpret_cast<uint16_t *>(r + 2 * kThreads * E::BYTES)[t] = o;
    }
  private:
    static __device__ __forceinline__ float val(const uint8_t *r, int i)
    {
        if constexpr (E::BYTES == 2)
            return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(r)[i]) << 16);
        else
            return reinterpret_cast<const float *>(r)[i];
    }
};
static_assert(Rec<Elt<float>>::BYTES <= kCandCap * sizeof(Cand), "a record fits a chunk's candidate area");
static_assert(Rec<Elt<uint16_t>>::BYTES % 16 == 0 && Rec<Elt<float>>::BYTES % 16 == 0,
              "records are whole 16-byte units (bulk copies)");

// ------------------------------------------------- sampler records -----
// Sampler only: one warp per packed row writes its row record (row_record)
// for the stream CTAs of later chunks and for the finish.
// (The other modes' stream CTAs all compute their own record while their
// copy is in flight; for the sampler, with its parameter loads, that costs
// its later CTAs more than this launch, while its first-chunk CTAs, whose
// copies take long anyway in the first wave, would otherwise wait for it.)
template <typename TIn>
__global__ void __launch_bounds__(256) sample_records_kernel(const VerifyParams p)
{
    // Launched as a programmatic dependent of whatever kernel precedes the
    // call (the previous call's finish, say), so its CTAs are resident when
    // that one ends.  Nothing is read before that kernel has completed, and
    // the stream kernel is released only then: its chunk copies (and its
    // first chunks' own row records) read the call's inputs without waiting
    // for this kernel.
    griddep_wait();
    griddep_launch_dependents();
    const int r = (blockIdx.x * 256 + threadIdx.x) >> 5;
    if (r >= p.R_cap) return;
    const RowInfo inf = row_record<TIn, MODE_SAMPLE>(p, r);
    if ((threadIdx.x & 31) == 0) reinterpret_cast<RowInfo *>(p.ws_info)[r] = inf;
}

// Mass of the staged chunk at temperature T: sum exp((z - m_c) / T) over
// this thread's vectors (packed f32x2 arithmetic for bf16).
template <typename E>
__device__ __forceinline__ float chunk_mass(const uint4 *body, int nb, float m_c, float sc)
{
    const float c0 = -m_c * sc;
    if constexpr (E::BYTES == 2) {
        uint64_t acc = f2_pack(0.f, 0.f);
        const uint64_t s2 = f2_pack(sc, sc), c2 = f2_pack(c0, c0);
#pragma unroll 4
        for (int i = threadIdx.x; i < nb; i += kThreads) {
            const uint4 v = body[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float e0, e1;
                f2_unpack(f2_fma(f2_pack(bf_lo(w[j]), bf_hi(w[j])), s2, c2), e0, e1);
                acc = f2_add(acc, f2_pack(ex2(e0), ex2(e1)));
            }
        }
        float a, b;
        f2_unpack(acc, a, b);
        return a + b;
    } else {
        float a = 0.f, b = 0.f;
        for (int i = threadIdx.x; i < nb; i += kThreads) {
            float x[4];
            E::unpack(body[i], x);
            a += ex2(fmaf(x[0], sc, c0)) + ex2(fmaf(x[2], sc, c0));
            b += ex2(fmaf(x[1], sc, c0)) + ex2(fmaf(x[3], sc, c0));
        }
        return a + b;
    }
}

// bf16 top-p alone, one chunk.  Counts of the kTopBins bf16 values at and
// below the chunk maximum (bin = key(max) - key(z)), the chunk's mass at
// temperature T, and a list of the elements of the counted range whose
// Gumbel score reaches the score s_top of the chunk's first maximum (the
// higher score, lower index on equal scores).  Every other element of the
// range scores below an element with a value at least its own, so when the
// nucleus threshold lies in the range the row's winner is a listed element
// or some chunk's first maximum.  An element can reach s_top only if
// -log u <= D = exp(z/T - s_top); as -log u >= 1 - u, a lattice uniform with
// 1 - u > D cannot, so its logarithms are skipped (one lattice step of
// margin for the rounding of D).  Writes the listed elements and the counts
// to the chunk's candidate area; sets sh.part.g / w / ncand.
template <typename E>
__device__ void summary_top_p_bf16(const VerifyParams &p, const uint4 *body, const ChunkGeom &g,
                                   const Filter &f, const Noise &nz, int64_t rc, Shared &sh)
{
    uint32_t *tally = sh.hist;             // [kTopBins] per-value counts
    const int tid = threadIdx.x;
    const float m_c = sh.part.m;
    const int32_t a_c = sh.part.amax;
    const uint32_t ktop = fkey(m_c) >> 16;
    const uint32_t kbot = (ktop >= static_cast<uint32_t>(kTopBins - 1)) ? ktop - (kTopBins - 1) : 0u;
    const float zbot = key16_value(kbot);
    for (int i = tid; i < kTopBins; i += kThreads) tally[i] = 0u;
    if (tid == 0) {
        sh.cand_n = 0;
        const uint4 w = nz.block(static_cast<uint32_t>(a_c) >> 2);
        sh.part.g = fmaf(m_c, f.invT, gumbel_of(word_of(w, static_cast<uint32_t>(a_c) & 3u)));
    }
    float mass = 0.f;
    if (f.T != 1.0f) mass = chunk_mass<E>(body, g.nb, m_c, f.sc);
    csync();
    const float s_top = sh.part.g;
    Front *fl = reinterpret_cast<Front *>(reinterpret_cast<Cand *>(p.ws_cand) + rc * kCandCap);
    auto list = [&](float v, int32_t ix, float s) {
        if (s > s_top || (s == s_top && ix < a_c)) {
            const int slot = warp_append(&sh.cand_n);
            if (slot < kFrontCap)
                fl[slot] = Front{s, (__float_as_uint(v) & 0xFFFF0000u) | static_cast<uint32_t>(ix - g.e0)};
        }
    };
    auto count = [&](float v) {
        if (v >= zbot) atomicAdd(&tally[ktop - (fkey(v) >> 16)], 1u);
    };
    // the head and tail elements first (plain loads, staged by the kernel)
    if (tid < g.n_extra) {
        const float xv = sh.extras_v[tid];
        const int32_t ix = sh.extras_i[tid];
        if (f.T != 1.0f) mass += ex2((xv - m_c) * f.sc);
        count(xv);
        if (xv >= zbot) list(xv, ix, nz.score(xv, ix, f.invT));
    }
    if ((g.a0 & 3) == 0) {
        // The body covers whole Philox blocks.  Pass A queues, per warp, the
        // blocks with an element in the counted range (about half of them):
        // some lane of a warp nearly always has one, so a lane-by-lane pass
        // would visit every block.  Pass B takes only the queued blocks,
        // packed by ballots: it counts their elements in the range and, if
        // the block's maximum can reach s_top with the largest noise, draws
        // its noise and lists the elements that reach it.
        const int lane = tid & 31;
        const unsigned lt = (1u << lane) - 1u;
        uint16_t *wq = reinterpret_cast<uint16_t *>(&sh + 1) + (tid >> 5) * kQueuePerWarp;
        int nq = 0;
        for (int i0 = tid - lane; i0 < g.nb; i0 += kThreads) {
            const int i = i0 + lane;
            bool q0 = false, q1 = false;
            if (i < g.nb) {
                const uint4 v = body[i];
                const uint32_t w0 = max_bf16x2(v.x, v.y), w1 = max_bf16x2(v.z, v.w);
                q0 = fmaxf(bf_lo(w0), bf_hi(w0)) >= zbot;
                q1 = fmaxf(bf_lo(w1), bf_hi(w1)) >= zbot;
            }
            const unsigned m0 = __ballot_sync(0xFFFFFFFFu, q0), m1 = __ballot_sync(0xFFFFFFFFu, q1);
            if (q0) wq[nq + __popc(m0 & lt)] = static_cast<uint16_t>(2 * i);
            nq += __popc(m0);
            if (q1) wq[nq + __popc(m1 & lt)] = static_cast<uint16_t>(2 * i + 1);
            nq += __popc(m1);
        }
        __syncwarp();
        const uint2 *halves = reinterpret_cast<const uint2 *>(body);
        const uint32_t ctr0 = static_cast<uint32_t>(g.a0) >> 2;
        for (int e = lane; e < nq; e += 32) {
            const uint32_t blk = wq[e];
            const uint2 u = halves[blk];
            const float x[4] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y)};
#pragma unroll
            for (int j = 0; j < 4; ++j) count(x[j]);
            const float bm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            // no element of the block can reach s_top (the noise is bounded)
            if (fmaf(bm, f.invT, kGumbelMax) < s_top) continue;
            const float D = ex2((bm * f.invT - s_top) * kLog2e);
            const float t = fmaf(-D, 16777216.f, 16777215.f) * 0.5f;
            const uint32_t kthr = (t >= 2.f) ? static_cast<uint32_t>(t) - 1u : 0u;
            const uint32_t wthr = kthr << 9;      // (w >> 9) >= kthr <=> w >= kthr << 9
            const uint4 w = nz.block(ctr0 + blk);
            if (max(max(w.x, w.y), max(w.z, w.w)) < wthr) continue;
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            const int32_t base = g.a0 + 4 * static_cast<int32_t>(blk);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (x[j] >= zbot && ws[j] >= wthr) list(x[j], base + j, fmaf(x[j], f.invT, gumbel_of(ws[j])));
        }
    } else {
        for (int i = tid; i < g.nb; i += kThreads) {
            const uint4 v = body[i];
            const float vm = E::vmax(v);
            if (!(vm >= zbot)) continue;
            float x[8];
            E::unpack(v, x);
#pragma unroll
            for (int q = 0; q < 8; ++q) count(x[q]);
            // no element of the vector can reach s_top (the noise is bounded)
            if (fmaf(vm, f.invT, kGumbelMax) < s_top) continue;
            const int32_t base = g.a0 + i * 8;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (x[q] >= zbot) list(x[q], base + q, nz.score(x[q], base + q, f.invT));
        }
    }
    if (f.T != 1.0f) mass = block_sum(mass, sh);
    else csync();
    uint16_t *tl = reinterpret_cast<uint16_t *>(fl + kFrontCap);
    for (int i = tid; i < kTopBins; i += kThreads) tl[i] = static_cast<uint16_t>(tally[i]);
    if (tid == 0) {
        sh.part.w = (f.T != 1.0f) ? mass : sh.part.s;
        sh.part.ncand = sh.cand_n;
    }
}

// Sampler summary of one chunk (T > 0), after pass 1 (sh.part holds the
// chunk's max, first argmax and sum).
template <typename E>
__device__ void summary_sampler(const VerifyParams &p, const RowInfo &info, const uint4 *body,
                                const ChunkGeom &g, float thread_max, int32_t thread_arg,
                                float thread_sec, int64_t rc, Shared &sh)
{
    constexpr int VEC = E::VEC;
    const int tid = threadIdx.x;
    const float m_c = sh.part.m;
    // top-k / min-p (and fp32 top-p alone), the commonest filtered rows,
    // first: they need neither 1/T nor the row's noise key
    const bool use_k = info.top_k > 0 && info.top_k < p.V, use_m = info.min_p > 0.f;
    if (use_k || use_m || (E::BYTES == 4 && info.top_p < 1.f)) {
        // per thread slot (the thread's elements of the chunk, extras
        // included) its maximum, its second largest element and the
        // maximum's offset in the chunk; for fp32 top-p alone also the
        // chunk's mass at temperature T
        Rec<E>::put(reinterpret_cast<uint8_t *>(reinterpret_cast<Cand *>(p.ws_cand) + rc * kCandCap), tid,
                    thread_max, thread_sec,
                    static_cast<uint16_t>(thread_max > -INFINITY ? thread_arg - g.e0 : 0));
        if (!use_k && !use_m && m_c > -INFINITY) {
            const Filter f(info, p.V);
            const float T = f.T;
            float mass = (T != 1.0f) ? chunk_mass<E>(body, g.nb, m_c, f.sc) : 0.f;
            if (T != 1.0f && tid < g.n_extra) mass += ex2((sh.extras_v[tid] - m_c) * f.sc);
            if (T != 1.0f) mass = block_sum(mass, sh);
            if (tid == 0) sh.part.w = (T != 1.0f) ? mass : sh.part.s;
        }
        return;
    }
    const Filter f(info, p.V);
    const float T = f.T, invT = f.invT;
    const Noise nz{static_cast<uint32_t>(info.pos), info.rid, p.step, info.seed_lo, info.seed_hi};
    if (f.unfiltered) {
        if (!(m_c > -INFINITY)) return;        // only -inf here: nothing to draw from
        // lower bound of the chunk's best score from the thread maxima; a
        // vector whose max z has z/T + kGumbelMax below it cannot win
        float best = -INFINITY;
        int32_t bi = INT_MAX;
        if (thread_max > -INFINITY) { best = nz.score(thread_max, thread_arg, invT); bi = thread_arg; }
        block_best(best, bi, sh);
        const float skip = (best - kGumbelMax) * T;
        const bool whole_blocks = (g.a0 & 3) == 0;
        for (int i = tid; i < g.nb; i += kThreads) {
            const uint4 v = body[i];
            const float vm = E::vmax(v);
            if (!(vm >= skip)) continue;
            const int32_t base = g.a0 + i * VEC;
            if (whole_blocks) {
                score_vec<E>(v, vm, base, invT, nz, best, bi);
            } else {
                float x[VEC];
                E::unpack(v, x);
#pragma unroll
                for (int q = 0; q < VEC; ++q) keep_best(nz.score(x[q], base + q, invT), base + q, best, bi);
            }
        }
        if (tid < g.n_extra)
            keep_best(nz.score(sh.extras_v[tid], sh.extras_i[tid], invT), sh.extras_i[tid], best, bi);
        block_best(best, bi, sh);
        if (tid == 0) { sh.part.g = best; sh.part.aux = bi; }
        return;
    }
    // bf16 top-p alone (the only case left)
    if constexpr (E::BYTES == 2)
        if (m_c > -INFINITY) summary_top_p_bf16<E>(p, body, g, f, nz, rc, sh);
}

// ------------------------------------------------------ stream kernel ----

// One CTA per (row, chunk); plain stores of the chunk summary only.  Many
// short CTAs per SM keep the bulk copies in flight.
template <typename TIn, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == MODE_SAMPLE ? 5 : 6)
    stream_chunks_kernel(const VerifyParams p)
{
    using E = Elt<TIn>;
    constexpr bool HAS_INFO = (MODE != MODE_CONF);
    extern __shared__ __align__(128) uint8_t smem[];
    const uint4 *body = reinterpret_cast<const uint4 *>(smem);
    Shared &sh = *reinterpret_cast<Shared *>(smem + kChunkBytes);

    const int tid = threadIdx.x;
    const int nchunk = p.nchunk;
    // the finish kernel's CTAs may become resident once every CTA of this
    // grid has started (they wait for its completion before reading)
    griddep_launch_dependents();
    // The sampler takes chunk-major order: a chunk's cost depends on its
    // row's filters, and this spreads every row's chunks evenly over the
    // grid, with the short tail chunks in the last wave.  So does the
    // confidence, whose grid is little more than one wave: its last CTAs are
    // then short tail chunks.  The other modes keep row-major order.  The
    // grid is two-dimensional with the faster index in x (chunk-major: x =
    // row, y = chunk; else x = chunk, y = row), so the order comes without
    // divisions; row-major grids of more than 65535 rows are one-dimensional.
    int r, c;
    if (MODE == MODE_SAMPLE || MODE == MODE_CONF) {
        r = static_cast<int>(blockIdx.x);
        c = static_cast<int>(blockIdx.y);
    } else if (gridDim.y > 1 || gridDim.x == static_cast<unsigned>(nchunk)) {
        c = static_cast<int>(blockIdx.x);
        r = static_cast<int>(blockIdx.y);
    } else {
        r = static_cast<int>(blockIdx.x) / nchunk;
        c = static_cast<int>(blockIdx.x) - r * nchunk;
    }
    const TIn *row = reinterpret_cast<const TIn *>(p.logits) + static_cast<int64_t>(r) * p.ld;
    const ChunkGeom g = chunk_geom<E>(row, c, p.V);
    // The sampler's first-chunk CTAs (chunk-major order puts them in the
    // grid's first wave) compute their row's record themselves while their
    // copy is in flight: the records kernel runs beside them, its loads
    // queued behind their copies, and waiting for it would hold the whole
    // first wave.  Later CTAs copy the record it wrote.  (Every CTA reads
    // only the call's inputs, visible since the records kernel, whose
    // launch released this grid, waited for the kernel before the call.)
    const bool own_rec = MODE == MODE_SAMPLE && c == 0;

    if (tid == 0) {
        // The logits buffer holds R_cap rows, so the chunk copy is issued
        // before anything else (in bounds even for rows past cu_rows[B]).
        sh.timeout = 0;
        mbar_init(&sh.mbar[0], 1);
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(g.nb) * 16u;
        mbar_arrive_expect_tx(&sh.mbar[0], bytes + ((MODE == MODE_SAMPLE && !own_rec) ? 64u : 0u));
        // (with no body and no record the arrival alone completes the phase)
        if (bytes) bulk_g2s_stream(smem, row + g.a0, bytes, &sh.mbar[0]);
        int32_t R = p.n_rows;
        if (MODE != MODE_CONF) R = __ldg(p.cu_rows + p.B);
        if (MODE == MODE_SAMPLE && !own_rec) {
            griddep_wait();                 // the sampler's row records
            bulk_g2s(&sh.info, reinterpret_cast<const RowInfo *>(p.ws_info) + r, 64u, &sh.mbar[0]);
        }
        if (!HAS_INFO) {
            RowInfo inf = {};
            inf.b = r; inf.valid = 1;
            sh.info = inf;
        }
        sh.R = min(R, p.R_cap);
    }
    if (HAS_INFO && (MODE != MODE_SAMPLE || own_rec) && tid < 32) {
        // the row record (owner request, position, parameters) while the
        // copy is in flight; outside the sampler the row's first chunk
        // stores it for the finish (the sampler's records kernel does)
        const RowInfo inf = row_record<TIn, MODE>(p, r);
        if (tid == 0) {
            sh.info = inf;
            if (MODE != MODE_SAMPLE && c == 0) reinterpret_cast<RowInfo *>(p.ws_info)[r] = inf;
        }
    }
    float xe = -INFINITY;
    int32_t ie = INT_MAX;
    if (tid < g.n_extra) {
        ie = (tid < g.n_head) ? g.e0 + tid : g.a1 + (tid - g.n_head);
        xe = E::load(row, ie);
        sh.extras_v[tid] = xe;
        sh.extras_i[tid] = ie;
    }
    csync();
    if (tid == 0 && !mbar_wait(&sh.mbar[0], 0)) {
        // the copy did not land in time: report it, give the copy one more
        // bounded wait, and leave without touching the buffer
        set_status(p.status, SPEC_STATUS_TIMEOUT);
        mbar_wait(&sh.mbar[0], 0);
        sh.timeout = 1;
    }
    csync();
    if (sh.timeout || r >= sh.R) return;
    const RowInfo &info = sh.info;
    if (!info.valid) return;

    // ---------------------------------------------------------- pass 1 --
    // the sum also serves as the chunk mass of a top-p-alone row at T = 1
    const bool need_sum = (MODE == MODE_CONF) || (p.row_lse != nullptr) ||
                          (MODE == MODE_SAMPLE && info.T == 1.0f && info.top_p < 1.f &&
                           !(info.top_k > 0 && info.top_k < p.V) && !(info.min_p > 0.f));
    const float zd = info.zd;
    float tmax = -INFINITY, tsum = 0.f, tsec = -INFINITY;
    int32_t targ = INT_MAX, tcnt = 0;
    // sampler rows bounded by top-k / min-p (and fp32 top-p alone) keep each
    // thread's two largest elements
    const bool top2 = MODE == MODE_SAMPLE && info.T > 0.f &&
                      ((info.top_k > 0 && info.top_k < p.V) || info.min_p > 0.f ||
                       (E::BYTES == 4 && info.top_p < 1.f));
    if (MODE == MODE_SAMPLE && top2) {
        if (need_sum) tmax = pass1<E, MODE, true, true>(body, g.nb, g.a0, zd, targ, tsum, tcnt, &tsec);
        else tmax = pass1<E, MODE, false, true>(body, g.nb, g.a0, zd, targ, tsum, tcnt, &tsec);
    } else {
        if (need_sum) tmax = pass1<E, MODE, true>(body, g.nb, g.a0, zd, targ, tsum, tcnt);
        else tmax = pass1<E, MODE, false>(body, g.nb, g.a0, zd, targ, tsum, tcnt);
    }
    if (tid < g.n_extra) {
        tsec = fmaxf(tsec, fminf(xe, tmax));
        combine(tmax, targ, tsum, tcnt, xe, ie, 1.f, (MODE == MODE_RELAXED && xe > zd) ? 1 : 0,
                need_sum);
    }
    const float thread_max = tmax;
    const int32_t thread_arg = targ;
    chunk_reduce<MODE>(tmax, targ, tsum, tcnt, need_sum, sh);

    const int64_t rc = static_cast<int64_t>(r) * nchunk + c;
    // (the summary's fields of sh.part are written by thread 0, the thread
    // that stores the part: no barrier before the store)
    if (MODE == MODE_SAMPLE && info.T > 0.f)
        summary_sampler<E>(p, info, body, g, thread_max, thread_arg, tsec, rc, sh);
    if (tid == 0) reinterpret_cast<ChunkPart *>(p.ws_part)[rc] = sh.part;
}

// ------------------------------------------------------- row finish -----

// Best score among the row's chunk first maxima and listed elements with a
// value at or above zF (bf16 top-p alone), lowest index on equal scores.
// The lists are read as one flat array (offsets from a warp scan of their
// lengths, in sh.offs), so the loads of every chunk go out together.
__device__ __forceinline__ void best_of_front(const VerifyParams &p, const ChunkPart *parts,
                                              int nchunk, int64_t r, float zF, Shared &sh,
                                              float &best, int32_t &bi)
{
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 32) {
        int tot = 0;
        for (int q0 = 0; q0 < nchunk; q0 += 32) {
            const int q = q0 + lane;
            const int nq = (q < nchunk && parts[q].m > -INFINITY) ? min(parts[q].ncand, kFrontCap) : 0;
            int incl = nq;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            if (q < nchunk) sh.offs[q] = tot + incl - nq;
            tot += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) sh.offs[nchunk] = tot;
    }
    csync();
    for (int q = tid; q < nchunk; q += kThreads)
        if (parts[q].m > -INFINITY && parts[q].m >= zF) keep_best(parts[q].g, parts[q].amax, best, bi);
    const int n = sh.offs[nchunk];
    constexpr int PER = 4;
    for (int e0 = 0; e0 < n; e0 += PER * kThreads) {
        uint2 v[PER];
        int32_t base[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = e0 + tid + u * kThreads;
            base[u] = -1;
            if (e < n) {
                int q = 0;
                while (sh.offs[q + 1] <= e) ++q;
                const uint2 *fl = reinterpret_cast<const uint2 *>(
                    reinterpret_cast<const Cand *>(p.ws_cand) + (r * nchunk + q) * kCandCap);
                v[u] = __ldcg(fl + (e - sh.offs[q]));
                base[u] = q * (kChunkBytes / 2);
            }
        }
#pragma unroll
        for (int u = 0; u < PER; ++u)
            if (base[u] >= 0 && __uint_as_float(v[u].y & 0xFFFF0000u) >= zF)
                keep_best(__uint_as_float(v[u].x), base[u] + static_cast<int32_t>(v[u].y & 0xFFFFu), best, bi);
    }
}

// bf16 top-p alone, at the row's finish: merge the chunks' value counts over
// the keys every chunk counted ([kcert, key(M)]), scan their mass from the
// top value (equal values share one weight) to the group where it first
// reaches top_p * W, and take the best score at or above that value.  False
// when a list overflowed or the counted values do not hold the target mass
// (the nucleus reaches below them).
__device__ bool finish_top_p_bf16(const VerifyParams &p, const RowInfo &info, const ChunkPart *parts,
                                  int nchunk, int64_t r, float M, uint16_t *tl, Shared &sh,
                                  float &best, int32_t &bi)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Filter f(info, p.V);
    const uint32_t KT = fkey(M) >> 16;
    if (nchunk > kCountChunks) return false;
    if (warp == 0) {
        float w = 0.f;
        uint32_t kc = 0u;
        int ovf = 0;
        for (int q0 = 0; q0 < nchunk; q0 += 32) {
            const int q = q0 + lane;
            const bool on = q < nchunk && parts[q].m > -INFINITY;
            float wq = on ? parts[q].w * ex2((parts[q].m - M) * f.sc) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wq += __shfl_xor_sync(0xFFFFFFFFu, wq, o);
            w += wq;
            uint32_t kb = 0u;
            if (on) {
                const uint32_t kt = fkey(parts[q].m) >> 16;
                kb = (kt >= static_cast<uint32_t>(kTopBins - 1)) ? kt - (kTopBins - 1) : 0u;
            }
            kc = max(kc, __reduce_max_sync(0xFFFFFFFFu, kb));
            ovf |= static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, (on && parts[q].ncand > kFrontCap) ? 1u : 0u));
        }
        if (lane == 0) {
            sh.W = w;
            sh.lkey = kc;
            sh.overflow = ovf;
        }
    }
    // stage every chunk's counts (kTopBins 16-bit counts each)
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.ws_cand);
        constexpr int PER = kTopBins * 2 / 16;            // 16-byte vectors per chunk's counts
        const int64_t stride = static_cast<int64_t>(kCandCap) * sizeof(Cand) / 16;
        constexpr int64_t off = static_cast<int64_t>(kFrontCap) * sizeof(Front) / 16;
        static_assert(kFrontCap * sizeof(Front) % 16 == 0, "counts start on a 16-byte boundary");
        for (int i = tid; i < nchunk * PER; i += kThreads) {
            const int q = i / PER, u = i - q * PER;
            reinterpret_cast<uint4 *>(tl)[i] = __ldcg(src + (r * nchunk + q) * stride + off + u);
        }
    }
    csync();
    if (sh.overflow) return false;
    const float target = info.top_p * sh.W;
    const uint32_t kc = sh.lkey;
    // thread t: the merged count of key KT - t, as a mass, in hist[255 - t]
    float wt = 0.f;
    const uint32_t k = KT - static_cast<uint32_t>(tid);
    if (tid < kTopBins && KT >= static_cast<uint32_t>(tid) && k >= kc) {
        uint32_t c = 0;
        for (int q = 0; q < nchunk; ++q) {
            if (!(parts[q].m > -INFINITY)) continue;
            const uint32_t d = (fkey(parts[q].m) >> 16) - k;     // wraps when the chunk max is below k
            if (d < static_cast<uint32_t>(kTopBins)) c += tl[q * kTopBins + d];
        }
        if (c) wt = static_cast<float>(c) * ex2((key16_value(k) - M) * f.sc);
    }
    float *hist = reinterpret_cast<float *>(sh.hist);
    static_assert(kTopBins == 256 && kThreads == 256, "one counted value per thread");
    hist[255 - tid] = wt;
    const float tot = block_sum(wt, sh);
    if (!(tot >= target * (1.f + kMassTol))) return false;
    find_crossing<float>(hist, target, sh);
    const int t_star = 255 - sh.sel_bin;
    const float zF = key16_value(KT - static_cast<uint32_t>(t_star));
    best_of_front(p, parts, nchunk, r, zF, sh, best, bi);
    block_best(best, bi, sh);
    (void)lane;
    return true;
}

// Every element of row r with a value at or above L, into lst (count in
// sh.cand_n; above cap the list is incomplete).  A thread slot (chunk q,
// thread t) whose maximum (from the records staged in recs) reaches L
// contributes that maximum; the few slots whose second largest element
// reaches L as well are collected into a flat list in shared memory and read
// back whole, four 16-byte vectors per thread loaded before any is used, so
// their loads go out in one batch.  Head / tail elements of a slot come with
// its first vector.
template <typename E, typename TIn>
__device__ void gather_above(const VerifyParams &p, const TIn *row, float L, const uint8_t *recs,
                             Cand *lst, int cap, int *slots, int slot_cap, Shared &sh)
{
    constexpr int VEC = E::VEC;
    constexpr int PER = kChunkBytes / 16 / kThreads;       // vectors of a thread slot
    const int tid = threadIdx.x;
    const int nchunk = p.nchunk;
    if (tid == 0) { sh.cand_n = 0; sh.total = 0; }
    csync();
    auto add = [&](float v, int32_t ix) {
        const int slot = warp_append(&sh.cand_n);
        if (slot < cap) { lst[slot].v = v; lst[slot].i = ix; }
    };
    constexpr int CE = kChunkBytes / E::BYTES;
    for (int q = 0; q < nchunk; ++q) {
        const uint8_t *rq = recs + q * Rec<E>::BYTES;
        const float m = Rec<E>::max(rq, tid);
        if (!(m >= L)) continue;
        if (Rec<E>::sec(rq, tid) >= L) {
            const int k = warp_append(&sh.total);
            if (k < slot_cap) slots[k] = q * kThreads + tid;
        } else {
            add(m, q * CE + static_cast<int32_t>(Rec<E>::off(rq, tid)));
        }
    }
    csync();
    const int ns = sh.total;
    if (ns > slot_cap) {                 // far too many: the caller falls back
        if (tid == 0) sh.cand_n = cap + 1;
        csync();
        return;
    }
    // the listed slots' vectors, four per thread loaded before any is used
    for (int e0 = 0; e0 < ns * PER; e0 += 4 * kThreads) {
        uint4 v[4];
        int32_t ix0[4], ixe[4];
        float xe[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads + tid;
            ix0[u] = -1;
            ixe[u] = -1;
            if (e < ns * PER) {
                const int sl = slots[e / PER], j = e - (e / PER) * PER;
                const int q = sl / kThreads, t = sl - q * kThreads;
                const ChunkGeom g = chunk_geom<E>(row, q, p.V);
                const int i = t + j * kThreads;
                if (i < g.nb) {
                    v[u] = __ldcg(reinterpret_cast<const uint4 *>(row + g.a0) + i);
                    ix0[u] = g.a0 + i * VEC;
                }
                if (j == 0 && t < g.n_extra) {
                    ixe[u] = (t < g.n_head) ? g.e0 + t : g.a1 + (t - g.n_head);
                    xe[u] = E::load(row, ixe[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (ixe[u] >= 0 && xe[u] >= L) add(xe[u], ixe[u]);
            if (ix0[u] < 0 || !(E::vmax(v[u]) >= L)) continue;
            float x[VEC];
            E::unpack(v[u], x);
            for (int w = 0; w < VEC; ++w)
                if (x[w] >= L) add(x[w], ix0[u] + w);
        }
    }
    csync();
}

// The k-th largest of the row's thread maxima (counting equal ones; from
// the records staged in recs): at least k elements of the row reach it, so
// the row's top k values lie at or above it.
template <typename E>
__device__ float kth_maximum(const VerifyParams &p, const uint8_t *recs, int k, float M, Shared &sh)
{
    const int nchunk = p.nchunk;
    if (k > nchunk * kThreads) return -INFINITY;
    // one round over the 256 16-bit keys just below the row maximum's (bin
    // = distance from it, so the maxima spread over the bins instead of
    // piling into the one or two bins of a first radix digit): for bf16 the
    // crossing bin is the exact key; for fp32 its 16-bit floor, a lower bound
    // that serves as well
    const uint32_t top = fkey(M) >> 16;
    sh.hist[threadIdx.x] = 0u;
    csync();
    for (int q = 0; q < nchunk; ++q) {
        const uint32_t d = top - (fkey(Rec<E>::max(recs + q * Rec<E>::BYTES, threadIdx.x)) >> 16);
        if (d < 256u) atomicAdd(&sh.hist[255u - d], 1u);
    }
    csync();
    find_crossing<uint32_t>(sh.hist, static_cast<uint32_t>(k), sh);
    if (sh.sel_found) {
        const uint32_t key16 = top - (255u - static_cast<uint32_t>(sh.sel_bin));
        csync();
        return key_floor(key16 << 16);
    }
    csync();
    // the k-th largest lies further below: the general select
    auto visit = [&](auto &&fn, float thr) {
        for (int q = 0; q < nchunk; ++q) {
            const float v = Rec<E>::max(recs + q * Rec<E>::BYTES, threadIdx.x);
            if (v >= thr) fn(v, 0);
        }
    };
    const uint32_t key = select_key<E, false>(visit, 0u, fkey(M), 0.f, static_cast<uint32_t>(k), M,
                                              0.f, sh);
    return key_floor(key);
}

// ------------------------------------------------------ finish kernel ----

// One CTA per packed row, after the stream kernel: combine the chunk
// summaries, pick the row's token, write the row results, run the chain.
template <typename TIn, int MODE>
__global__ void __launch_bounds__(kThreads, 5) finish_rows_kernel(const VerifyParams p)
{
    using E = Elt<TIn>;
    extern __shared__ __align__(128) uint8_t smem[];
    Shared &sh = *reinterpret_cast<Shared *>(smem);
    ChunkPart *parts = reinterpret_cast<ChunkPart *>(smem + sizeof(Shared));     // [kMaxChunks]
    uint8_t *scratch = reinterpret_cast<uint8_t *>(parts + kMaxChunks);          // [kFinScratch]
    Cand *lst = reinterpret_cast<Cand *>(scratch);                              // [kListCap]
    uint8_t *recs = scratch + kFinScratch;                      // sampler: [nchunk] chunk records
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int nchunk = p.nchunk;

    // a following call's first kernel may become resident (it waits for
    // this grid's completion before it reads anything)
    griddep_launch_dependents();
    if (MODE != MODE_CONF && r >= p.R_cap) {
        // extra CTAs: the outputs of requests without a valid row range
        // (nothing of the stream kernel is read)
        bad_request_outputs(p, (r - p.R_cap) * kThreads + tid);
        return;
    }
    griddep_wait();                        // the stream kernel's stores are visible
    if (tid == 32) {
        // the row record, by another warp than the one issuing the copies
        // below (its loads would hold them back)
        if (MODE != MODE_CONF) {
            sh.info = reinterpret_cast<const RowInfo *>(p.ws_info)[r];
            sh.info.valid = sh.info.valid && r < min(__ldg(p.cu_rows + p.B), p.R_cap);
        } else {
            RowInfo inf = {};
            inf.b = r; inf.valid = 1;
            sh.info = inf;
        }
    }
    if (tid == 0) {
        sh.ph[0] = sh.ph[1] = 0u;
        sh.timeout = 0;
        mbar_init(&sh.mbar[0], 1);
        mbar_init(&sh.mbar[1], 1);
        fence_mbar_init();
        if (MODE == MODE_SAMPLE) {
            // every chunk's record, whatever the row's filters (it is not
            // known yet): the copies run with the loads below, and a
            // top-k / min-p row finds its records on chip
            const uint8_t *src = reinterpret_cast<const uint8_t *>(
                reinterpret_cast<const Cand *>(p.ws_cand) + static_cast<int64_t>(r) * nchunk * kCandCap);
            mbar_arrive_expect_tx(&sh.mbar[0], static_cast<uint32_t>(nchunk * Rec<E>::BYTES));
            for (int q = 0; q < nchunk; ++q)
                bulk_g2s(recs + q * Rec<E>::BYTES, src + static_cast<int64_t>(q) * kCandCap * sizeof(Cand),
                         Rec<E>::BYTES, &sh.mbar[0]);
        }
    }
    if (tid < nchunk) {
        const ChunkPart *rp = reinterpret_cast<const ChunkPart *>(p.ws_part) + static_cast<int64_t>(r) * nchunk;
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(rp + tid));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(rp + tid) + 1);
        ChunkPart cp;
        cp.m = a.x; cp.amax = __float_as_int(a.y); cp.s = a.z; cp.aux = __float_as_int(a.w);
        cp.g = b.x; cp.w = b.y; cp.ncand = __float_as_int(b.z); cp.lev = b.w;
        parts[tid] = cp;
    }
    if (MODE == MODE_SAMPLE && tid == 0) {
        if (!mbar_wait(&sh.mbar[0], 0)) {
            // the records did not land in time: reported; one more bounded
            // wait for the copies, and the row is not settled from them
            set_status(p.status, SPEC_STATUS_TIMEOUT);
            mbar_wait(&sh.mbar[0], 0);
            sh.timeout = 1;
        }
        sh.ph[0] = 1u;      // the row streaming below continues from phase 1
    }
    csync();
    const RowInfo &info = sh.info;
    if (!info.valid) return;
    const TIn *row = reinterpret_cast<const TIn *>(p.logits) + static_cast<int64_t>(r) * p.ld;
    const bool need_sum = (MODE == MODE_CONF) || (p.row_lse != nullptr);

    // combine the chunk summaries (warp 0): per lane its chunks, then the
    // warp's maximum, the lowest index attaining it, the rescaled sums and
    // the counts
    if (warp == 0) {
        float m = -INFINITY, s = 0.f;
        int32_t a = INT_MAX, cc = 0;
        for (int q = lane; q < nchunk; q += 32)
            combine(m, a, s, cc, parts[q].m, parts[q].amax, parts[q].s,
                    (MODE == MODE_RELAXED) ? parts[q].aux : 0, need_sum);
        const float mw = warp_max_f32(m);
        const int32_t aw = __reduce_min_sync(0xFFFFFFFFu, (m == mw) ? a : INT_MAX);
        float sw = 0.f;
        if (need_sum) {
            sw = (m > -INFINITY) ? s * ex2((m - mw) * kLog2e) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xFFFFFFFFu, sw, o);
        }
        const int32_t cw = __reduce_add_sync(0xFFFFFFFFu, cc);
        if (lane == 0) {
            sh.M = mw; sh.S = sw; sh.CNT = cw;
            sh.AMAX = (mw == -INFINITY) ? 0 : aw;
        }
    }
    csync();
    const float M = sh.M;
    const int32_t AMAX = sh.AMAX;
    int32_t y = AMAX;
    int32_t flag = 0;
    if (MODE == MODE_RELAXED)
        flag = (info.draft >= 0 && info.draft < p.V && sh.CNT < info.K) ? 1 : 0;
    // margin: the first argmax, or a gap max - z[d] (fp32) within the margin
    if (MODE == MODE_GREEDY && p.margin)
        flag = (info.draft == AMAX || M - info.zd <= __ldg(p.margin + info.b)) ? 1 : 0;

    if (MODE == MODE_SAMPLE && info.T > 0.f && M > -INFINITY) {
        const Filter f(info, p.V);
        const float T = f.T, sc = f.sc;
        const uint32_t keyM = fkey(M);
        const Noise nz{static_cast<uint32_t>(info.pos), info.rid, p.step, info.seed_lo, info.seed_hi};
        GumbelScorer gs{f.invT, nz, 0xFFFFFFFFu, make_uint4(0, 0, 0, 0)};
        float best = -INFINITY;
        int32_t bi = INT_MAX;
        auto score_all = [&](float v, int32_t ix) { keep_best(gs(v, ix), ix, best, bi); };
        bool whole = false;            // settle the row with exact selects over the whole row
        if (f.unfiltered) {
            for (int q = tid; q < nchunk; q += kThreads)
                if (parts[q].m > -INFINITY) keep_best(parts[q].g, parts[q].aux, best, bi);
            block_best(best, bi, sh);
        } else if (f.pure_p && E::BYTES == 2) {
            whole = !finish_top_p_bf16(p, info, parts, nchunk, r, M,
                                       reinterpret_cast<uint16_t *>(scratch), sh, best, bi);
        } else {
            // the bound every survivor reaches: the min-p threshold, the k-th
            // largest thread maximum (top-k), the 64-th (fp32 top-p alone)
            const float th_m = f.use_m ? M + T * logf(info.min_p) : -INFINITY;
            float L = th_m;
            const int kk = f.use_k ? info.top_k : (f.pure_p ? kPureListK : 0);
            if (kk > 0) L = fmaxf(L, kth_maximum<E>(p, recs, kk, M, sh));
            // the gathered slots' list shares the scratch with the
            // candidates: slots from the top, candidates from the bottom
            constexpr int kSlotCap = 1024;
            static_assert(kListCap * sizeof(Cand) + kSlotCap * sizeof(int) <= kFinScratch, "slots fit");
            gather_above<E, TIn>(p, row, L, recs, lst, kListCap,
                                 reinterpret_cast<int *>(scratch + kFinScratch) - kSlotCap, kSlotCap, sh);
            const int n_list = sh.timeout ? kListCap + 1 : sh.cand_n;
            auto visit_lst = [&](auto &&fn, float thr) {
                for (int i = tid; i < n_list; i += kThreads) {
                    const Cand e = lst[i];
                    if (e.v >= thr) fn(e.v, e.i);
                }
            };
            if (n_list > kListCap) {
                whole = true;
            } else if (f.pure_p) {
                // fp32 top-p alone: every value at or above L is listed; when
                // they hold the target mass the nucleus lies among them
                if (warp == 0) {
                    float w = 0.f;
                    for (int q0 = 0; q0 < nchunk; q0 += 32) {
                        const int q = q0 + lane;
                        float wq = (q < nchunk && parts[q].m > -INFINITY) ? parts[q].w * ex2((parts[q].m - M) * sc) : 0.f;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) wq += __shfl_xor_sync(0xFFFFFFFFu, wq, o);
                        w += wq;
                    }
                    if (lane == 0) sh.W = w;
                }
                csync();
                const float target = info.top_p * sh.W;
                float wl = 0.f;
                visit_lst([&](float v, int32_t) { wl += ex2((v - M) * sc); }, L);
                wl = block_sum(wl, sh);
                if (!(wl >= target * (1.f + kMassTol))) {
                    whole = true;
                } else {
                    const uint32_t kF = select_key<E, true>(visit_lst, fkey(L), keyM, target, 0u, M, sc, sh);
                    visit_lst([&](float v, int32_t ix) {
                        if (fkey(v) >= kF) score_all(v, ix);
                    }, key_floor(kF));
                    block_best(best, bi, sh);
                }
            } else {
                // ---- top-k and / or min-p (then top-p over the survivors) --
                uint32_t *cnt = reinterpret_cast<uint32_t *>(lst + kListCap);
                // a short list gives its k-th largest value by rank counts, one
                // entry per thread, with no radix rounds
                uint32_t key_k = 0xFFFFFFFFu;
                if (f.use_k && n_list <= kThreads) {
                    if (tid == 0) sh.sel_excl_u = fkey(L);      // fewer than k listed: all survive
                    csync();
                    if (tid < n_list) {
                        const float v = lst[tid].v;
                        int gt = 0, ge = 0;
                        for (int j = 0; j < n_list; ++j) {
                            const float w = lst[j].v;
                            gt += (w > v) ? 1 : 0;
                            ge += (w >= v) ? 1 : 0;
                        }
                        if (gt < info.top_k && info.top_k <= ge) sh.sel_excl_u = fkey(v);
                    }
                    csync();
                    key_k = sh.sel_excl_u;
                    csync();
                }
                settle_from_list<E>(visit_lst, info, f, M, fkey(L), key_k, cnt,
                                    reinterpret_cast<unsigned long long *>(cnt + kTally), gs, best, bi, sh);
            }
        }
        if (whole) {
            // The summaries cannot settle the row (a nucleus reaching below
            // every chunk's counted values, a list overflow): exact selects
            // over the whole row, streamed again through the scratch (its
            // lists are spent).  After a timed-out records copy the
            // barriers' state is not known: the row keeps its argmax
            // (TIMEOUT is reported).
            csync();
            bi = INT_MAX;
            if (!sh.timeout) {
                const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
                const int h = min(mis ? static_cast<int>((16u - mis) / E::BYTES) : 0, p.V);
                bi = exact_row_token<E>(row, p.V, h, M, info, nz, scratch, sh, sh.ph);
            }
        }
        y = (bi == INT_MAX) ? AMAX : bi;
    }

    // ---------------------------------------------------- row results ---
    csync();
    if (tid == 0) {
        const float S = sh.S;
        if (p.row_max) p.row_max[r] = M;
        if (p.row_lse) p.row_lse[r] = (S > 0.f) ? M + logf(S) : -INFINITY;
        if (p.row_argmax) p.row_argmax[r] = AMAX;
        if (MODE == MODE_CONF) {
            const int32_t s = p.selected ? __ldg(p.selected + r) : AMAX;
            float cf = 0.f;
            if (s >= 0 && s < p.V) {
                // the argmax's own logit is the row maximum: no load
                const float zs = p.selected ? E::load(row, s) : M;
                cf = (S > 0.f) ? ex2((zs - M) * kLog2e) / S : 0.f;
            } else {
                set_status(p.status, SPEC_STATUS_BAD_SELECTED);
            }
            p.conf[r] = cf;
            p.draft_token[r] = s;
        } else {
            // active vocabulary: the argmax column's full token id
            if (MODE == MODE_GREEDY && p.vocab_ids) y = __ldg(p.vocab_ids + AMAX);
            if (p.row_token) p.row_token[r] = y;
            p.ws_tok[r] = y;
            if (MODE == MODE_RELAXED || (MODE == MODE_GREEDY && p.margin)) p.ws_flag[r] = flag;
        }
    }
    if (MODE != MODE_CONF && warp == 0) {
        // the request ticket: the row finishing its request runs the chain
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

// ------------------------------------------------------------- host -----

int chunks_per_row(int32_t V, int elt)
{
    const int64_t ce = kChunkBytes / elt;
    return static_cast<int>((static_cast<int64_t>(V) + ce - 1) / ce);
}

size_t max_row_bytes() { return static_cast<size_t>(kMaxChunks) * kChunkBytes; }

template <typename TIn, int MODE>
static cudaError_t launch_t(const VerifyParams &p, cudaStream_t stream)
{
    const size_t smem = kChunkBytes + sizeof(Shared) + ((MODE == MODE_SAMPLE && sizeof(TIn) == 2) ? kQueueBytes : 0);
    // the sampler's finish stages the records of the row's nchunk chunks
    // after its scratch; the scratch (and the records) also serve as the
    // two stages of a row streamed again for exact selects
    const size_t fin_base = sizeof(Shared) + kMaxChunks * sizeof(ChunkPart);
    const size_t fin_stage = (MODE == MODE_SAMPLE) ? fin_base + 2 * kRowStage : 0;
    const size_t smem_fin_max = std::max(fin_stage, fin_base + kFinScratch +
        (MODE == MODE_SAMPLE ? static_cast<size_t>(kMaxChunks) * Rec<Elt<TIn>>::BYTES : 0));
    const size_t smem_fin = std::max(fin_stage, fin_base + kFinScratch +
        (MODE == MODE_SAMPLE ? static_cast<size_t>(p.nchunk) * Rec<Elt<TIn>>::BYTES : 0));
    auto kstream = stream_chunks_kernel<TIn, MODE>;
    auto kfin = finish_rows_kernel<TIn, MODE>;
    // raise the dynamic shared-memory limits and prefer shared memory over
    // L1 (the stream kernel wants as many resident CTAs as it allows), once
    // per device
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        e = cudaFuncSetAttribute(kstream, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kstream, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kfin, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_fin_max));
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    const int rows = (MODE == MODE_CONF) ? p.n_rows : p.R_cap;
    // the finish kernel's extra CTAs write the outputs of requests without a
    // valid row range
    const int req_blocks = (MODE == MODE_CONF) ? 0 : (p.B + kThreads - 1) / kThreads;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (MODE == MODE_SAMPLE) {
        cudaLaunchConfig_t cr = {};
        cr.gridDim = dim3(static_cast<unsigned>((static_cast<int64_t>(rows) * 32 + 255) / 256), 1, 1);
        cr.blockDim = dim3(256, 1, 1);
        cr.stream = stream;
        cr.attrs = attr;
        cr.numAttrs = 1;
        e = cudaLaunchKernelEx(&cr, sample_records_kernel<TIn>, p);
        if (e != cudaSuccess) return e;
    }
    // one CTA per (row, chunk); the entry points bound rows * nchunk by 2^31 - 1
    cudaLaunchConfig_t cfg = {};
    if (MODE == MODE_SAMPLE || MODE == MODE_CONF)
        cfg.gridDim = dim3(static_cast<unsigned>(rows), static_cast<unsigned>(p.nchunk), 1);
    else if (rows <= 65535)
        cfg.gridDim = dim3(static_cast<unsigned>(p.nchunk), static_cast<unsigned>(rows), 1);
    else
        cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(rows) * p.nchunk), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    // the first kernel of a greedy-family call runs in plain stream order,
    // after everything the caller queued before (the previous call
    // included); the sampler's follows its records kernel
    cfg.numAttrs = (MODE == MODE_SAMPLE) ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kstream, p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cf = {};
    cf.gridDim = dim3(static_cast<unsigned>(rows + req_blocks), 1, 1);
    cf.blockDim = dim3(kThreads, 1, 1);
    cf.dynamicSmemBytes = smem_fin;
    cf.stream = stream;
    cf.attrs = attr;
    cf.numAttrs = 1;
    return cudaLaunchKernelEx(&cf, kfin, p);
}

// Rows at or above which bf16 relaxed top-K verification takes the row
// path (one CTA per row): twice the SM count, so that the row CTAs fill the
// GPU.  Greedy rows stay on the chunk path, which measured faster for them.
static cudaError_t row_path_threshold(int &rows)
{
    static int sms[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!sms[dev]) {
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    rows = 2 * sms[dev];
    return cudaSuccess;
}

cudaError_t launch_verify(int mode, int dtype, const VerifyParams &p, cudaStream_t stream)
{
    if (dtype == SPEC_BF16 && mode == MODE_RELAXED) {
        int th = 0;
        const cudaError_t e = row_path_threshold(th);
        if (e != cudaSuccess) return e;
        if (p.R_cap >= th) return launch_relaxed_rows(p, stream);
    }
    if (dtype == SPEC_BF16) {
        switch (mode) {
        case MODE_GREEDY: return launch_t<uint16_t, MODE_GREEDY>(p, stream);
        case MODE_RELAXED: return launch_t<uint16_t, MODE_RELAXED>(p, stream);
        case MODE_SAMPLE: return launch_t<uint16_t, MODE_SAMPLE>(p, stream);
        case MODE_CONF: return launch_t<uint16_t, MODE_CONF>(p, stream);
        }
    } else {
        switch (mode) {
        case MODE_GREEDY: return launch_t<float, MODE_GREEDY>(p, stream);
        case MODE_RELAXED: return launch_t<float, MODE_RELAXED>(p, stream);
        case MODE_SAMPLE: return launch_t<float, MODE_SAMPLE>(p, stream);
        case MODE_CONF: return launch_t<float, MODE_CONF>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace specv
