// verify.cu -- kernels for ragged packed logits: fused max / LSE / argmax,
// greedy acceptance (strict, loosened by a confidence margin, or over an
// active vocabulary), relaxed top-K acceptance, the filtered Gumbel-max
// sampler with the point-mass rejection chain, and the draft confidence.
//
// Kernels per call, chained with programmatic dependent launch:
//
//   prologue, one warp per packed row: the owner request (32-way search of
//     cu_rows), the row's position and validity and the owner's parameters,
//     as a 64-byte row record; requests without a valid row range get their
//     outputs here.  With a confidence margin it also decides whether the
//     margin applies to the row (position, generated-token count, a warp
//     scan of the protected ids) and records the draft's logit (NaN if not).
//   stream, one CTA per (row, chunk of kChunkBytes) on a two-dimensional
//     grid (the sampler chunk-major, the other modes row-major): thread 0
//     issues one 1-D TMA bulk copy of the chunk's 16-byte-aligned body into
//     shared memory first, then one of the row record on the same mbarrier
//     once the prologue has finished (the row is read from HBM exactly once;
//     unaligned head/tail elements use plain loads); many short CTAs per SM
//     keep the copies in flight.  Pass 1 takes two loops over the thread's
//     16-byte vectors: the maximum and the first vector holding it (selects
//     only), then sum exp(z - max) against it (packed f32x2 arithmetic for
//     bf16) and the count of logits above the draft's logit for relaxed
//     top-K; warp reductions (redux.sync) and a CTA reduction give the chunk
//     summary.  For the sampler (T > 0):
//       no filter   - the chunk's own Gumbel-max winner (vectors that cannot
//                     beat a lower bound taken from the thread maxima are
//                     skipped, and so are the logarithms of elements whose
//                     uniform cannot reach the running best);
//       top-k/min-p - the survivors form an upper set {z >= th}; the chunk
//                     bounds th from below (exact k-th largest of the thread
//                     maxima; chunk max + T ln min_p) and stores the elements
//                     above the bound as candidates;
//       top-p only  - the mass exp((z - m_c)/T) in bins of an absolute grid
//                     floor(z * 8/T) (per-warp fixed-point integer sums, each
//                     bin scaled by its own distance so the precision is
//                     relative), the total mass, and a candidate list above
//                     the 64-th largest thread maximum.
//     Only plain stores: nothing in this kernel waits for, or fences
//     against, another CTA.
//   finish, one CTA per row: combine the chunk summaries, then for the
//     sampler run radix selects (exact k-th largest value, exact top-p mass
//     crossing) over the candidate lists staged in shared memory and
//     Gumbel-max over the survivors with Philox4x32-10 uniforms (greedy
//     rows: the argmax, mapped to its full id over an active vocabulary;
//     with a margin, a per-row flag from the gap max - z[d]); bf16
//     survivors spanning at most kTally values take top-p over per-value
//     tallies instead.  Pure top-p brackets the nucleus boundary with the
//     combined bins; when the lists cover the undecided band the row is
//     settled from them.  A row that needs its logits again (a nucleus wider
//     than the lists, or a list or band overflow) is queued for the heavy
//     kernel with a short record.  The CTA finishing the last row of a
//     request (atomic ticket) runs the accept-while-equal prefix scan with
//     one warp ballot and writes the request's tokens and the optional
//     prefix-acceptance counters.
//   heavy (sampler only), persistent over the queued rows' half-chunks:
//     each piece is staged by TMA, its nucleus and band values are compacted
//     in shared memory and the nucleus scored with all lanes busy; its band
//     values go to a per-piece list, or, for a narrow bf16 band, to
//     per-value tallies.  The CTA finishing a row's last piece (atomic
//     ticket) settles the band exactly, or runs exact selects over the whole
//     row when a band or list overflowed, then runs the chain.
//
// Definitions: xLLM docs "自适应投机推理" §"启动示例" (ragged rejection
// sampler with packed-row owners, point-mass draft, replacement / bonus,
// temperature 0 = greedy, ordinary top-k/top-p/min-p semantics),
// §"基于 MTP logits 的自适应 target 验证" (exp(selected - logsumexp)),
// "vllm-hust-vSpec" README §"EAGLE 功能" (strict top-1 and relaxed top-K
// acceptance with a strict prefix, no per-request host sync, the active
// vocabulary with a full token-id map), §"启动" and §"通用参数" (the
// confidence margin and its position, token-count and protected-id options).
#include <cfloat>
#include <climits>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace specv {

constexpr int kCandCap = kWsCandCap;    // candidates one chunk may store
constexpr int kBins = kWsBins;          // pure top-p mass bins per chunk
constexpr float kBinsPerT = 8.0f;       // bin width T/8
constexpr float kFix = 1048576.0f;      // fixed-point scale of one bin weight (2^20)
constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23: adding it leaves integer parts in the low bits
constexpr int32_t kNoBins = INT_MIN;    // chunk grid origin too large for exact bins
constexpr int kBandCap = 2048;          // undecided values kept on chip
constexpr int kListCap = 2048;          // candidates the finish kernel stages on chip
constexpr int kPieceBytes = kChunkBytes / 2;   // heavy kernel: half a chunk per work item
constexpr int kSureH = 1024;            // heavy kernel: values >= zband compacted per piece
constexpr int kPieceList = kCandCap / 2;        // heavy kernel: band list entries per piece
constexpr int kFineBand = 64;           // heavy kernel: distinct bf16 band values tallied per chunk
constexpr int kTally = 128;             // finish kernel: bf16 values a top-p tally covers
constexpr int kRowStage = 16 * 1024;    // heavy kernel: bytes per row-streaming stage
constexpr int kPureListK = 64;          // pure top-p: list above the 64-th thread maximum
constexpr float kMassTol = 1e-5f;       // relative slack of the bin bracket
// Largest Gumbel noise of the uniform lattice: u <= 1 - 2^-24 gives
// -log(-log u) <= 24 ln 2 = 16.636; the bound used leaves a margin.
constexpr float kGumbelMax = 16.75f;

// row record written by the prologue (64 bytes)
struct __align__(16) RowInfo {
    int32_t b, pos, k_b, valid;
    int32_t draft, K, top_k, bad;
    float T, top_p, min_p, zd;
    uint32_t seed_lo, seed_hi, rid, sel;
};
static_assert(sizeof(RowInfo) == 64, "row record is 64 bytes");

// chunk summary kept in the workspace (32 bytes)
struct __align__(16) ChunkPart {
    float m;        // chunk max
    int32_t amax;   // first argmax in the chunk
    float s;        // sum exp(z - m)
    int32_t cnt;    // relaxed: logits above the draft's
    float gbest;    // sampler, no filter: best Gumbel score; top-p only: chunk mass
    int32_t gidx;   //   and its index; top-p only: bin-grid origin floor(m * 8/T)
    int32_t ncand;  // sampler with a bound: candidates (> kCandCap: overflow)
    float lev;      // sampler with a bound: the level the candidates lie above
};
static_assert(sizeof(ChunkPart) == 32, "chunk summary is 32 bytes");
static_assert(kChunkBytes / 16 <= 32 * kThreads, "a thread's vectors of a chunk fit a 32-bit mask");
static_assert(2 * kRowStage <= kChunkBytes, "a chunk buffer holds two row stages");
static_assert(2 * kRowStage <= kPieceBytes + (kSureH + kBandCap) * 8,
              "the heavy kernel streams rows through its piece, compaction and band space");
static_assert(kPieceBytes / 16 <= 32 * kThreads, "a thread's vectors of a piece fit a 32-bit mask");
static_assert(kFineBand * 12 <= kPieceList * 8, "a piece's value tallies fit its list space");

// Record of a row queued for the heavy kernel (32 bytes, at the start of the
// row's bin area, whose bins are no longer needed).
constexpr int32_t kHeavyBand = 1;       // settle the band over the chunks
constexpr int32_t kHeavyWhole = 2;      // exact selects over the whole row
struct __align__(16) HeavyRec {
    int32_t mode, qin, qband, amax;
    float M, target;
    float zin, zband;   // the same classes as value thresholds: abs_bin(z) >= q iff z >= zq
};
static_assert(sizeof(HeavyRec) == 32, "heavy record is 32 bytes");

// per-piece result of the heavy pass (16 bytes each, after the record)
struct __align__(16) HeavyPart {
    float best;     // best Gumbel score among the piece's nucleus values
    int32_t bi;     //   and its index
    float mass;     // their mass exp((z - M)/T)
    int32_t nband;  // band values stored in the piece's list (> kPieceList: overflow)
};

// shared scratch common to the row kernels
struct __align__(16) Shared {
    RowInfo info;
    ChunkPart part;
    uint32_t hist[256];
    uint32_t scan[kWarps];
    float red_f[kWarps * 2];
    int32_t red_i[kWarps * 2];
    int32_t offs[2 * kMaxChunks + 1];
    float M, S, W, sel_excl_f, theta;
    int32_t AMAX, CNT, sel_bin, sel_found, total, overflow, cand_n, R, J, nobins, last, heavy;
    uint32_t sel_excl_u, lkey;
    float extras_v[16];
    int32_t extras_i[16];
    int32_t timeout;
    uint64_t mbar[2];
};

struct Cand {
    float v;
    int32_t i;
};

// ------------------------------------------------------------ helpers -----

// combine two (max, first-argmax, scaled sum, count) partials
__device__ __forceinline__ void combine(float &m, int32_t &a, float &s, int32_t &c, float om,
                                        int32_t oa, float os, int32_t oc, bool need_sum)
{
    const float nm = fmaxf(m, om);
    if (need_sum) {
        const float s1 = (m > -INFINITY) ? s * ex2((m - nm) * kLog2e) : 0.f;
        const float s2 = (om > -INFINITY) ? os * ex2((om - nm) * kLog2e) : 0.f;
        s = s1 + s2;
    }
    if (om > m || (om == m && oa < a)) a = oa;
    m = nm;
    c += oc;
}

// Block-wide search, from the top bin (255) down, of the bin where the running
// total first reaches `target` (thread t holds bin 255 - t).  Writes
// sh.sel_bin and the total above that bin; when rounding keeps the float
// total below the target, the lowest non-empty bin is taken.
template <typename V>
__device__ void find_crossing(const V *hist, V target, Shared &sh)
{
    constexpr bool IS_F = std::is_same<V, float>::value;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const V v = hist[255 - t];
    V incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    V *wt = reinterpret_cast<V *>(sh.scan);
    if (lane == 31) wt[warp] = incl;
    if (t == 0) sh.sel_found = 0;
    __syncthreads();
    V off = V(0);
    for (int w = 0; w < warp; ++w) off += wt[w];
    incl += off;
    const V excl = incl - v;
    if (v > V(0) && excl < target && target <= incl) {
        sh.sel_found = 1;
        sh.sel_bin = 255 - t;
        if constexpr (IS_F) sh.sel_excl_f = excl;
        else sh.sel_excl_u = excl;
    }
    __syncthreads();
    if (!sh.sel_found) {
        if (t == 0) {
            int best = -1;
            V run = V(0), before = V(0);
            for (int q = 255; q >= 0; --q)
                if (hist[q] > V(0)) { best = q; before = run; run += hist[q]; }
            sh.sel_bin = best;
            if constexpr (IS_F) sh.sel_excl_f = before;
            else sh.sel_excl_u = before;
        }
        __syncthreads();
    }
}

// Float threshold equivalent to "key >= k": -inf for the keys below -inf's.
__device__ __forceinline__ float key_floor(uint32_t k)
{
    return (k <= 0x007FFFFFu) ? -INFINITY : key_value(k);
}

// Radix select over the keys of the values produced by `visit(fn, thr)`
// (fn(v, i) for every element >= thr).  Values are compared through their
// order-preserving keys; bf16 values have 16 significant key bits, fp32 32.
// Only keys in [lo, hi] take part (hi must bound every such key from above).
// The first digit holds the 8 bits below and including the highest bit where
// lo and hi differ (the bits above are common), so it spreads the values
// over the bins; later digits take the next 8 bits (the last one fewer).
//   COUNT (MASS = false): the key of the k-th largest value.
//   MASS: the key of the value group where the cumulative weight
//     exp((z - M) * sc), counted from the top, first reaches `target`.
// On the last digit every bin holds one value, so the weights there come
// from integer counts (no float atomics).
template <typename E, bool MASS, typename Visit>
__device__ uint32_t select_key(Visit &&visit, uint32_t lo, uint32_t hi, float target, uint32_t k,
                               float M, float sc, Shared &sh)
{
    constexpr int VS = (E::BYTES == 2) ? 16 : 0;
    const uint32_t vlo = lo >> VS, vhi = hi >> VS;
    const uint32_t x = vlo ^ vhi;
    const int top = x ? 31 - __clz(x) : 0;
    int shift = max(top - 7, 0);
    int width = top - shift + 1;
    uint32_t prefix = (top + 1 >= 32) ? 0u : (vhi >> (top + 1));
    const float thr = key_floor(lo);
    const int t = threadIdx.x;
    for (;;) {
        sh.hist[t] = 0u;
        __syncthreads();
        const int above = shift + width;
        const uint32_t dmask = (1u << width) - 1u;
        const bool wide = MASS && shift > 0;
        visit([&](float v, int32_t) {
            const uint32_t fk = fkey(v);
            if (fk < lo) return;
            const uint32_t vk = fk >> VS;
            if (above < 32 && (vk >> above) != prefix) return;
            const uint32_t bin = (vk >> shift) & dmask;
            if (wide) atomicAdd(reinterpret_cast<float *>(&sh.hist[bin]), ex2((v - M) * sc));
            else atomicAdd(&sh.hist[bin], 1u);
        }, thr);
        __syncthreads();
        if (MASS && shift == 0) {
            // one value per bin: weight = count * exp((value - M) * sc)
            const uint32_t c = sh.hist[t];
            float w = 0.f;
            if (c) {
                const uint32_t vk = (prefix << width) | static_cast<uint32_t>(t);
                const uint32_t fk = VS ? ((vk << 16) | ((vk & 0x8000u) ? 0u : 0xFFFFu)) : vk;
                w = static_cast<float>(c) * ex2((key_value(fk) - M) * sc);
            }
            __syncthreads();
            reinterpret_cast<float *>(sh.hist)[t] = w;
            __syncthreads();
        }
        if (MASS) find_crossing<float>(reinterpret_cast<const float *>(sh.hist), target, sh);
        else find_crossing<uint32_t>(sh.hist, k, sh);
        const int bin = sh.sel_bin;
        if (MASS) target -= sh.sel_excl_f;
        else k -= sh.sel_excl_u;
        prefix = (prefix << width) | static_cast<uint32_t>(bin < 0 ? 0 : bin);
        __syncthreads();
        if (shift == 0) break;
        width = min(8, shift);
        shift -= width;
    }
    if (VS) return (prefix << 16) | ((prefix & 0x8000u) ? 0u : 0xFFFFu);
    return prefix;
}

// Warp-aggregated append to a counter: one atomic per group of lanes that
// call it together; returns this lane's slot.
__device__ __forceinline__ int warp_append(int *counter)
{
    const unsigned mask = __activemask();
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(mask));
    base = __shfl_sync(mask, base, leader);
    return base + __popc(mask & ((1u << lane) - 1u));
}

// block reduction of a float sum (result in every thread)
__device__ __forceinline__ float block_sum(float v, Shared &sh)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((threadIdx.x & 31) == 0) sh.red_f[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int q = 0; q < kWarps; ++q) t += sh.red_f[q];
    __syncthreads();
    return t;
}

// block reduction of a (score, index) maximum, lowest index on ties
__device__ __forceinline__ void block_best(float &best, int32_t &bi, Shared &sh)
{
    // the warp's best score, then the lowest index attaining it
    const float wb = warp_max_f32(best);
    bi = static_cast<int32_t>(__reduce_min_sync(0xFFFFFFFFu, (best == wb) ? static_cast<uint32_t>(bi) : 0xFFFFFFFFu));
    best = wb;
    if ((threadIdx.x & 31) == 0) { sh.red_f[threadIdx.x >> 5] = best; sh.red_i[threadIdx.x >> 5] = bi; }
    __syncthreads();
    best = -INFINITY;
    bi = INT_MAX;
    for (int q = 0; q < kWarps; ++q)
        if (sh.red_f[q] > best || (sh.red_f[q] == best && sh.red_i[q] < bi)) { best = sh.red_f[q]; bi = sh.red_i[q]; }
    __syncthreads();
}

// block minimum and maximum of a key (result in every thread)
__device__ __forceinline__ void block_minmax(uint32_t &mn, uint32_t &mx, Shared &sh)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if ((threadIdx.x & 31) == 0) {
        sh.red_i[threadIdx.x >> 5] = static_cast<int32_t>(mn);
        sh.red_i[kWarps + (threadIdx.x >> 5)] = static_cast<int32_t>(mx);
    }
    __syncthreads();
    mn = 0xFFFFFFFFu;
    mx = 0u;
    for (int q = 0; q < kWarps; ++q) {
        mn = min(mn, static_cast<uint32_t>(sh.red_i[q]));
        mx = max(mx, static_cast<uint32_t>(sh.red_i[kWarps + q]));
    }
    __syncthreads();
}

// Top-k bound inside a chunk for k above the thread count: the highest level
// L = m_c - D (D from a fixed ladder) with at least k thread maxima >= L.
// Thread maxima are distinct elements, so at least k elements of the chunk
// are >= L and the chunk's share of the row's top k lies above it.  False
// if no level qualifies.
__device__ __forceinline__ bool kth_level(float thread_max, float m_c, int k, float &level,
                                          Shared &sh)
{
    constexpr int NL = 8;
    const float ladder[NL] = {0.25f, 0.5f, 1.f, 2.f, 3.f, 4.f, 6.f, 8.f};
    int cnt[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) cnt[l] = (thread_max >= m_c - ladder[l]) ? 1 : 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt[l] += __shfl_xor_sync(0xFFFFFFFFu, cnt[l], o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int *wc = reinterpret_cast<int *>(sh.hist);        // [kWarps][NL]
    if (lane == 0)
#pragma unroll
        for (int l = 0; l < NL; ++l) wc[warp * NL + l] = cnt[l];
    __syncthreads();
    int sel = -1;
    for (int l = 0; l < NL; ++l) {
        int t = 0;
        for (int w = 0; w < kWarps; ++w) t += wc[w * NL + l];
        if (t >= k) { sel = l; break; }
    }
    __syncthreads();
    if (sel < 0) return false;
    level = m_c - ladder[sel];
    return true;
}

// Philox4x32-10 stream of one row: counter (i >> 2, position, request id,
// step), key (seed lo, seed hi); element i takes word i & 3.
struct Noise {
    uint32_t pos, rid, step, k0, k1;
    __device__ __forceinline__ uint4 block(uint32_t ctr) const
    {
        return philox4x32_10(make_uint4(ctr, pos, rid, step), k0, k1);
    }
    // Gumbel-perturbed score z/T - log(-log u_i) of element i
    __device__ __forceinline__ float score(float v, int32_t ix, float invT) const
    {
        const uint4 w = block(static_cast<uint32_t>(ix) >> 2);
        return fmaf(v, invT, gumbel_of(word_of(w, static_cast<uint32_t>(ix) & 3u)));
    }
};

// keep the better of (s, ix) and (best, bi): higher score, lower index on ties
__device__ __forceinline__ void keep_best(float s, int32_t ix, float &best, int32_t &bi)
{
    if (s > best || (s == best && ix < bi)) { best = s; bi = ix; }
}

// Scores of the VEC elements of one vector starting at element `base`, a
// multiple of 4 (the vector covers whole Philox blocks), whose largest value
// is vm.  An element can only reach `best` if its Gumbel noise -log(-log u)
// reaches best - z/T, i.e. -log u <= D = exp(z/T - best) <= exp(vm/T - best);
// as -log u >= 1 - u, an element with 1 - u > D cannot, and for u on the
// lattice (2k + 1) 2^-24 (k = word >> 9) that is k < (2^24 - 1 - D 2^24) / 2.
// Those are skipped without the logarithms (one below the bound, for the
// rounding of D); the others are scored as usual.
template <int VEC>
__device__ __forceinline__ void score_vec(const float (&x)[VEC], float vm, int32_t base, float invT,
                                          const Noise &nz, float &best, int32_t &bi)
{
    const float D = ex2((vm * invT - best) * kLog2e);
    const float t = fmaf(-D, 16777216.f, 16777215.f) * 0.5f;
    const uint32_t kthr = (t >= 2.f) ? static_cast<uint32_t>(t) - 1u : 0u;
#pragma unroll
    for (int h = 0; h < VEC / 4; ++h) {
        const uint4 w = nz.block((static_cast<uint32_t>(base) >> 2) + h);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if ((ws[j] >> 9) >= kthr)
                keep_best(fmaf(x[4 * h + j], invT, gumbel_of(ws[j])), base + 4 * h + j, best, bi);
    }
}

// Gumbel scorer for elements visited one at a time; caches the last block.
struct GumbelScorer {
    float invT;
    Noise nz;
    uint32_t cached;
    uint4 words;
    __device__ __forceinline__ float operator()(float v, int32_t ix)
    {
        const uint32_t ctr = static_cast<uint32_t>(ix) >> 2;
        if (ctr != cached) {
            words = nz.block(ctr);
            cached = ctr;
        }
        return fmaf(v, invT, gumbel_of(word_of(words, static_cast<uint32_t>(ix) & 3u)));
    }
};

// Absolute bin of a value on the grid of width T/8: floor(z * s8), s8 = 8/T,
// clamped.  Monotone non-decreasing in z, and computed the same way by the
// stream and finish kernels, so both classify every value identically.
__device__ __forceinline__ float bin_scale(float T) { return kBinsPerT / T; }

__device__ __forceinline__ int32_t abs_bin(float z, float s8)
{
    const float f = fminf(fmaxf(floorf(z * s8), -536870912.f), 536870912.f);
    return static_cast<int32_t>(f);
}

// The smallest float z with abs_bin(z, s8) >= q (abs_bin is monotone, so the
// set of such z is {z >= result}): a binary search over the order-preserving
// keys of the floats from -inf to +inf.
__device__ __forceinline__ float bin_floor_value(int32_t q, float s8)
{
    if (abs_bin(-INFINITY, s8) >= q) return -INFINITY;
    // the answer lies within a few floats of q / s8: walk there first
    {
        uint32_t k = fkey(static_cast<float>(q) / s8);
        for (int it = 0; it < 16; ++it) {
            if (k <= fkey(-INFINITY) || k >= fkey(INFINITY)) break;
            const bool in = abs_bin(key_value(k), s8) >= q;
            if (in && abs_bin(key_value(k - 1), s8) < q) return key_value(k);
            k = in ? k - 1 : k + 1;
        }
    }
    uint32_t lo = fkey(-INFINITY), hi = fkey(INFINITY);   // abs_bin(+inf) is the largest bin
    while (hi - lo > 1) {
        const uint32_t mid = lo + (hi - lo) / 2;
        if (abs_bin(key_value(mid), s8) >= q) hi = mid;
        else lo = mid;
    }
    return key_value(hi);
}

// Pass 1 over this thread's 16-byte vectors of the staged chunk, in two
// loops.  The first finds the thread's maximum and the first vector holding
// it with selects only (a running-max update with per-vector rescaling is
// taken by some lane of the warp on most iterations, so the warp would run
// it nearly every time); the first index attaining the maximum comes from
// that vector.  The second loop sums exp(z - max) against the fixed maximum
// (SUM) and counts z > zd (relaxed mode).  The maximum starts at a finite
// sentinel far below any logit, so -inf logits contribute exp(-inf) = 0; a
// chunk of only -inf reports -inf.
constexpr float kSentinel = -1.0e38f;

template <typename E, int MODE, bool SUM>
__device__ __forceinline__ float pass1(const uint4 *body, int nb, int a0, float zd, int32_t &targ,
                                       float &tsum, int32_t &tcnt)
{
    constexpr int VEC = E::VEC;
    float tmax = kSentinel;
    int jmax = -1;
#pragma unroll 4
    for (int i = threadIdx.x, j = 0; i < nb; i += kThreads, ++j) {
        const float vm = E::vmax(body[i]);
        jmax = (vm > tmax) ? j : jmax;
        tmax = fmaxf(tmax, vm);
    }
    if (jmax >= 0) {
        const int i = threadIdx.x + jmax * kThreads;
        float x[VEC];
        E::unpack(body[i], x);
        int first = VEC - 1;
#pragma unroll
        for (int q = VEC - 1; q >= 0; --q)
            if (x[q] == tmax) first = q;
        targ = a0 + i * VEC + first;
    }
    if (SUM || MODE == MODE_RELAXED) {
        const float c0 = -tmax * kLog2e;
        if constexpr (E::BYTES == 2) {
            // the two halves of each 32-bit word are one f32x2 pair: packed
            // exponent arguments and two packed accumulators
            uint64_t acc = f2_pack(0.f, 0.f);
            const uint64_t l2 = f2_pack(kLog2e, kLog2e), c2 = f2_pack(c0, c0);
#pragma unroll 4
            for (int i = threadIdx.x; i < nb; i += kThreads) {
                const uint4 v = body[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float lo = bf_lo(w[j]), hi = bf_hi(w[j]);
                    if (SUM) {
                        float e0, e1;
                        f2_unpack(f2_fma(f2_pack(lo, hi), l2, c2), e0, e1);
                        acc = f2_add(acc, f2_pack(ex2(e0), ex2(e1)));
                    }
                    if (MODE == MODE_RELAXED) tcnt += ((lo > zd) ? 1 : 0) + ((hi > zd) ? 1 : 0);
                }
            }
            float s0, s1;
            f2_unpack(acc, s0, s1);
            tsum = s0 + s1;
        } else {
            float s0 = 0.f, s1 = 0.f;     // two accumulators: independent add chains
            for (int i = threadIdx.x; i < nb; i += kThreads) {
                float x[VEC];
                E::unpack(body[i], x);
#pragma unroll
                for (int j = 0; j < VEC; j += 2) {
                    if (SUM) {
                        s0 += ex2(fmaf(x[j], kLog2e, c0));
                        s1 += ex2(fmaf(x[j + 1], kLog2e, c0));
                    }
                    if (MODE == MODE_RELAXED) tcnt += ((x[j] > zd) ? 1 : 0) + ((x[j + 1] > zd) ? 1 : 0);
                }
            }
            tsum = s0 + s1;
        }
    }
    if (tmax == kSentinel) { tmax = -INFINITY; tsum = 0.f; }
    return tmax;
}

// chunk c of a row: elements [e0, e1); 16-byte-aligned body of nb vectors
// from element a0; head [e0, a0) and tail [a1, e1) use plain loads
struct ChunkGeom {
    int e0, e1, a0, nb, a1, n_head, n_extra, h;
};

template <typename E>
__device__ __forceinline__ ChunkGeom chunk_geom(const void *row, int c, int V)
{
    constexpr int CE = kChunkBytes / E::BYTES;
    ChunkGeom g;
    const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
    g.h = min(mis ? static_cast<int>((16u - mis) / E::BYTES) : 0, V);
    g.e0 = c * CE;
    g.e1 = min(V, g.e0 + CE);
    g.a0 = min(g.e0 + g.h, g.e1);
    g.nb = (g.e1 - g.a0) / E::VEC;
    g.a1 = g.a0 + g.nb * E::VEC;
    g.n_head = g.a0 - g.e0;
    g.n_extra = g.n_head + (g.e1 - g.a1);
    return g;
}

// ---------------------------------------------------------- prologue -----
// One warp per packed row: owner request (largest b with cu_rows[b] <= r),
// position, validity and the owner's parameters.  Extra CTAs handle the
// requests without a valid row range.
template <typename TIn, int MODE>
__global__ void __launch_bounds__(256) row_info_kernel(const VerifyParams p, int row_blocks)
{
    using E = Elt<TIn>;
    griddep_launch_dependents();
    // the heavy-row queue of the sampler starts empty (the previous call's
    // heavy kernel has completed before this kernel starts)
    if (MODE == MODE_SAMPLE && blockIdx.x == 0 && threadIdx.x == 0) p.ws_hrows[0] = 0;
    const int lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) >= row_blocks) {
        const int b = (blockIdx.x - row_blocks) * 256 + threadIdx.x;
        if (b >= p.B) return;
        const int32_t c0 = __ldg(p.cu_rows), lo = __ldg(p.cu_rows + b), hi = __ldg(p.cu_rows + b + 1);
        const int32_t n = hi - lo;
        if (c0 != 0 || n < 1 || n - 1 > p.k_max || hi > p.R_cap) {
            p.accepted_len[b] = 0;
            p.next_token[b] = -1;
            for (int j = 0; j <= p.k_max; ++j) p.out_tokens[static_cast<int64_t>(b) * (p.k_max + 1) + j] = -1;
            set_status(p.status, SPEC_STATUS_BAD_ROWS);
        }
        return;
    }
    const int r = (blockIdx.x * 256 + threadIdx.x) >> 5;
    if (r >= p.R_cap) return;
    RowInfo inf;
    inf.sel = 0; inf.bad = 0; inf.zd = INFINITY; inf.K = 1;
    inf.T = 0.f; inf.top_k = 0; inf.top_p = 1.f; inf.min_p = 0.f;
    inf.seed_lo = inf.seed_hi = inf.rid = 0;
    int lo = 0, hi = p.B - 1;
    while (hi > lo) {
        const int step = (hi - lo + 31) / 32;
        const int idx = min(lo + lane * step, hi);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, __ldg(p.cu_rows + idx) <= r);
        const int L = m ? 31 - __clz(m) : 0;
        const int nlo = min(lo + L * step, hi);
        const int nhi = (L == 31) ? hi : min(lo + (L + 1) * step - 1, hi);
        lo = nlo;
        hi = nhi;
    }
    const int b = lo;
    const int32_t c0 = __ldg(p.cu_rows), rb = __ldg(p.cu_rows + b), re = __ldg(p.cu_rows + b + 1);
    inf.b = b;
    inf.pos = r - rb;
    inf.k_b = re - rb - 1;
    inf.valid = (c0 == 0 && rb <= r && r < re && inf.k_b >= 0 && inf.k_b <= p.k_max && re <= p.R_cap);
    inf.draft = __ldg(p.draft_ids + r);
    if (MODE == MODE_SAMPLE) {
        float T = __ldg(p.temperature + b), tp = __ldg(p.top_p + b), mp = __ldg(p.min_p + b);
        int32_t tk = __ldg(p.top_k + b);
        if (!(T >= 0.f) || isinf(T)) { inf.bad |= SPEC_STATUS_BAD_TEMPERATURE; T = 0.f; }
        if (tk < 0) { inf.bad |= SPEC_STATUS_BAD_TOP_K; tk = 0; }
        if (!(tp > 0.f && tp <= 1.f)) { inf.bad |= SPEC_STATUS_BAD_TOP_P; tp = 1.f; }
        if (!(mp >= 0.f && mp <= 1.f)) { inf.bad |= SPEC_STATUS_BAD_MIN_P; mp = 0.f; }
        inf.T = T; inf.top_k = tk; inf.top_p = tp; inf.min_p = mp;
        const uint64_t sd = __ldg(reinterpret_cast<const unsigned long long *>(p.seed) + b);
        inf.seed_lo = static_cast<uint32_t>(sd);
        inf.seed_hi = static_cast<uint32_t>(sd >> 32);
        inf.rid = p.request_id ? __ldg(p.request_id + b) : static_cast<uint32_t>(b);
    }
    if (MODE == MODE_GREEDY && p.margin) {
        // the margin applies to a draft row at an eligible position whose
        // draft is in the vocabulary and not protected; elsewhere zd is NaN,
        // which fails the gap test in the finish
        const float mg = __ldg(p.margin + b);
        if (isnan(mg)) inf.bad |= SPEC_STATUS_BAD_MARGIN;
        const int32_t gen = p.generated ? __ldg(p.generated + b) : 0;
        const int32_t d = inf.draft;
        bool elig = inf.valid && inf.pos < inf.k_b && d >= 0 && d < p.V && !isnan(mg) &&
                    inf.pos >= p.from_position &&
                    static_cast<int64_t>(gen) + inf.pos >= static_cast<int64_t>(p.after_tokens);
        if (elig && p.n_protected > 0) {
            bool hit = false;
            for (int i = lane; i < p.n_protected; i += 32) hit |= (__ldg(p.protected_ids + i) == d);
            elig = !__any_sync(0xFFFFFFFFu, hit);
        }
        inf.zd = __int_as_float(0x7FC00000);
        if (elig) {
            const TIn *row = reinterpret_cast<const TIn *>(p.logits) + static_cast<int64_t>(r) * p.ld;
            inf.zd = E::load(row, d);
        }
    }
    if (MODE == MODE_RELAXED) {
        int32_t K = __ldg(p.relaxed_k + b);
        if (K < 1) { inf.bad |= SPEC_STATUS_BAD_RELAXED_K; K = 1; }
        inf.K = K;
        const TIn *row = reinterpret_cast<const TIn *>(p.logits) + static_cast<int64_t>(r) * p.ld;
        if (inf.draft >= 0 && inf.draft < p.V) inf.zd = E::load(row, inf.draft);
    }
    if (lane == 0) reinterpret_cast<RowInfo *>(p.ws_info)[r] = inf;
}

// ------------------------------------------------------ stream kernel ----

// The k-th largest of the CTA's thread maxima (k <= kThreads): at least k
// distinct elements of the chunk are >= it.  The maxima's order-preserving
// keys go to shared memory; warp 0 holds eight each and searches bit by bit
// below the bits the smallest and largest share, keeping a bit when at least
// k keys reach the prefix with it set (a warp sum per bit, no CTA barrier).
template <typename E>
__device__ __forceinline__ float kth_thread_max(float v, int k, float m_c, Shared &sh)
{
    constexpr int VS = (E::BYTES == 2) ? 16 : 0;
    (void)m_c;
    const int lane = threadIdx.x & 31;
    sh.hist[threadIdx.x] = fkey(v) >> VS;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t kv[kThreads / 32];
        uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
        for (int j = 0; j < kThreads / 32; ++j) {
            kv[j] = sh.hist[lane + 32 * j];
            mn = min(mn, kv[j]);
            mx = max(mx, kv[j]);
        }
        mn = __reduce_min_sync(0xFFFFFFFFu, mn);
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        const uint32_t x = mn ^ mx;
        const int top = x ? 31 - __clz(x) : -1;
        // every key lies in [mn, mx]: the bits above `top` are theirs
        uint32_t ans = (top >= 31) ? 0u : (mx >> (top + 1)) << (top + 1);
        for (int bit = top; bit >= 0; --bit) {
            const uint32_t cand = ans | (1u << bit);
            uint32_t c = 0;
#pragma unroll
            for (int j = 0; j < kThreads / 32; ++j) c += (kv[j] >= cand) ? 1u : 0u;
            if (__reduce_add_sync(0xFFFFFFFFu, c) >= static_cast<uint32_t>(k)) ans = cand;
        }
        if (lane == 0) sh.sel_excl_u = ans;
    }
    __syncthreads();
    const uint32_t ans = sh.sel_excl_u;
    const uint32_t key = VS ? ((ans << 16) | ((ans & 0x8000u) ? 0u : 0xFFFFu)) : ans;
    return key_floor(key);
}

// CTA reduction of the per-thread (max, first argmax, sum exp(z - max),
// count) into the chunk summary sh.part: the maximum first, then the lowest
// index attaining it, the sums rescaled once to the maximum, the counts.
template <int MODE>
__device__ __forceinline__ void chunk_reduce(float tmax, int32_t targ, float tsum, int32_t tcnt,
                                             bool need_sum, Shared &sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp maximum, then the lowest index attaining it (indices are >= 0)
    const float wm = warp_max_f32(tmax);
    const int32_t wa = __reduce_min_sync(0xFFFFFFFFu, (tmax == wm) ? targ : INT_MAX);
    float ws = 0.f;
    if (need_sum) {
        ws = (tmax > -INFINITY) ? tsum * ex2((tmax - wm) * kLog2e) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, o);
    }
    int32_t wc = 0;
    if (MODE == MODE_RELAXED) wc = __reduce_add_sync(0xFFFFFFFFu, tcnt);
    if (lane == 0) {
        sh.red_f[warp] = wm; sh.red_f[kWarps + warp] = ws;
        sh.red_i[warp] = wa; sh.red_i[kWarps + warp] = wc;
    }
    __syncthreads();
    if (warp == 0) {
        const bool on = lane < kWarps;
        const float m0 = on ? sh.red_f[lane] : -INFINITY;
        const float m = warp_max_f32(m0);
        const int32_t a = __reduce_min_sync(0xFFFFFFFFu, (on && m0 == m) ? sh.red_i[lane] : INT_MAX);
        float sm_ = 0.f;
        if (need_sum) {
            sm_ = (on && m0 > -INFINITY) ? sh.red_f[kWarps + lane] * ex2((m0 - m) * kLog2e) : 0.f;
#pragma unroll
            for (int o = kWarps / 2; o > 0; o >>= 1) sm_ += __shfl_xor_sync(0xFFFFFFFFu, sm_, o);
        }
        const int32_t cc = __reduce_add_sync(0xFFFFFFFFu, on ? sh.red_i[kWarps + lane] : 0);
        if (lane == 0) {
            sh.part.m = m; sh.part.amax = a; sh.part.s = sm_; sh.part.cnt = cc;
            sh.part.gbest = -INFINITY; sh.part.gidx = INT_MAX; sh.part.ncand = 0;
            sh.part.lev = -INFINITY;
        }
    }
    __syncthreads();
}

// One CTA per (row, chunk); plain stores of the chunk summary only.  Many
// short CTAs per SM keep the bulk copies in flight.
template <typename TIn, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == MODE_SAMPLE ? 5 : 6)
    stream_chunks_kernel(const VerifyParams p)
{
    using E = Elt<TIn>;
    constexpr int VEC = E::VEC;
    constexpr bool HAS_INFO = (MODE != MODE_CONF);
    extern __shared__ __align__(128) uint8_t smem[];
    const uint4 *body = reinterpret_cast<const uint4 *>(smem);
    Shared &sh = *reinterpret_cast<Shared *>(smem + kChunkBytes);
    Cand *cand = reinterpret_cast<Cand *>(reinterpret_cast<uint8_t *>(&sh) + sizeof(Shared));
    uint32_t *wbins = reinterpret_cast<uint32_t *>(cand + kCandCap);   // [kWarps][kBins] (sampler)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = p.nchunk;
    // The sampler takes chunk-major order: a chunk's cost depends on its
    // row's filters, and this spreads every row's chunks evenly over the
    // grid, with the short tail chunks in the last wave.  Uniform modes keep
    // row-major order.  The grid is two-dimensional with the faster index in
    // x (sampler: x = row, y = chunk; else x = chunk, y = row), so the order
    // comes without divisions; row-major grids of more than 65535 rows are
    // one-dimensional.
    int r, c;
    if (MODE == MODE_SAMPLE) {
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

    if (tid == 0) {
        // The logits buffer holds R_cap rows, so the chunk copy is issued
        // before anything else (in bounds even for rows past cu_rows[B]).
        sh.timeout = 0;
        mbar_init(&sh.mbar[0], 1);
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(g.nb) * 16u;
        mbar_arrive_expect_tx(&sh.mbar[0], bytes + (HAS_INFO ? 64u : 0u));
        if (bytes) bulk_g2s(smem, row + g.a0, bytes, &sh.mbar[0]);
        int32_t R = p.n_rows;
        if (MODE != MODE_CONF) R = __ldg(p.cu_rows + p.B);
        if (HAS_INFO) {
            griddep_wait();                 // row records of the prologue
            bulk_g2s(&sh.info, reinterpret_cast<const RowInfo *>(p.ws_info) + r, 64u, &sh.mbar[0]);
        } else {
            RowInfo inf = {};
            inf.b = r; inf.valid = 1;
            sh.info = inf;
        }
        sh.R = min(R, p.R_cap);
    }
    float xe = -INFINITY;
    int32_t ie = INT_MAX;
    if (tid < g.n_extra) {
        ie = (tid < g.n_head) ? g.e0 + tid : g.a1 + (tid - g.n_head);
        xe = E::load(row, ie);
        sh.extras_v[tid] = xe;
        sh.extras_i[tid] = ie;
    }
    __syncthreads();
    if (tid == 0 && !mbar_wait(&sh.mbar[0], 0)) {
        // the copy did not land in time: report it, give the copy one more
        // bounded wait, and leave without touching the buffer
        set_status(p.status, SPEC_STATUS_TIMEOUT);
        mbar_wait(&sh.mbar[0], 0);
        sh.timeout = 1;
    }
    __syncthreads();
    if (sh.timeout || r >= sh.R) return;
    const RowInfo &info = sh.info;
    if (!info.valid) return;

    // ---------------------------------------------------------- pass 1 --
    const bool need_sum = (MODE == MODE_CONF) || (p.row_lse != nullptr);
    const float zd = info.zd;
    float tmax = -INFINITY, tsum = 0.f;
    int32_t targ = INT_MAX, tcnt = 0;
    if (need_sum) tmax = pass1<E, MODE, true>(body, g.nb, g.a0, zd, targ, tsum, tcnt);
    else tmax = pass1<E, MODE, false>(body, g.nb, g.a0, zd, targ, tsum, tcnt);
    if (tid < g.n_extra)
        combine(tmax, targ, tsum, tcnt, xe, ie, 1.f, (MODE == MODE_RELAXED && xe > zd) ? 1 : 0,
                need_sum);
    const float thread_max = tmax;
    const int32_t thread_arg = targ;
    chunk_reduce<MODE>(tmax, targ, tsum, tcnt, need_sum, sh);

    // ------------------------------------------ sampler: chunk summary --
    const int64_t rc = static_cast<int64_t>(r) * nchunk + c;
    if (MODE == MODE_SAMPLE && info.T > 0.f) {
        const float T = info.T;
        const float invT = 1.0f / T;
        const float sc = invT * kLog2e;
        const bool use_k = info.top_k > 0 && info.top_k < p.V;
        const bool use_m = info.min_p > 0.f;
        const bool use_p = info.top_p < 1.f;
        const bool unfiltered = !use_k && !use_m && !use_p;
        const bool pure_p = !use_k && !use_m && use_p;
        const float m_c = sh.part.m;
        const Noise nz{static_cast<uint32_t>(info.pos), info.rid, p.step, info.seed_lo, info.seed_hi};
        auto visit_chunk = [&](auto &&fn, float thr) {
            for (int i = tid; i < g.nb; i += kThreads) {
                const uint4 v = body[i];
                if (!(E::vmax(v) >= thr)) continue;
                float x[VEC];
                E::unpack(v, x);
#pragma unroll
                for (int q = 0; q < VEC; ++q)
                    if (x[q] >= thr) fn(x[q], g.a0 + i * VEC + q);
            }
            if (tid < g.n_extra && sh.extras_v[tid] >= thr) fn(sh.extras_v[tid], sh.extras_i[tid]);
        };
        if (!(m_c > -INFINITY)) {
            // only -inf here: no candidates, no mass, no bins
            if (pure_p && tid < kBins) p.ws_bins[rc * kBins + tid] = 0.f;
            if (pure_p && tid == 0) { sh.part.gbest = 0.f; sh.part.gidx = INT_MIN + 1; }
        } else if (unfiltered) {
            // lower bound of the chunk's best score from the thread maxima;
            // a vector whose max z has z/T + kGumbelMax below it cannot win
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
                float x[VEC];
                E::unpack(v, x);
                const int32_t base = g.a0 + i * VEC;
                if (whole_blocks) {
                    score_vec<VEC>(x, vm, base, invT, nz, best, bi);
                } else {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) keep_best(nz.score(x[q], base + q, invT), base + q, best, bi);
                }
            }
            if (tid < g.n_extra)
                keep_best(nz.score(sh.extras_v[tid], sh.extras_i[tid], invT), sh.extras_i[tid], best, bi);
            block_best(best, bi, sh);
            if (tid == 0) { sh.part.gbest = best; sh.part.gidx = bi; }
        } else {
            // level the candidates lie above: min-p relative to the chunk
            // maximum (<= the row maximum); for top-k the exact k-th largest
            // thread maximum (the ladder above the thread count); pure top-p
            // keeps a short list used when it covers the nucleus boundary
            float lo = use_m ? m_c + T * logf(info.min_p) : -INFINITY;
            bool bounded = use_m;
            const int kk = use_k ? info.top_k : (pure_p ? kPureListK : 0);
            if (kk > 0) {
                if (kk <= kThreads) {
                    lo = fmaxf(lo, kth_thread_max<E>(thread_max, kk, m_c, sh));
                    bounded = true;
                } else {
                    float tlo = -INFINITY;
                    if (kth_level(thread_max, m_c, kk, tlo, sh)) {
                        lo = fmaxf(lo, tlo);
                        bounded = true;
                    }
                }
            }
            int n = INT_MAX;                     // unbounded: overflow marker
            if (bounded) {
                if (tid == 0) sh.cand_n = 0;
                __syncthreads();
                // count this thread's elements >= lo and remember which of
                // its vectors hold them (compares only), reserve a range per
                // warp with one atomic, then re-read just those vectors
                // (the vectors are screened first and only the few that
                // hold candidates are unpacked: a fused loop keeps the
                // rare per-element work on every iteration)
                uint32_t hits = 0;
                for (int i = tid, j = 0; i < g.nb; i += kThreads, ++j)
                    hits |= ((E::vmax(body[i]) >= lo) ? 1u : 0u) << j;
                int cnt = 0;
                for (uint32_t hh = hits; hh; hh &= hh - 1) {
                    float x[VEC];
                    E::unpack(body[tid + (__ffs(hh) - 1) * kThreads], x);
#pragma unroll
                    for (int q = 0; q < VEC; ++q) cnt += (x[q] >= lo) ? 1 : 0;
                }
                const bool xin = tid < g.n_extra && sh.extras_v[tid] >= lo;
                cnt += xin ? 1 : 0;
                int off = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, off, o);
                    if (lane >= o) off += y;
                }
                int base = 0;
                if (lane == 31 && off) base = atomicAdd(&sh.cand_n, off);
                base = __shfl_sync(0xFFFFFFFFu, base, 31);
                off += base - cnt;
                while (hits) {
                    const int j = __ffs(hits) - 1;
                    hits &= hits - 1;
                    const int i = tid + j * kThreads;
                    const uint4 v = body[i];
                    float x[VEC];
                    E::unpack(v, x);
#pragma unroll
                    for (int q = 0; q < VEC; ++q)
                        if (x[q] >= lo) {
                            if (off < kCandCap) { cand[off].v = x[q]; cand[off].i = g.a0 + i * VEC + q; }
                            ++off;
                        }
                }
                if (xin) {
                    if (off < kCandCap) { cand[off].v = sh.extras_v[tid]; cand[off].i = sh.extras_i[tid]; }
                    ++off;
                }
                __syncthreads();
                n = sh.cand_n;
                Cand *ws_list = reinterpret_cast<Cand *>(p.ws_cand) + rc * kCandCap;
                for (int i = tid; i < min(n, kCandCap); i += kThreads) ws_list[i] = cand[i];
            }
            if (tid == 0) { sh.part.ncand = n; sh.part.lev = lo; }
            if (pure_p) {
                // mass exp((z - m_c)/T) on the absolute grid; bin t (0 =
                // the chunk max's bin) holds its elements' weights scaled by
                // e^(t/8), which keeps each in (e^-1/8, e^1/8), as 2^20
                // fixed point per warp (no float atomics); the rest of the
                // mass is summed in registers
                for (int q = tid; q < kWarps * kBins; q += kThreads) wbins[q] = 0u;
                __syncthreads();
                const float s8 = bin_scale(T);
                const int32_t jt = abs_bin(m_c, s8);
                uint32_t *mine = wbins + warp * kBins;
                float tail = 0.f;
                if (jt >= -(1 << 21) && jt <= (1 << 21)) {
                    // Integer parts without conversions: for |u| < 2^22,
                    // u + 1.5*2^23 rounded down is floor(u) + 1.5*2^23, an
                    // integer in [2^23, 2^24) whose bit pattern differs from
                    // the constant's by floor(u).  u = z*s8 rounded as in
                    // abs_bin, raised to jt - 2*kBins (those values land in
                    // the tail either way), so the bin equals abs_bin(z).
                    // The fixed-point weight uses the same trick with
                    // round-to-nearest (w < 4 here).
                    const float ulo = static_cast<float>(jt - 2 * kBins);
                    const float yt = static_cast<float>(jt) + kMagic;
                    const uint32_t ytb = __float_as_uint(yt);
                    const uint64_t s8_2 = f2_pack(s8, s8), mg2 = f2_pack(kMagic, kMagic);
                    const uint64_t yt2 = f2_pack(yt, yt), m1_2 = f2_pack(-1.f, -1.f);
                    const uint64_t nm2 = f2_pack(-m_c, -m_c), sc2 = f2_pack(sc, sc);
                    const float c8 = kLog2e / kBinsPerT;
                    const uint64_t c8_2 = f2_pack(c8, c8);
                    auto bin_add = [&](float w, uint32_t t) {
                        if (t < static_cast<uint32_t>(kBins))
                            atomicAdd(mine + t, __float_as_uint(fmaf(w, kFix, kMagic)) - __float_as_uint(kMagic));
                        else
                            tail += w;
                    };
                    auto bin_pair = [&](uint64_t xx) {
                        float u0, u1;
                        f2_unpack(f2_mul(xx, s8_2), u0, u1);
                        const uint64_t y = f2_add_rm(f2_pack(fmaxf(u0, ulo), fmaxf(u1, ulo)), mg2);
                        const uint64_t ds = f2_mul(f2_add(xx, nm2), sc2);
                        const uint64_t in = f2_fma(f2_fma(y, m1_2, yt2), c8_2, ds);
                        float y0, y1, a0, a1, b0, b1;
                        f2_unpack(y, y0, y1);
                        f2_unpack(in, a0, a1);
                        f2_unpack(ds, b0, b1);
                        const uint32_t t0 = ytb - __float_as_uint(y0), t1 = ytb - __float_as_uint(y1);
                        bin_add(ex2(t0 < static_cast<uint32_t>(kBins) ? a0 : b0), t0);
                        bin_add(ex2(t1 < static_cast<uint32_t>(kBins) ? a1 : b1), t1);
                    };
                    for (int i = tid; i < g.nb; i += kThreads) {
                        const uint4 v = body[i];
                        if constexpr (E::BYTES == 2) {
                            bin_pair(f2_pack(bf_lo(v.x), bf_hi(v.x)));
                            bin_pair(f2_pack(bf_lo(v.y), bf_hi(v.y)));
                            bin_pair(f2_pack(bf_lo(v.z), bf_hi(v.z)));
                            bin_pair(f2_pack(bf_lo(v.w), bf_hi(v.w)));
                        } else {
                            bin_pair(f2_pack(__uint_as_float(v.x), __uint_as_float(v.y)));
                            bin_pair(f2_pack(__uint_as_float(v.z), __uint_as_float(v.w)));
                        }
                    }
                    if (tid < g.n_extra) {
                        const float xv = sh.extras_v[tid];
                        const float y0 = __fadd_rd(fmaxf(xv * s8, ulo), kMagic);
                        const uint32_t t0 = ytb - __float_as_uint(y0);
                        const float d = (xv - m_c) * sc;
                        bin_add(ex2(t0 < static_cast<uint32_t>(kBins) ? fmaf(yt - y0, c8, d) : d), t0);
                    }
                } else {
                    // no bin resolution at this grid origin: the chunk's
                    // mass only (the combine treats the row as binless)
                    visit_chunk([&](float v, int32_t) { tail += ex2((v - m_c) * sc); }, -INFINITY);
                }
                __syncthreads();
                float mass = 0.f;
                if (tid < kBins) {
                    uint64_t s = 0;
                    for (int w = 0; w < kWarps; ++w) s += wbins[w * kBins + tid];
                    mass = static_cast<float>(s) * (1.0f / kFix) *
                           ex2(-static_cast<float>(tid) * (kLog2e / kBinsPerT));
                    p.ws_bins[rc * kBins + tid] = mass;
                }
                const float Wc = block_sum(mass + tail, sh);
                if (tid == 0) {
                    sh.part.gbest = Wc;
                    // grid origins beyond 2^21 lose the bin resolution
                    sh.part.gidx = (jt > (1 << 21) || jt < -(1 << 21)) ? kNoBins : jt;
                }
            }
        }
        __syncthreads();
    }
    if (tid == 0) reinterpret_cast<ChunkPart *>(p.ws_part)[rc] = sh.part;
}

// ------------------------------------------------------ row helpers ------

// Visit every element of a row with value >= thr as fn(value, index): the
// aligned body streams through two shared-memory stages by TMA bulk copies
// (phase bits in ph), the unaligned head / tail use plain loads.  Called by
// all threads of the CTA.
template <typename E, typename F>
__device__ void visit_row(const void *row_v, int V, int h, uint8_t *stage_mem, Shared &sh,
                          uint32_t *ph, float thr, F &&fn)
{
    using T = typename std::conditional<E::BYTES == 2, uint16_t, float>::type;
    constexpr int VEC = E::VEC;
    constexpr int PER = kRowStage / 16;
    const T *row = reinterpret_cast<const T *>(row_v);
    const int tid = threadIdx.x;
    const int nv = (V - h) / VEC;
    const int npieces = (nv + PER - 1) / PER;
    const uint4 *src = reinterpret_cast<const uint4 *>(row + h);
    auto issue = [&](int q) {
        const int s = q & 1;
        const uint32_t bytes = static_cast<uint32_t>(min(PER, nv - q * PER)) * 16u;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&sh.mbar[s], bytes);
        bulk_g2s(stage_mem + s * kRowStage, src + static_cast<int64_t>(q) * PER, bytes, &sh.mbar[s]);
    };
    if (tid == 0)
        for (int q = 0; q < min(2, npieces); ++q) issue(q);
    for (int q = 0; q < npieces; ++q) {
        const int s = q & 1;
        if (tid == 0 && !mbar_wait(&sh.mbar[s], ph[s])) sh.timeout = 1;
        __syncthreads();
        const uint4 *buf = reinterpret_cast<const uint4 *>(stage_mem + s * kRowStage);
        const int n = min(PER, nv - q * PER), base = h + q * PER * VEC;
        for (int i = tid; i < n; i += kThreads) {
            const uint4 v = buf[i];
            if (!(E::vmax(v) >= thr)) continue;
            float x[VEC];
            E::unpack(v, x);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (x[j] >= thr) fn(x[j], base + i * VEC + j);
        }
        __syncthreads();
        if (tid == 0) {
            ph[s] ^= 1u;
            if (q + 2 < npieces) issue(q + 2);
        }
    }
    const int t0 = h + nv * VEC;
    if (tid < h) { const float v = E::load(row, tid); if (v >= thr) fn(v, tid); }
    if (tid < V - t0) { const float v = E::load(row, t0 + tid); if (v >= thr) fn(v, t0 + tid); }
}

// Filter parameters of a sampler row, as every row kernel reads them.
struct Filter {
    float T, invT, sc;
    bool use_k, use_m, use_p, unfiltered, pure_p;
    __device__ __forceinline__ Filter(const RowInfo &info, int V)
    {
        T = info.T;
        invT = 1.0f / T;
        sc = invT * kLog2e;
        use_k = info.top_k > 0 && info.top_k < V;
        use_m = info.min_p > 0.f;
        use_p = info.top_p < 1.f;
        unfiltered = !use_k && !use_m && !use_p;
        pure_p = !use_k && !use_m && use_p;
    }
};

// The sampled token of a row from exact selects over the whole row (one
// CTA; the fallback when candidate lists or bands overflow): survivors of
// top-k and min-p {z >= th_S}, the nucleus of their mass {z >= th_F}, then
// Gumbel-max over it.  Returns INT_MAX when nothing survives.
template <typename E>
__device__ int32_t exact_row_token(const void *row, int V, int h, float M, const RowInfo &info,
                                   const Noise &nz, uint8_t *stage_mem, Shared &sh, uint32_t *ph)
{
    const Filter f(info, V);
    const uint32_t keyM = fkey(M);
    auto visit_all = [&](auto &&fn, float thr) {
        visit_row<E>(row, V, h, stage_mem, sh, ph, thr, fn);
    };
    uint32_t key_S = f.use_m ? fkey(M + f.T * logf(info.min_p)) : 0u;
    if (f.use_k)
        key_S = max(key_S, select_key<E, false>(visit_all, key_S, keyM, 0.f,
                                                static_cast<uint32_t>(info.top_k), M, f.sc, sh));
    uint32_t key_F = key_S;
    if (f.use_p) {
        float w = 0.f;
        const uint32_t kS = key_S;
        visit_all([&](float v, int32_t) {
            if (fkey(v) >= kS) w += ex2((v - M) * f.sc);
        }, key_floor(key_S));
        const float Wt = block_sum(w, sh);
        key_F = max(key_S, select_key<E, true>(visit_all, key_S, keyM, info.top_p * Wt, 0u, M,
                                               f.sc, sh));
    }
    GumbelScorer gs{f.invT, nz, 0xFFFFFFFFu, make_uint4(0, 0, 0, 0)};
    float best = -INFINITY;
    int32_t bi = INT_MAX;
    const uint32_t kF = key_F;
    visit_all([&](float v, int32_t ix) {
        if (fkey(v) >= kF) keep_best(gs(v, ix), ix, best, bi);
    }, key_floor(key_F));
    block_best(best, bi, sh);
    return bi;
}

// The request chain, run by warp 0 of the CTA that settles row r's token:
// the CTA finishing the last row of the request (atomic ticket) runs the
// accept-while-equal prefix scan with one ballot and writes the request's
// tokens and the optional prefix-acceptance counters.
template <int MODE>
__device__ __forceinline__ void request_chain(const VerifyParams &p, const RowInfo &info, int r)
{
    const int lane = threadIdx.x & 31;
    uint32_t t = 0;
    if (lane == 0) {
        fence_acq_rel_gpu();
        t = atomicAdd(p.ws_ticket + info.b, 1u);
        if (t == static_cast<uint32_t>(info.k_b)) fence_acq_rel_gpu();
    }
    t = __shfl_sync(0xFFFFFFFFu, t, 0);
    if (t != static_cast<uint32_t>(info.k_b)) return;
    const int b = info.b, k = info.k_b, r0 = r - info.pos;
    const int j = lane;
    const int32_t yj = (j <= k) ? __ldcg(p.ws_tok + r0 + j) : -1;
    const int32_t dj = (j < k) ? __ldg(p.draft_ids + r0 + j) : -1;
    bool ok;
    if (MODE == MODE_RELAXED || (MODE == MODE_GREEDY && p.margin))
        ok = (j < k) && __ldcg(p.ws_flag + r0 + j) != 0;
    else ok = (j < k) && (yj == dj);
    const unsigned mism = __ballot_sync(0xFFFFFFFFu, (j < k) && !ok);
    const int a = mism ? (__ffs(mism) - 1) : k;
    const int32_t tok = __shfl_sync(0xFFFFFFFFu, yj, a);
    if (j <= p.k_max)
        p.out_tokens[static_cast<int64_t>(b) * (p.k_max + 1) + j] = (j < a) ? dj : (j == a ? tok : -1);
    if (j == 0) {
        p.accepted_len[b] = a;
        p.next_token[b] = tok;
        p.ws_ticket[b] = 0u;
        set_status(p.status, static_cast<uint32_t>(info.bad));
        if (p.hist) atomicAdd(reinterpret_cast<unsigned long long *>(p.hist + a), 1ull);
    }
    if (j < p.k_max) {
        if (p.acc && a > j) atomicAdd(reinterpret_cast<unsigned long long *>(p.acc + j), 1ull);
        if (p.ver && k > j) atomicAdd(reinterpret_cast<unsigned long long *>(p.ver + j), 1ull);
    }
}

// The key of the smallest bf16 value whose order-preserving key is >= k.
__device__ __forceinline__ uint32_t bf16_key_ceil(uint32_t k)
{
    const uint32_t h = k >> 16;
    const uint32_t full = (h << 16) | ((h & 0x8000u) ? 0u : 0xFFFFu);
    return (full >= k) ? h : h + 1u;
}

// Top-p over a set of bf16 values tallied per value (d = ktop - key, below
// kTally): a count and the best Gumbel score packed with its index.  Equal
// values share their weight exp((z - M)/T), so the running mass from the
// top value is exact per value group.  `visit` yields every value of the set
// (all values with key in [klo, ktop]); the target is frac times their total
// mass (frac > 0) or target_abs, which the total must exceed by kMassTol
// relative (else false: the set does not hold the boundary).  On success the
// best score among the values down to the boundary value is in best / bi.
template <typename Visit>
__device__ bool tally_top_p(Visit &&visit, uint32_t klo, uint32_t ktop, float M, float sc,
                            GumbelScorer &gs, float frac, float target_abs, uint32_t *cnt,
                            unsigned long long *bst, float &best, int32_t &bi, Shared &sh)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < kTally) { cnt[tid] = 0u; bst[tid] = 0ull; }
    __syncthreads();
    visit([&](float v, int32_t ix) {
        const uint32_t d = ktop - (fkey(v) >> 16);
        atomicAdd(cnt + d, 1u);
        atomicMax(bst + d, (static_cast<unsigned long long>(fkey(gs(v, ix))) << 32) |
                               static_cast<uint32_t>(~ix));
    }, key_floor((klo << 16) | ((klo & 0x8000u) ? 0u : 0xFFFFu)));
    __syncthreads();
    float w = 0.f;
    if (tid < kTally && cnt[tid]) {
        const uint32_t k = ktop - static_cast<uint32_t>(tid);
        w = static_cast<float>(cnt[tid]) * ex2((key_value((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu)) - M) * sc);
    }
    float cum = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xFFFFFFFFu, cum, o);
        if (lane >= o) cum += u;
    }
    float *wt = reinterpret_cast<float *>(sh.scan);
    if (lane == 31) wt[warp] = cum;
    __syncthreads();
    float total = 0.f;
    for (int w2 = 0; w2 < kTally / 32; ++w2) {
        if (w2 < warp) cum += wt[w2];
        total += wt[w2];
    }
    const float target = (frac > 0.f) ? frac * total : target_abs;
    const bool ok = (frac > 0.f) || total >= target_abs * (1.f + kMassTol);
    if (!ok) {
        __syncthreads();
        return false;
    }
    const int dstar = min(__syncthreads_count(tid < kTally && cum < target), kTally - 1);
    unsigned long long sb = (tid < kTally && tid <= dstar) ? bst[tid] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sb = max(sb, __shfl_xor_sync(0xFFFFFFFFu, sb, o));
    unsigned long long *wb = reinterpret_cast<unsigned long long *>(sh.hist);
    if (lane == 0) wb[warp] = sb;
    __syncthreads();
    sb = 0ull;
    for (int w2 = 0; w2 < kWarps; ++w2) sb = max(sb, wb[w2]);
    best = -INFINITY;
    bi = INT_MAX;
    if (sb != 0ull) {
        best = key_value(static_cast<uint32_t>(sb >> 32));
        bi = static_cast<int32_t>(~static_cast<uint32_t>(sb));
    }
    __syncthreads();
    return true;
}

// ------------------------------------------------------ finish kernel ----

// One CTA per packed row, after the stream kernel: combine the chunk
// summaries, pick the row's token, write the row results, run the chain;
// rows that need their logits again are queued for the heavy kernel.
template <typename TIn, int MODE>
__global__ void __launch_bounds__(kThreads, 5) finish_rows_kernel(const VerifyParams p)
{
    using E = Elt<TIn>;
    extern __shared__ __align__(128) uint8_t smem[];
    Shared &sh = *reinterpret_cast<Shared *>(smem);
    ChunkPart *parts = reinterpret_cast<ChunkPart *>(smem + sizeof(Shared));       // [kMaxChunks]
    Cand *band = reinterpret_cast<Cand *>(parts + kMaxChunks);                     // [kBandCap]
    Cand *lst = band + kBandCap;                                                   // [kListCap]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int nchunk = p.nchunk;

    griddep_launch_dependents();
    griddep_wait();                        // the stream kernel's stores are visible
    if (tid == 0) {
        if (MODE != MODE_CONF) {
            sh.info = reinterpret_cast<const RowInfo *>(p.ws_info)[r];
            sh.info.valid = sh.info.valid && r < min(__ldg(p.cu_rows + p.B), p.R_cap);
        } else {
            RowInfo inf = {};
            inf.b = r; inf.valid = 1;
            inf.sel = p.selected ? static_cast<uint32_t>(__ldg(p.selected + r)) : 0xFFFFFFFFu;
            sh.info = inf;
        }
        sh.heavy = 0;
    }
    if (tid < nchunk) {
        const ChunkPart *rp = reinterpret_cast<const ChunkPart *>(p.ws_part) + static_cast<int64_t>(r) * nchunk;
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(rp + tid));
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(rp + tid) + 1);
        ChunkPart cp;
        cp.m = a.x; cp.amax = __float_as_int(a.y); cp.s = a.z; cp.cnt = __float_as_int(a.w);
        cp.gbest = b.x; cp.gidx = __float_as_int(b.y); cp.ncand = __float_as_int(b.z); cp.lev = b.w;
        parts[tid] = cp;
    }
    __syncthreads();
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
            combine(m, a, s, cc, parts[q].m, parts[q].amax, parts[q].s, parts[q].cnt, need_sum);
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
    __syncthreads();
    const float M = sh.M;
    const int32_t AMAX = sh.AMAX;
    int32_t y = AMAX;
    int32_t flag = 0;
    if (MODE == MODE_RELAXED)
        flag = (info.draft >= 0 && info.draft < p.V && sh.CNT < info.K) ? 1 : 0;
    // margin: the first argmax, or a gap max - z[d] (fp32) within the margin
    if (MODE == MODE_GREEDY && p.margin)
        flag = (info.draft == AMAX || M - info.zd <= __ldg(p.margin + info.b)) ? 1 : 0;

    HeavyRec hrec = {};                    // thread 0: the queued row's record
    if (MODE == MODE_SAMPLE && info.T > 0.f && M > -INFINITY) {
        const Filter f(info, p.V);
        const float T = f.T, sc = f.sc;
        const uint32_t keyM = fkey(M);
        GumbelScorer gs{f.invT, Noise{static_cast<uint32_t>(info.pos), info.rid, p.step,
                                      info.seed_lo, info.seed_hi},
                        0xFFFFFFFFu, make_uint4(0, 0, 0, 0)};
        float best = -INFINITY;
        int32_t bi = INT_MAX;
        auto score_all = [&](float v, int32_t ix) { keep_best(gs(v, ix), ix, best, bi); };
        int heavy = 0;
        if (f.unfiltered) {
            for (int q = tid; q < nchunk; q += kThreads) keep_best(parts[q].gbest, parts[q].gidx, best, bi);
            block_best(best, bi, sh);
        } else {
            // candidate lists: offsets (a warp scan), overflow, the lowest
            // and highest levels they lie above
            if (warp == 0) {
                int tot = 0, ovf = 0;
                float th = -INFINITY, lmin = INFINITY;
                for (int q0 = 0; q0 < nchunk; q0 += 32) {
                    const int q = q0 + lane;
                    const bool on = q < nchunk && parts[q].m > -INFINITY;
                    const int nq = on ? parts[q].ncand : 0;
                    const int nc = min(nq, kCandCap);
                    int incl = nc;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    if (q < nchunk) sh.offs[q] = tot + incl - nc;
                    tot += __shfl_sync(0xFFFFFFFFu, incl, 31);
                    ovf |= static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, (on && nq > kCandCap) ? 1u : 0u));
                    th = fmaxf(th, warp_max_f32(on ? parts[q].lev : -INFINITY));
                    lmin = fminf(lmin, warp_min_f32(on ? parts[q].lev : INFINITY));
                }
                if (lane == 0) {
                    sh.offs[nchunk] = tot;
                    sh.total = tot;
                    sh.overflow = ovf;
                    sh.theta = th;
                    sh.lkey = (lmin == INFINITY) ? 0u : fkey(lmin);
                }
            }
            __syncthreads();
            const int n_list = sh.total;
            const bool staged = !sh.overflow && n_list <= kListCap;
            auto stage_lists = [&]() {
                // n_list <= kListCap: at most kListCap / kThreads entries per
                // thread, all loads issued before any is used
                constexpr int PER = kListCap / kThreads;
                const float2 *wl = reinterpret_cast<const float2 *>(p.ws_cand) +
                                   static_cast<int64_t>(r) * nchunk * kCandCap;
                float2 v[PER];
#pragma unroll
                for (int u = 0; u < PER; ++u) {
                    const int e = tid + u * kThreads;
                    if (e < n_list) {
                        int q = 0;
                        while (sh.offs[q + 1] <= e) ++q;
                        v[u] = __ldcg(wl + static_cast<int64_t>(q) * kCandCap + (e - sh.offs[q]));
                    }
                }
#pragma unroll
                for (int u = 0; u < PER; ++u) {
                    const int e = tid + u * kThreads;
                    if (e < n_list) {
                        lst[e].v = v[u].x;
                        lst[e].i = __float_as_int(v[u].y);
                    }
                }
                __syncthreads();
            };
            auto visit_lst = [&](auto &&fn, float thr) {
                for (int i = tid; i < n_list; i += kThreads) {
                    const Cand e = lst[i];
                    if (e.v >= thr) fn(e.v, e.i);
                }
            };
            // lists in global memory (more than fit on chip)
            auto visit_gl = [&](auto &&fn, float thr) {
                for (int q = 0; q < nchunk; ++q) {
                    if (!(parts[q].m > -INFINITY)) continue;
                    const int nq = min(parts[q].ncand, kCandCap);
                    const float2 *lq = reinterpret_cast<const float2 *>(p.ws_cand) +
                                       (static_cast<int64_t>(r) * nchunk + q) * kCandCap;
                    for (int i = tid; i < nq; i += kThreads) {
                        const float2 e = __ldcg(lq + i);
                        if (e.x >= thr) fn(e.x, __float_as_int(e.y));
                    }
                }
            };
            if (f.pure_p) {
                // ---- top-p alone: bracket the boundary with the bins ----
                const float s8 = bin_scale(T);
                if (warp == 0) {
                    // the row's mass, the highest grid origin, chunks without bins
                    float w = 0.f;
                    int32_t J = INT_MIN, nob = 0;
                    for (int q0 = 0; q0 < nchunk; q0 += 32) {
                        const int q = q0 + lane;
                        const bool on = q < nchunk && parts[q].m > -INFINITY;
                        float wq = on ? parts[q].gbest * ex2((parts[q].m - M) * sc) : 0.f;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) wq += __shfl_xor_sync(0xFFFFFFFFu, wq, o);
                        w += wq;
                        nob |= static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, (on && parts[q].gidx == kNoBins) ? 1u : 0u));
                        J = max(J, __reduce_max_sync(0xFFFFFFFFu, on ? parts[q].gidx : INT_MIN));
                    }
                    if (lane == 0) {
                        sh.W = w;
                        sh.J = J;
                        sh.nobins = nob;
                    }
                }
                __syncthreads();
                const float target = info.top_p * sh.W;
                const int32_t J = sh.J;
                bool settled = false, listed = false;
                if (E::BYTES == 2 && staged) {
                    // every value at or above the highest list level is
                    // listed: when they span at most kTally bf16 values and
                    // hold the target mass, their tally settles the row
                    const uint32_t klo = bf16_key_ceil(fkey(sh.theta)), ktop = keyM >> 16;
                    if (ktop >= klo && ktop - klo < static_cast<uint32_t>(kTally)) {
                        stage_lists();
                        listed = true;
                        uint32_t *cnt = reinterpret_cast<uint32_t *>(band);
                        settled = tally_top_p(visit_lst, klo, ktop, M, sc, gs, 0.f, target, cnt,
                                              reinterpret_cast<unsigned long long *>(cnt + kTally), best, bi, sh);
                    }
                }
                heavy = (!settled && sh.nobins) ? kHeavyWhole : 0;
                int32_t qin = 0, qband = 0;
                if (!settled && !heavy) {
                    // combined mass of absolute bin J - t, then C(t) = mass of
                    // bins J - t .. J (thread t)
                    // the row's bins staged in shared memory by all threads
                    // at once (the band and list scratch, 32 KiB, holds 64
                    // chunks of them)
                    float *sb = reinterpret_cast<float *>(band);
                    {
                        const float *rb = p.ws_bins + static_cast<int64_t>(r) * nchunk * kBins;
#pragma unroll 4
                        for (int i = tid; i < nchunk * kBins; i += kThreads) sb[i] = __ldcg(rb + i);
                    }
                    __syncthreads();
                    float hb = 0.f;
                    if (tid < kBins) {
                        for (int q = 0; q < nchunk; ++q) {
                            if (!(parts[q].m > -INFINITY)) continue;
                            const int tq = tid - (J - parts[q].gidx);
                            if (tq >= 0 && tq < kBins) hb += sb[q * kBins + tq] * ex2((parts[q].m - M) * sc);
                        }
                    }
                    float cum = hb;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float n = __shfl_up_sync(0xFFFFFFFFu, cum, o);
                        if (lane >= o) cum += n;
                    }
                    float *wt = reinterpret_cast<float *>(sh.scan);
                    if (lane == 31) wt[warp] = cum;
                    __syncthreads();
                    for (int w = 0; w < warp; ++w) cum += wt[w];
                    // bins 0..a are surely inside (mass above < target), bins
                    // from b on surely outside; the band between is settled
                    // exactly
                    const int n_in = __syncthreads_count(tid < kBins && cum < target * (1.f - kMassTol));
                    const int n_out = __syncthreads_count(tid < kBins && cum >= target * (1.f + kMassTol));
                    const int a = n_in - 1, b = kBins - n_out;
                    if (b >= kBins) heavy = kHeavyWhole;      // the nucleus reaches below the bins
                    qin = J - a;
                    qband = J - b;
                }
                // the lists cover the band when every value below the highest
                // list level falls in a bin below the band
                if (!settled && !heavy && !(staged && abs_bin(sh.theta, s8) < qband)) heavy = kHeavyBand;
                if (!settled && !heavy) {
                    if (!listed) stage_lists();
                    if (tid == 0) sh.cand_n = 0;
                    __syncthreads();
                    float mass_in = 0.f;
                    visit_lst([&](float v, int32_t ix) {
                        const int32_t qz = abs_bin(v, s8);
                        if (qz >= qin) {
                            mass_in += ex2((v - M) * sc);
                            score_all(v, ix);
                        } else if (qz >= qband) {
                            const int slot = warp_append(&sh.cand_n);
                            if (slot < kBandCap) { band[slot].v = v; band[slot].i = ix; }
                        }
                    }, -INFINITY);
                    mass_in = block_sum(mass_in, sh);
                    const int nband = min(sh.cand_n, kBandCap);
                    const float tgt = target - mass_in;
                    if (nband > 0 && tgt > 0.f) {
                        uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
                        for (int i = tid; i < nband; i += kThreads) {
                            const uint32_t k = fkey(band[i].v);
                            kmn = min(kmn, k);
                            kmx = max(kmx, k);
                        }
                        block_minmax(kmn, kmx, sh);
                        auto visit_band = [&](auto &&fn, float t2) {
                            for (int i = tid; i < nband; i += kThreads)
                                if (band[i].v >= t2) fn(band[i].v, band[i].i);
                        };
                        const uint32_t kF = select_key<E, true>(visit_band, kmn, kmx, tgt, 0u, M, sc, sh);
                        visit_band([&](float v, int32_t ix) {
                            if (fkey(v) >= kF) score_all(v, ix);
                        }, -INFINITY);
                    }
                    block_best(best, bi, sh);
                } else if (heavy && tid == 0) {
                    hrec.mode = heavy;
                    hrec.amax = AMAX;
                    hrec.qin = qin;
                    hrec.qband = qband;
                    hrec.M = M;
                    hrec.target = target;
                    if (heavy == kHeavyBand) {
                        hrec.zin = bin_floor_value(qin, s8);
                        hrec.zband = bin_floor_value(qband, s8);
                    }
                }
            } else if (sh.overflow) {
                // ---- top-k / min-p with an overflowed list ----
                heavy = kHeavyWhole;
                if (tid == 0) { hrec.mode = heavy; hrec.amax = AMAX; hrec.M = M; }
            } else {
                // ---- top-k and / or min-p (then top-p over the survivors) --
                if (staged) stage_lists();
                auto visit = [&](auto &&fn, float thr) {
                    if (staged) visit_lst(fn, thr);
                    else visit_gl(fn, thr);
                };
                const float th_m = f.use_m ? M + T * logf(info.min_p) : -INFINITY;
                uint32_t key_S = f.use_m ? fkey(th_m) : 0u;
                // every list element lies above its chunk's level
                const uint32_t lo_k = max(key_S, sh.lkey);
                if (f.use_k && n_list >= info.top_k)
                    key_S = max(key_S, select_key<E, false>(visit, lo_k, keyM, 0.f,
                                                            static_cast<uint32_t>(info.top_k), M,
                                                            sc, sh));
                bool tallied = false;
                if (E::BYTES == 2 && f.use_p) {
                    // the survivors tallied per value when they span at most
                    // kTally bf16 values
                    const uint32_t klo = bf16_key_ceil(key_S), ktop = keyM >> 16;
                    if (ktop >= klo && ktop - klo < static_cast<uint32_t>(kTally)) {
                        uint32_t *cnt = reinterpret_cast<uint32_t *>(band);
                        tally_top_p(visit, klo, ktop, M, sc, gs, info.top_p, 0.f, cnt,
                                    reinterpret_cast<unsigned long long *>(cnt + kTally), best, bi, sh);
                        tallied = true;
                    }
                }
                if (!tallied) {
                    uint32_t key_F = key_S;
                    if (f.use_p) {
                        float w = 0.f;
                        const uint32_t kS = key_S;
                        visit([&](float v, int32_t) {
                            if (fkey(v) >= kS) w += ex2((v - M) * sc);
                        }, key_floor(key_S));
                        const float Wt = block_sum(w, sh);
                        key_F = max(key_S, select_key<E, true>(visit, key_S, keyM, info.top_p * Wt, 0u,
                                                               M, sc, sh));
                    }
                    const uint32_t kF = key_F;
                    visit([&](float v, int32_t ix) {
                        if (fkey(v) >= kF) score_all(v, ix);
                    }, key_floor(key_F));
                    block_best(best, bi, sh);
                }
            }
        }
        if (heavy && tid == 0) {
            // queue the row: record in the row's bin area, then the list slot
            reinterpret_cast<HeavyRec *>(p.ws_bins + static_cast<int64_t>(r) * nchunk * kBins)[0] = hrec;
            const int slot = atomicAdd(p.ws_hrows, 1);
            p.ws_hrows[1 + slot] = r;
            sh.heavy = 1;
        }
        y = (bi == INT_MAX) ? AMAX : bi;
    }

    // ---------------------------------------------------- row results ---
    __syncthreads();
    const bool queued = sh.heavy != 0;
    if (tid == 0) {
        const float S = sh.S;
        if (p.row_max) p.row_max[r] = M;
        if (p.row_lse) p.row_lse[r] = (S > 0.f) ? M + logf(S) : -INFINITY;
        if (p.row_argmax) p.row_argmax[r] = AMAX;
        if (MODE == MODE_CONF) {
            const int32_t s = p.selected ? static_cast<int32_t>(info.sel) : AMAX;
            float cf = 0.f;
            if (s >= 0 && s < p.V) {
                const float zs = E::load(row, s);
                cf = (S > 0.f) ? ex2((zs - M) * kLog2e) / S : 0.f;
            } else {
                set_status(p.status, SPEC_STATUS_BAD_SELECTED);
            }
            p.conf[r] = cf;
            p.draft_token[r] = s;
        } else if (!queued) {
            // active vocabulary: the argmax column's full token id
            if (MODE == MODE_GREEDY && p.vocab_ids) y = __ldg(p.vocab_ids + AMAX);
            if (p.row_token) p.row_token[r] = y;
            p.ws_tok[r] = y;
            if (MODE == MODE_RELAXED || (MODE == MODE_GREEDY && p.margin)) p.ws_flag[r] = flag;
        }
    }
    if (MODE != MODE_CONF && !queued && warp == 0) request_chain<MODE>(p, info, r);
}

// ------------------------------------------------------- heavy kernel ----

// Persistent over the pieces (half-chunks) of the rows the finish kernel
// queued.  A row queued for its band: every piece is staged by TMA; its
// values at or above the band's upper edge are in the nucleus, the values in
// the band are collected; both are compacted in shared memory (counts, a CTA
// scan, a scatter: no per-element branches that diverge) and the nucleus is
// scored with all lanes busy; each piece's band values go to its own list,
// or to per-value tallies when a bf16 band spans at most kFineBand values.
// The CTA finishing the row's last piece (atomic ticket) settles the band
// (a scan of the tallies, or an exact mass select over the lists) and runs
// the request chain.  A row queued whole: the CTA of its first piece runs
// the exact selects over the row.
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 4) heavy_rows_kernel(const VerifyParams p)
{
    using E = Elt<TIn>;
    constexpr int VEC = E::VEC;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *chunk = smem;                                   // one piece; from here 32 KiB of row stages
    Cand *sure = reinterpret_cast<Cand *>(smem + kPieceBytes);                      // [kSureH]
    Cand *band = sure + kSureH;                                                     // [kBandCap]
    Shared &sh = *reinterpret_cast<Shared *>(band + kBandCap);
    __shared__ uint32_t ph[2];
    __shared__ HeavyRec rec_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = p.nchunk;
    const int npc = 2 * nchunk;             // pieces per row: the halves of its chunks

    griddep_wait();                         // the finish kernel's queue is complete
    const int n_heavy = __ldcg(p.ws_hrows);
    const int64_t n_items = static_cast<int64_t>(n_heavy) * npc;
    if (static_cast<int64_t>(blockIdx.x) >= n_items) return;
    if (tid == 0) {
        mbar_init(&sh.mbar[0], 1);
        mbar_init(&sh.mbar[1], 1);
        fence_mbar_init();
        ph[0] = ph[1] = 0u;
        sh.timeout = 0;
    }
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int hr = static_cast<int>(it / npc);
        const int pc = static_cast<int>(it - static_cast<int64_t>(hr) * npc);
        const int c = pc >> 1, half = pc & 1;
        const int r = __ldcg(p.ws_hrows + 1 + hr);
        float *area = p.ws_bins + static_cast<int64_t>(r) * nchunk * kBins;
        const TIn *row = reinterpret_cast<const TIn *>(p.logits) + static_cast<int64_t>(r) * p.ld;
        ChunkGeom g = chunk_geom<E>(row, c, p.V);
        // this half of the chunk's body: vectors [pv0, pv0 + g.nb) after the
        // split; the chunk's unaligned head and tail go with half 0
        const int nb0 = (g.nb + 1) / 2;
        const int pv0 = half ? nb0 : 0;
        g.nb = half ? g.nb - nb0 : nb0;
        if (half) g.n_extra = 0;
        const int32_t a0p = g.a0 + pv0 * VEC;
        if (tid == 0) {
            // the piece's copy first (in bounds for any queued row), then the
            // row's record and parameters while it is in flight
            const uint32_t bytes = static_cast<uint32_t>(g.nb) * 16u;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sh.mbar[0], bytes);
            if (bytes) bulk_g2s(chunk, row + a0p, bytes, &sh.mbar[0]);
            sh.info = reinterpret_cast<const RowInfo *>(p.ws_info)[r];
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(area));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(area) + 1);
            rec_s.mode = __float_as_int(a.x);
            rec_s.qin = __float_as_int(a.y);
            rec_s.qband = __float_as_int(a.z);
            rec_s.amax = __float_as_int(a.w);
            rec_s.M = b.x;
            rec_s.target = b.y;
            rec_s.zin = b.z;
            rec_s.zband = b.w;
            sh.last = 0;
        }
        float xe = -INFINITY;
        int32_t ie = INT_MAX;
        if (tid < g.n_extra) {
            ie = (tid < g.n_head) ? g.e0 + tid : g.a1 + (tid - g.n_head);
            xe = E::load(row, ie);
        }
        if (tid == 0) {
            if (!mbar_wait(&sh.mbar[0], ph[0])) {
                sh.timeout = 1;
                set_status(p.status, SPEC_STATUS_TIMEOUT);
            }
            ph[0] ^= 1u;
        }
        __syncthreads();
        const RowInfo info = sh.info;
        const HeavyRec rec = rec_s;
        const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(row) & 15u);
        const int h = min(mis ? static_cast<int>((16u - mis) / E::BYTES) : 0, p.V);
        const Noise nz{static_cast<uint32_t>(info.pos), info.rid, p.step, info.seed_lo, info.seed_hi};
        const Filter f(info, p.V);
        const float M = rec.M;
        int32_t y = INT_MAX;
        bool settle = false;
        if (rec.mode == kHeavyWhole) {
            if (pc == 0) {
                y = exact_row_token<E>(row, p.V, h, M, info, nz, chunk, sh, ph);
                settle = true;
            }
        } else {
            // ---- one piece of a band row ----
            const float sc = f.sc;
            const float zin = rec.zin, zband = rec.zband;
            float2 *blist = reinterpret_cast<float2 *>(p.ws_cand) +
                            static_cast<int64_t>(r) * nchunk * kCandCap;
            // A bf16 band of at most kFineBand distinct values (keys kt - d)
            // is tallied per value instead of listed: equal values share
            // their weight, so a count and the best Gumbel score with its
            // index settle the band exactly.
            const uint32_t kt = fkey(zin) >> 16, kb = fkey(zband) >> 16;
            const bool fine = E::BYTES == 2 && kt >= kb && kt - kb < static_cast<uint32_t>(kFineBand);
            uint32_t *fcnt = reinterpret_cast<uint32_t *>(band);                            // [kFineBand]
            unsigned long long *fbst = reinterpret_cast<unsigned long long *>(fcnt + kFineBand);
            if (fine && tid < kFineBand) { fcnt[tid] = 0u; fbst[tid] = 0ull; }
            auto band_take = [&](float v, int32_t ix) {
                if (fine) {
                    const uint32_t d = kt - (fkey(v) >> 16);
                    atomicAdd(fcnt + d, 1u);
                    atomicMax(fbst + d, (static_cast<unsigned long long>(fkey(nz.score(v, ix, f.invT))) << 32) |
                                            static_cast<uint32_t>(~ix));
                } else {
                    const int slot = warp_append(&sh.total);
                    if (slot < kPieceList) { band[slot].v = v; band[slot].i = ix; }
                }
            };
            float mass = 0.f, best = -INFINITY;
            int32_t bi = INT_MAX;
            const uint4 *body = reinterpret_cast<const uint4 *>(chunk);
            // count this thread's values >= zband (one compare each) and mark
            // the vectors that hold them; a CTA scan gives each thread its
            // range of `sure`; the marked vectors are read again to scatter
            uint32_t hits = 0;
            for (int i = tid, j = 0; i < g.nb; i += kThreads, ++j)
                hits |= ((E::vmax(body[i]) >= zband) ? 1u : 0u) << j;
            int cnt = 0;
            for (uint32_t hh = hits; hh; hh &= hh - 1) {
                float x[VEC];
                E::unpack(body[tid + (__ffs(hh) - 1) * kThreads], x);
#pragma unroll
                for (int q = 0; q < VEC; ++q) cnt += (x[q] >= zband) ? 1 : 0;
            }
            const bool xin = tid < g.n_extra && xe >= zband;
            cnt += xin ? 1 : 0;
            int off = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, off, o);
                if (lane >= o) off += y;
            }
            if (lane == 31) sh.red_i[warp] = off;
            if (tid == 0) sh.total = 0;
            __syncthreads();
            int tot = 0;
            for (int w = 0; w < kWarps; ++w) {
                if (w < warp) off += sh.red_i[w];
                tot += sh.red_i[w];
            }
            off -= cnt;
            // scatter into `sure` up to its capacity (a plain store per value)
            const uint32_t hits0 = hits;
            const int off0 = off;
            while (hits) {
                const int j = __ffs(hits) - 1;
                hits &= hits - 1;
                const int i = tid + j * kThreads;
                const uint4 v = body[i];
                float x[VEC];
                E::unpack(v, x);
#pragma unroll
                for (int q = 0; q < VEC; ++q)
                    if (x[q] >= zband) {
                        if (off < kSureH) { sure[off].v = x[q]; sure[off].i = a0p + i * VEC + q; }
                        ++off;
                    }
            }
            if (xin) {
                if (off < kSureH) { sure[off].v = xe; sure[off].i = ie; }
                ++off;
            }
            if (tot > kSureH) {
                // rare: the values past the buffer are handled where they are
                auto direct = [&](float v, int32_t ix) {
                    if (v >= zin) {
                        mass += ex2((v - M) * sc);
                        keep_best(nz.score(v, ix, f.invT), ix, best, bi);
                    } else {
                        band_take(v, ix);
                    }
                };
                int o2 = off0;
                uint32_t hh = hits0;
                while (hh) {
                    const int j = __ffs(hh) - 1;
                    hh &= hh - 1;
                    const int i = tid + j * kThreads;
                    const uint4 v = body[i];
                    float x[VEC];
                    E::unpack(v, x);
                    for (int q = 0; q < VEC; ++q)
                        if (x[q] >= zband) {
                            if (o2 >= kSureH) direct(x[q], a0p + i * VEC + q);
                            ++o2;
                        }
                }
                if (xin && o2 >= kSureH) direct(xe, ie);
            }
            __syncthreads();
            // the collected values with all lanes busy: nucleus values add
            // their mass and their Gumbel score, band values go to the band
            const int n_sel = min(tot, kSureH);
            for (int i = tid; i < n_sel; i += kThreads) {
                const Cand e = sure[i];
                if (e.v >= zin) {
                    mass += ex2((e.v - M) * sc);
                    keep_best(nz.score(e.v, e.i, f.invT), e.i, best, bi);
                } else {
                    band_take(e.v, e.i);
                }
            }
            __syncthreads();
            // the piece's band values (or tallies) to its own list space (no
            // global atomics)
            const int tb = sh.total;
            float2 *clist = blist + static_cast<int64_t>(pc) * kPieceList;
            if (fine) {
                uint32_t *oc = reinterpret_cast<uint32_t *>(clist);
                if (tid < kFineBand) {
                    oc[tid] = fcnt[tid];
                    reinterpret_cast<unsigned long long *>(oc + kFineBand)[tid] = fbst[tid];
                }
            } else {
                for (int i = tid; i < min(tb, kPieceList); i += kThreads)
                    clist[i] = make_float2(band[i].v, __int_as_float(band[i].i));
            }
            block_best(best, bi, sh);
            mass = block_sum(mass, sh);
            if (tid == 0) {
                HeavyPart hp;
                hp.best = best;
                hp.bi = bi;
                hp.mass = mass;
                hp.nband = tb;
                reinterpret_cast<HeavyPart *>(area + 8)[pc] = hp;
                // publish the piece's results and list, then count
                fence_acq_rel_gpu();
                const uint32_t t = atomicAdd(p.ws_rticket + r, 1u);
                if (t == static_cast<uint32_t>(npc - 1)) {
                    fence_acq_rel_gpu();
                    sh.last = 1;
                }
            }
            __syncthreads();
            if (sh.last) {
                // ---- the row's last piece: settle the band ----
                // the row's piece results, loaded by one thread each
                float4 *hps = reinterpret_cast<float4 *>(band);
                if (tid < npc)
                    hps[tid] = __ldcg(reinterpret_cast<const float4 *>(reinterpret_cast<const HeavyPart *>(area + 8) + tid));
                __syncthreads();
                if (tid == 0) {
                    float bsum = 0.f, bb = -INFINITY;
                    int32_t bbi = INT_MAX, tot = 0, ovf = 0;
                    for (int q = 0; q < npc; ++q) {
                        const float4 e = hps[q];
                        bsum += e.z;
                        keep_best(e.x, __float_as_int(e.y), bb, bbi);
                        const int nq = __float_as_int(e.w);
                        sh.offs[q] = tot;
                        ovf |= (nq > kPieceList);
                        tot += min(nq, kPieceList);
                    }
                    sh.offs[npc] = tot;
                    sh.W = bsum;
                    sh.red_f[0] = bb;
                    sh.red_i[0] = bbi;
                    sh.total = tot;
                    sh.overflow = ovf;
                    p.ws_rticket[r] = 0u;
                }
                __syncthreads();
                const float mass_in = sh.W;
                best = sh.red_f[0];
                bi = sh.red_i[0];
                const int nband = sh.total;
                const bool ovf = sh.overflow != 0;
                __syncthreads();
                if (fine) {
                    // per value: the pieces' counts and best scores; the
                    // running band mass from the top value first reaches
                    // the target at the boundary value (all values when
                    // rounding keeps it short); the best score among the
                    // values down to it joins the nucleus's
                    const float tgt = rec.target - mass_in;
                    uint32_t n = 0;
                    unsigned long long bb = 0ull;
                    if (tid < kFineBand) {
                        for (int q = 0; q < npc; ++q) {
                            const uint32_t *oc = reinterpret_cast<const uint32_t *>(blist + static_cast<int64_t>(q) * kPieceList);
                            n += __ldcg(oc + tid);
                            bb = max(bb, __ldcg(reinterpret_cast<const unsigned long long *>(oc + kFineBand) + tid));
                        }
                    }
                    float w = 0.f;
                    if (n) {
                        const uint32_t k = kt - static_cast<uint32_t>(tid);
                        const float v = key_value((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu));
                        w = static_cast<float>(n) * ex2((v - M) * sc);
                    }
                    float cum = w;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float u = __shfl_up_sync(0xFFFFFFFFu, cum, o);
                        if (lane >= o) cum += u;
                    }
                    float *wt = reinterpret_cast<float *>(sh.scan);
                    if (lane == 31) wt[warp] = cum;
                    __syncthreads();
                    for (int w2 = 0; w2 < warp; ++w2) cum += wt[w2];
                    const int dstar = min(__syncthreads_count(tid < kFineBand && cum < tgt), kFineBand - 1);
                    unsigned long long sb = (tgt > 0.f && tid <= dstar) ? bb : 0ull;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) sb = max(sb, __shfl_xor_sync(0xFFFFFFFFu, sb, o));
                    unsigned long long *wb = reinterpret_cast<unsigned long long *>(sh.hist);
                    if (lane == 0) wb[warp] = sb;
                    __syncthreads();
                    sb = 0ull;
                    for (int w2 = 0; w2 < kWarps; ++w2) sb = max(sb, wb[w2]);
                    if (sb != 0ull)
                        keep_best(key_value(static_cast<uint32_t>(sb >> 32)), static_cast<int32_t>(~static_cast<uint32_t>(sb)),
                                  best, bi);
                    y = bi;
                } else if (ovf || nband > kBandCap) {
                    y = exact_row_token<E>(row, p.V, h, M, info, nz, chunk, sh, ph);
                } else {
                    const float tgt = rec.target - mass_in;
                    if (nband > 0 && tgt > 0.f) {
                        for (int e = tid; e < nband; e += kThreads) {
                            int q = 0;
                            while (sh.offs[q + 1] <= e) ++q;
                            const float2 v = __ldcg(blist + static_cast<int64_t>(q) * kPieceList + (e - sh.offs[q]));
                            band[e].v = v.x;
                            band[e].i = __float_as_int(v.y);
                        }
                        __syncthreads();
                        uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
                        for (int i = tid; i < nband; i += kThreads) {
                            const uint32_t k = fkey(band[i].v);
                            kmn = min(kmn, k);
                            kmx = max(kmx, k);
                        }
                        block_minmax(kmn, kmx, sh);
                        auto visit_band = [&](auto &&fn, float t2) {
                            for (int i = tid; i < nband; i += kThreads)
                                if (band[i].v >= t2) fn(band[i].v, band[i].i);
                        };
                        const uint32_t kF = select_key<E, true>(visit_band, kmn, kmx, tgt, 0u, M, sc, sh);
                        visit_band([&](float v, int32_t ix) {
                            if (fkey(v) >= kF) keep_best(nz.score(v, ix, f.invT), ix, best, bi);
                        }, -INFINITY);
                    }
                    block_best(best, bi, sh);
                    y = bi;
                }
                settle = true;
            }
        }
        if (settle) {
            if (y == INT_MAX) y = rec.amax;
            if (tid == 0) {
                if (p.row_token) p.row_token[r] = y;
                p.ws_tok[r] = y;
                if (sh.timeout) set_status(p.status, SPEC_STATUS_TIMEOUT);
            }
            __syncthreads();
            if (warp == 0) request_chain<MODE_SAMPLE>(p, info, r);
        }
        __syncthreads();
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
    size_t smem = kChunkBytes + sizeof(Shared);
    if (MODE == MODE_SAMPLE)
        smem += static_cast<size_t>(kCandCap) * sizeof(Cand) + static_cast<size_t>(kWarps) * kBins * 4;
    const size_t smem_fin = sizeof(Shared) + kMaxChunks * sizeof(ChunkPart) +
                            static_cast<size_t>(kBandCap + kListCap) * sizeof(Cand);
    const size_t smem_heavy = kPieceBytes + sizeof(Shared) +
                              static_cast<size_t>(kSureH + kBandCap) * sizeof(Cand);
    auto kstream = stream_chunks_kernel<TIn, MODE>;
    auto kfin = finish_rows_kernel<TIn, MODE>;
    auto kheavy = heavy_rows_kernel<TIn>;
    // raise the dynamic shared-memory limits, prefer shared memory over L1
    // (the row kernels want as many resident CTAs as it allows) and read the
    // SM count, once per device
    static bool done[64] = {false};
    static int sms[64] = {0};
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
                                 static_cast<int>(smem_fin));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kfin, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        if (MODE == MODE_SAMPLE) {
            e = cudaFuncSetAttribute(kheavy, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_heavy));
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kheavy, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    const int nsm = sms[dev] > 0 ? sms[dev] : 1;
    const int rows = (MODE == MODE_CONF) ? p.n_rows : p.R_cap;
    if (MODE != MODE_CONF) {
        const int row_blocks = static_cast<int>((static_cast<int64_t>(p.R_cap) * 32 + 255) / 256);
        const int req_blocks = (p.B + 255) / 256;
        row_info_kernel<TIn, MODE><<<row_blocks + req_blocks, 256, 0, stream>>>(p, row_blocks);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // one CTA per (row, chunk); the entry points bound rows * nchunk by 2^31 - 1
    cudaLaunchConfig_t cfg = {};
    if (MODE == MODE_SAMPLE)
        cfg.gridDim = dim3(static_cast<unsigned>(rows), static_cast<unsigned>(p.nchunk), 1);
    else if (rows <= 65535)
        cfg.gridDim = dim3(static_cast<unsigned>(p.nchunk), static_cast<unsigned>(rows), 1);
    else
        cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(rows) * p.nchunk), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = (MODE != MODE_CONF) ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kstream, p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cf = {};
    cf.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cf.blockDim = dim3(kThreads, 1, 1);
    cf.dynamicSmemBytes = smem_fin;
    cf.stream = stream;
    cf.attrs = attr;
    cf.numAttrs = 1;
    e = cudaLaunchKernelEx(&cf, kfin, p);
    if (e != cudaSuccess || MODE != MODE_SAMPLE) return e;
    // heavy rows: persistent over the pieces of whatever the finish kernel queued
    cudaLaunchConfig_t ch = {};
    ch.gridDim = dim3(static_cast<unsigned>(4 * nsm), 1, 1);
    ch.blockDim = dim3(kThreads, 1, 1);
    ch.dynamicSmemBytes = smem_heavy;
    ch.stream = stream;
    ch.attrs = attr;
    ch.numAttrs = 1;
    return cudaLaunchKernelEx(&ch, kheavy, p);
}

cudaError_t launch_verify(int mode, int dtype, const VerifyParams &p, cudaStream_t stream)
{
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
