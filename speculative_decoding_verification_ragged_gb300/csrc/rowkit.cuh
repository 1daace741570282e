// rowkit.cuh -- block-level building blocks of the verification kernels
// (sm_103a): row records and chunk summaries, CTA reductions, radix selects
// over order-preserving value keys, Philox4x32-10 Gumbel noise, the fused
// pass 1 (max / first argmax / sum of exponentials / relaxed count), chunk
// geometry, a row-streaming visitor with 1-D TMA bulk copies, the exact
// whole-row sampler and the request chain.
//
// Every function here is called by all kThreads threads of a CTA unless its
// comment says otherwise; functions that synchronise use csync().
#pragma once

#include <cfloat>
#include <climits>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace specv {

constexpr int kCandCap = kWsCandCap;    // candidates one chunk may store
constexpr int kListCap = 2048;          // candidates a finishing CTA stages on chip
constexpr int kTally = 128;             // bf16 values a top-p tally over the survivors covers
constexpr int kRowStage = 16 * 1024;    // bytes per stage when a CTA streams a whole row
constexpr int kPureListK = 64;          // fp32 top-p alone: candidates above the 64-th thread maximum
constexpr float kMassTol = 1e-5f;       // relative slack of a mass that must hold the top-p target
// Largest Gumbel noise of the uniform lattice: u <= 1 - 2^-24 gives
// -log(-log u) <= 24 ln 2 = 16.636; the bound used leaves a margin.
constexpr float kGumbelMax = 16.75f;

// row record (64 bytes): computed by warp 0 of each stream CTA and stored
// by the row's first chunk for the finish; for the sampler, written by the
// records kernel before the stream kernel
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
    float s;        // sum exp(z - m) (raw logits: the row LSE)
    int32_t aux;    // relaxed: logits above the draft's; sampler, no filter: index of g
    float g;        // sampler: no filter - the chunk's best Gumbel score; bf16 top-p
                    //   alone - the score of the chunk's first maximum
    float w;        // sampler, top-p alone: chunk mass sum exp((z - m) / T)
    int32_t ncand;  // sampler: entries listed (> the list capacity: overflow)
    float lev;      // sampler, top-k / min-p / fp32 top-p alone: the level the list lies above
};
static_assert(sizeof(ChunkPart) == 32, "chunk summary is 32 bytes");

// shared scratch of the row kernel
struct __align__(16) Shared {
    RowInfo info;
    ChunkPart part;
    uint32_t hist[256];
    uint32_t scan[kWarps];
    float red_f[kWarps * 2];
    int32_t red_i[kWarps * 2];
    int32_t offs[2 * kMaxChunks + 1];
    float M, S, W, sel_excl_f, theta;
    int32_t AMAX, CNT, sel_bin, sel_found, total, overflow, cand_n, R;
    uint32_t sel_excl_u, lkey;
    float extras_v[16];
    int32_t extras_i[16];
    int32_t timeout, fin;
    uint32_t ph[2];     // phases of mbar (thread 0)
    uint64_t mbar[2];   // whole-row streaming stages
};

struct Cand {
    float v;
    int32_t i;
};

// bf16 value of a 16-bit order-preserving key
__device__ __forceinline__ float key16_value(uint32_t k)
{
    return key_value((k << 16) | ((k & 0x8000u) ? 0u : 0xFFFFu));
}

// ------------------------------------------------------ row records -----

// Outputs of request b when its row range is not valid (cu_rows[0] != 0, an
// empty or over-long request, or rows past R_cap): nothing accepted, no next
// token, -1 tokens, and the BAD_ROWS status bit.  One thread per request.
__device__ __forceinline__ void bad_request_outputs(const VerifyParams &p, int b)
{
    if (b >= p.B) return;
    const int32_t c0 = __ldg(p.cu_rows), lo = __ldg(p.cu_rows + b), hi = __ldg(p.cu_rows + b + 1);
    const int32_t n = hi - lo;
    if (c0 != 0 || n < 1 || n - 1 > p.k_max || hi > p.R_cap) {
        p.accepted_len[b] = 0;
        p.next_token[b] = -1;
        for (int j = 0; j <= p.k_max; ++j) p.out_tokens[static_cast<int64_t>(b) * (p.k_max + 1) + j] = -1;
        set_status(p.status, SPEC_STATUS_BAD_ROWS);
    }
}

// The row record of packed row r, computed by one full warp (every lane
// returns it): the owner request (largest b with cu_rows[b] <= r), position,
// validity and the owner's parameters.  With a
// confidence margin it also decides whether the margin applies to the row
// (position, generated-token count, a warp scan of the protected ids) and
// records the draft's logit (NaN if not); relaxed top-K records the draft's
// logit.
template <typename TIn, int MODE>
__device__ RowInfo row_record(const VerifyParams &p, int r)
{
    using E = Elt<TIn>;
    const int lane = threadIdx.x & 31;
    RowInfo inf;
    inf.sel = 0; inf.bad = 0; inf.zd = INFINITY; inf.K = 1;
    inf.T = 0.f; inf.top_k = 0; inf.top_p = 1.f; inf.min_p = 0.f;
    inf.seed_lo = inf.seed_hi = inf.rid = 0;
    inf.draft = __ldg(p.draft_ids + r);
    // The owner: the largest b < B with cu_rows[b] <= r.  Outside the
    // sampler, for 33 to 159 requests, the warp loads all of cu_rows[0..B]
    // at once (lane l holds entries l*P .. l*P+P-1); when they are
    // non-decreasing, b is the count of entries <= r less one and the range
    // ends come by shuffles: one round of loads where the search below
    // takes two.  Otherwise (the sampler, whose stream kernel measured
    // slower with it; up to 32 requests, one round of the search anyway;
    // more requests; offsets out of order) a 32-way search narrows
    // [0, B-1] round by round.
    int b = -1;
    int32_t c0 = 0, rb = 0, re = 0;
    if (MODE != MODE_SAMPLE && p.B > 32 && p.B <= 159) {
        constexpr int kPer = 5;
        const int P = (p.B + 1 + 31) / 32;
        int32_t v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int idx = lane * P + j;
            v[j] = (j < P && idx <= p.B) ? __ldg(p.cu_rows + idx) : INT_MAX;
        }
        int cnt = 0;
        bool mono = true;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int idx = lane * P + j;
            if (j < P && idx < p.B && v[j] <= r) ++cnt;
            if (j + 1 < kPer && j + 1 < P && v[j] > v[j + 1]) mono = false;
        }
        // the next lane's first entry continues this lane's last
        int32_t last = v[0];
#pragma unroll
        for (int j = 1; j < kPer; ++j)
            if (j < P) last = v[j];
        const int32_t next_first = __shfl_down_sync(0xFFFFFFFFu, v[0], 1);
        if (lane < 31 && last > next_first) mono = false;
        if (__all_sync(0xFFFFFFFFu, mono)) {
            b = max(__reduce_add_sync(0xFFFFFFFFu, cnt) - 1, 0);
            // entries b and b + 1 (b + 1 <= B): lane and slot of each
            int32_t sb = v[0], se = v[0];
#pragma unroll
            for (int j = 1; j < kPer; ++j) {
                if (j == b % P) sb = v[j];
                if (j == (b + 1) % P) se = v[j];
            }
            c0 = __shfl_sync(0xFFFFFFFFu, v[0], 0);
            rb = __shfl_sync(0xFFFFFFFFu, sb, b / P);
            re = __shfl_sync(0xFFFFFFFFu, se, (b + 1) / P);
        }
    }
    if (b < 0) {
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
        b = lo;
        c0 = __ldg(p.cu_rows);
        rb = __ldg(p.cu_rows + b);
        re = __ldg(p.cu_rows + b + 1);
    }
    inf.b = b;
    inf.pos = r - rb;
    inf.k_b = re - rb - 1;
    inf.valid = (c0 == 0 && rb <= r && r < re && inf.k_b >= 0 && inf.k_b <= p.k_max && re <= p.R_cap);
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
    return inf;
}

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
    csync();
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
    csync();
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
        csync();
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
        csync();
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
        csync();
        if (MASS && shift == 0) {
            // one value per bin: weight = count * exp((value - M) * sc)
            const uint32_t c = sh.hist[t];
            float w = 0.f;
            if (c) {
                const uint32_t vk = (prefix << width) | static_cast<uint32_t>(t);
                const uint32_t fk = VS ? ((vk << 16) | ((vk & 0x8000u) ? 0u : 0xFFFFu)) : vk;
                w = static_cast<float>(c) * ex2((key_value(fk) - M) * sc);
            }
            csync();
            reinterpret_cast<float *>(sh.hist)[t] = w;
            csync();
        }
        if (MASS) find_crossing<float>(reinterpret_cast<const float *>(sh.hist), target, sh);
        else find_crossing<uint32_t>(sh.hist, k, sh);
        const int bin = sh.sel_bin;
        if (MASS) target -= sh.sel_excl_f;
        else k -= sh.sel_excl_u;
        prefix = (prefix << width) | static_cast<uint32_t>(bin < 0 ? 0 : bin);
        csync();
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
    csync();
    float t = 0.f;
    for (int q = 0; q < kWarps; ++q) t += sh.red_f[q];
    csync();
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
    csync();
    best = -INFINITY;
    bi = INT_MAX;
    for (int q = 0; q < kWarps; ++q)
        if (sh.red_f[q] > best || (sh.red_f[q] == best && sh.red_i[q] < bi)) { best = sh.red_f[q]; bi = sh.red_i[q]; }
    csync();
}

// Philox4x32-10 stream of one row: counter (i >> 2, position, request id,
// step), key (seed lo, seed hi); element i takes word i & 3.
struct Noise {
    Philox ph;
    // counter (i >> 2, position, request id, step), key = the 64-bit seed
    __device__ __forceinline__ Noise(uint32_t pos, uint32_t rid, uint32_t step, uint32_t seed_lo,
                                     uint32_t seed_hi)
        : ph(Philox::make(pos, rid, step, seed_lo, seed_hi))
    {
    }
    __device__ __forceinline__ uint4 block(uint32_t ctr) const { return ph(ctr); }
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

// Element q of a 16-byte vector (q known at compile time after unrolling).
template <typename E>
__device__ __forceinline__ float elt_of(uint4 v, int q)
{
    if constexpr (E::BYTES == 2) {
        const uint32_t w = (q >> 1) == 0 ? v.x : ((q >> 1) == 1 ? v.y : ((q >> 1) == 2 ? v.z : v.w));
        return (q & 1) ? bf_hi(w) : bf_lo(w);
    } else {
        return __uint_as_float(q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w)));
    }
}

// Scores of the elements of the 16-byte vector v starting at element
// `base`, a multiple of 4 (the vector covers whole Philox blocks), whose
// largest value is vm.  An element can only reach `best` if its Gumbel
// noise -log(-log u) reaches best - z/T, i.e. -log u <= D = exp(z/T - best)
// <= exp(vm/T - best); as -log u >= 1 - u, an element with 1 - u > D cannot,
// and for u on the lattice (2k + 1) 2^-24 (k = word >> 9) that is
// k < (2^24 - 1 - D 2^24) / 2.  Those are skipped without the logarithms
// (one below the bound, for the rounding of D); the others are scored as
// usual.  The values stay packed until an element is scored: fewer live
// registers across the Philox rounds.
template <typename E>
__device__ __forceinline__ void score_vec(uint4 v, float vm, int32_t base, float invT,
                                          const Noise &nz, float &best, int32_t &bi)
{
    const float D = ex2((vm * invT - best) * kLog2e);
    const float t = fmaf(-D, 16777216.f, 16777215.f) * 0.5f;
    const uint32_t kthr = (t >= 2.f) ? static_cast<uint32_t>(t) - 1u : 0u;
    // (w >> 9) >= kthr  <=>  w >= kthr << 9 (kthr < 2^23); one test of the
    // block's largest word passes over the usual block with nothing to score
    const uint32_t wthr = kthr << 9;
#pragma unroll
    for (int h = 0; h < E::VEC / 4; ++h) {
        const uint4 w = nz.block((static_cast<uint32_t>(base) >> 2) + h);
        if (max(max(w.x, w.y), max(w.z, w.w)) < wthr) continue;
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (ws[j] >= wthr)
                keep_best(fmaf(elt_of<E>(v, 4 * h + j), invT, gumbel_of(ws[j])), base + 4 * h + j, best, bi);
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

//
// With TOP2 it also gives the thread's second largest element (tsec; equal
// to the maximum when the maximum repeats): the largest of the other
// vectors' maxima, or of the maximum's vector without its first maximum.
template <typename E, int MODE, bool SUM, bool TOP2 = false>
__device__ __forceinline__ float pass1(const uint4 *body, int nb, int a0, float zd, int32_t &targ,
                                       float &tsum, int32_t &tcnt, float *tsec = nullptr)
{
    constexpr int VEC = E::VEC;
    float tmax = kSentinel, t2 = kSentinel;
    int jmax = -1;
#pragma unroll 4
    for (int i = threadIdx.x, j = 0; i < nb; i += kThreads, ++j) {
        const float vm = E::vmax(body[i]);
        if (TOP2) t2 = fmaxf(t2, fminf(vm, tmax));
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
        if (TOP2) {
#pragma unroll
            for (int q = 0; q < VEC; ++q)
                if (q != first) t2 = fmaxf(t2, x[q]);
        }
    }
    if (TOP2) *tsec = (t2 == kSentinel) ? -INFINITY : t2;
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

// ------------------------------------------------------ stream kernel ----

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
    csync();
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
            sh.part.m = m; sh.part.amax = a; sh.part.s = sm_; sh.part.aux = cc;
            sh.part.g = -INFINITY; sh.part.w = 0.f; sh.part.ncand = 0;
            sh.part.lev = -INFINITY;
        }
    }
    csync();
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
        if (tid == 0 && !mbar_wait(&sh.mbar[s], ph[s])) {
            // report it, give this copy and the other one in flight one more
            // bounded wait each, and stop reading the row
            sh.timeout = 1;
            mbar_wait(&sh.mbar[s], ph[s]);
            if (q + 1 < npieces) mbar_wait(&sh.mbar[s ^ 1], ph[s ^ 1]);
        }
        csync();
        if (sh.timeout) break;
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
        csync();
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

// The request chain of request b (k drafts, rows r0 .. r0 + k), run by one
// full warp once every row of the request has its token (and, for relaxed
// or margin acceptance, its flag): the accept-while-equal prefix scan with
// one ballot, the request's tokens and the optional prefix-acceptance
// counters.  The caller has acquired the rows' results (an acquire fence
// after the last ticket of the request).
template <int MODE>
__device__ __forceinline__ void chain_request(const VerifyParams &p, int b, int k, int r0,
                                              uint32_t bad)
{
    const int j = threadIdx.x & 31;
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
        set_status(p.status, bad);
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
    csync();
    visit([&](float v, int32_t ix) {
        const uint32_t d = ktop - (fkey(v) >> 16);
        atomicAdd(cnt + d, 1u);
        atomicMax(bst + d, (static_cast<unsigned long long>(fkey(gs(v, ix))) << 32) |
                               static_cast<uint32_t>(~ix));
    }, key_floor((klo << 16) | ((klo & 0x8000u) ? 0u : 0xFFFFu)));
    csync();
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
    csync();
    float total = 0.f;
    for (int w2 = 0; w2 < kTally / 32; ++w2) {
        if (w2 < warp) cum += wt[w2];
        total += wt[w2];
    }
    const float target = (frac > 0.f) ? frac * total : target_abs;
    const bool ok = (frac > 0.f) || total >= target_abs * (1.f + kMassTol);
    if (!ok) {
        csync();
        return false;
    }
    const int dstar = min(csync_count(tid < kTally && cum < target), kTally - 1);
    unsigned long long sb = (tid < kTally && tid <= dstar) ? bst[tid] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sb = max(sb, __shfl_xor_sync(0xFFFFFFFFu, sb, o));
    unsigned long long *wb = reinterpret_cast<unsigned long long *>(sh.hist);
    if (lane == 0) wb[warp] = sb;
    csync();
    sb = 0ull;
    for (int w2 = 0; w2 < kWarps; ++w2) sb = max(sb, wb[w2]);
    best = -INFINITY;
    bi = INT_MAX;
    if (sb != 0ull) {
        best = key_value(static_cast<uint32_t>(sb >> 32));
        bi = static_cast<int32_t>(~static_cast<uint32_t>(sb));
    }
    csync();
    return true;
}


// The token of a sampler row filtered by top-k and / or min-p (then top-p
// over their survivors), from a candidate list that holds every element of
// the row at or above a bound whose key is klist (visit_lst yields them): the
// survivors of top-k and min-p are the upper set {z >= th_S} (th_S from the
// min-p level and the exact k-th value of the list, given as key_k or
// selected here); top-p keeps the
// group where their mass, counted from the top, first reaches top_p times
// their total (per-value tallies when the survivors span at most kTally
// bf16 values, else an exact mass select); Gumbel-max over what is left.
// cnt [kTally] and bst [kTally] are shared scratch.  Result in best / bi.
template <typename E, typename Visit>
__device__ void settle_from_list(Visit &&visit_lst, const RowInfo &info, const Filter &f, float M,
                                 uint32_t klist, uint32_t key_k, uint32_t *cnt, unsigned long long *bst,
                                 GumbelScorer &gs, float &best, int32_t &bi, Shared &sh)
{
    const float sc = f.sc;
    const uint32_t keyM = fkey(M);
    const float th_m = f.use_m ? M + f.T * logf(info.min_p) : -INFINITY;
    uint32_t key_S = f.use_m ? fkey(th_m) : 0u;
    // key_k: the k-th largest value's key when the caller already has it
    // (0xFFFFFFFF: not known, select it)
    if (f.use_k)
        key_S = max(key_S, key_k != 0xFFFFFFFFu
                               ? key_k
                               : select_key<E, false>(visit_lst, max(key_S, klist), keyM, 0.f,
                                                      static_cast<uint32_t>(info.top_k), M, sc, sh));
    if (E::BYTES == 2 && f.use_p) {
        // the survivors tallied per value when they span at most kTally
        // bf16 values
        const uint32_t klo = bf16_key_ceil(key_S), ktop = keyM >> 16;
        if (ktop >= klo && ktop - klo < static_cast<uint32_t>(kTally)) {
            tally_top_p(visit_lst, klo, ktop, M, sc, gs, info.top_p, 0.f, cnt, bst, best, bi, sh);
            return;
        }
    }
    uint32_t key_F = key_S;
    if (f.use_p) {
        float w = 0.f;
        const uint32_t kS = key_S;
        visit_lst([&](float v, int32_t) {
            if (fkey(v) >= kS) w += ex2((v - M) * sc);
        }, key_floor(key_S));
        const float Wt = block_sum(w, sh);
        key_F = max(key_S, select_key<E, true>(visit_lst, key_S, keyM, info.top_p * Wt, 0u, M, sc, sh));
    }
    const uint32_t kF = key_F;
    visit_lst([&](float v, int32_t ix) {
        if (fkey(v) >= kF) keep_best(gs(v, ix), ix, best, bi);
    }, key_floor(key_F));
    block_best(best, bi, sh);
}

}  // namespace specv
