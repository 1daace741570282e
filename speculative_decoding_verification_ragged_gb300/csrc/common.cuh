// common.cuh -- device helpers shared by the verification kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used on the hot path: 1-D TMA bulk
// copies global -> shared (cp.async.bulk ... mbarrier::complete_tx) and
// mbarrier waits that suspend the thread (with an overall time limit).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "spec_verify.h"

namespace specv {

constexpr int kThreads = 256;              // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kChunkBytes = 32 * 1024;     // bytes of a row one CTA stages on chip
constexpr int kMaxChunks = 64;             // chunks per row (rows up to 2 MiB)
constexpr uint32_t kWaitTries = 1024;      // suspended mbarrier tries before giving up
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- PTX -----

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// try_wait that lets the hardware suspend the thread for up to `ns`
// nanoseconds while the phase is incomplete (no busy polling)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier.  Each try may suspend the thread
// for up to 1 ms; after kWaitTries tries (about a second) it gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitTries; ++i)
        if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    return false;
}

// Order this thread's view of shared memory (generic proxy) before a
// following bulk copy into it (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start
// early / wait until the previous kernel's results are visible.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 eviction-first hint: for data read exactly once
// (the logits), so that it does not push out the small per-chunk summaries
// the next kernel reads back.
__device__ __forceinline__ void bulk_g2s_stream(void *dst, const void *src, uint32_t bytes,
                                                uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], pol;\n\t}"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Barrier of the CTA's compute warps only (named barrier 2, kThreads
// threads): the ticket warp of the row kernel never joins it.
__device__ __forceinline__ void csync()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
}

// csync() that also counts the threads whose predicate is true
__device__ __forceinline__ int csync_count(bool pred)
{
    int r;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.popc.u32 %0, 2, %2, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kThreads)
        : "memory");
    return r;
}

// Release / acquire fence at GPU scope (orders this CTA's earlier writes,
// made visible to this thread by a CTA barrier, before a following atomic;
// or a preceding atomic before later reads).
__device__ __forceinline__ void fence_acq_rel_gpu()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Maximum of a float over the full warp (NaN operands ignored, as fmaxf).
__device__ __forceinline__ float warp_max_f32(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of fp32 in one 64-bit register (Blackwell f32x2 arithmetic:
// two independent IEEE fp32 operations per instruction, each rounded as the
// scalar one).
__device__ __forceinline__ uint64_t f2_pack(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ------------------------------------------------------------ values -----

// Order-preserving 32-bit key of a float; -0.0 and +0.0 map to one key.
__device__ __forceinline__ uint32_t fkey(float x)
{
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// bf16 pair packed in one 32-bit word -> two floats (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max of the 8 bf16 values of a 16-byte vector, as float: packed bf16x2
// maxima on the 32-bit words themselves (no detour through memory)
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return m;
}

__device__ __forceinline__ float vmax_bf16(uint4 v)
{
    const uint32_t w = max_bf16x2(max_bf16x2(v.x, v.y), max_bf16x2(v.z, v.w));
    return fmaxf(bf_lo(w), bf_hi(w));
}

// Element traits: 16-byte vectors of bf16 (8 values) or fp32 (4 values).
template <typename T> struct Elt;
template <> struct Elt<uint16_t> {
    static constexpr int VEC = 8;
    static constexpr int BYTES = 2;
    static __device__ __forceinline__ void unpack(uint4 v, float (&x)[8])
    {
        x[0] = bf_lo(v.x); x[1] = bf_hi(v.x); x[2] = bf_lo(v.y); x[3] = bf_hi(v.y);
        x[4] = bf_lo(v.z); x[5] = bf_hi(v.z); x[6] = bf_lo(v.w); x[7] = bf_hi(v.w);
    }
    static __device__ __forceinline__ float vmax(uint4 v) { return vmax_bf16(v); }
    static __device__ __forceinline__ float load(const void *p, int64_t i)
    {
        return __uint_as_float(static_cast<uint32_t>(
                                   __ldg(reinterpret_cast<const unsigned short *>(p) + i))
                               << 16);
    }
};
template <> struct Elt<float> {
    static constexpr int VEC = 4;
    static constexpr int BYTES = 4;
    static __device__ __forceinline__ void unpack(uint4 v, float (&x)[4])
    {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ float vmax(uint4 v)
    {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    static __device__ __forceinline__ float load(const void *p, int64_t i)
    {
        return __ldg(reinterpret_cast<const float *>(p) + i);
    }
};

// ------------------------------------------------------------ Philox -----
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): each round
// multiplies counter words 0 and 2 by fixed odd constants, swaps the
// halves, and mixes in the round key; the key advances by Weyl increments.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// the 64-bit product of two words as (lo, hi): one wide multiply
__device__ __forceinline__ void mulhilo32(uint32_t a, uint32_t b, uint32_t &lo, uint32_t &hi)
{
    const uint64_t m = static_cast<uint64_t>(a) * b;
    lo = static_cast<uint32_t>(m);
    hi = static_cast<uint32_t>(m >> 32);
}

// Philox4x32-10 blocks for counters (ctr, w1, w2, w3) in which only ctr
// varies.  Round 0 multiplies word 2 (= w2) and round 1 multiplies word 0
// (a function of w1, w2 and the key alone), so those two products and the
// words they feed are fixed per (w1, w2, w3, key) and computed once; a
// block then costs two wide multiplies for rounds 0-1 and two per later
// round.  Identical output to the round-by-round definition.
struct Philox {
    uint32_t C, D, E, F;        // words entering rounds 0-1 that do not depend on ctr
    uint32_t k0, k1;            // the key of round 2
    __device__ __forceinline__ static Philox make(uint32_t w1, uint32_t w2, uint32_t w3,
                                                  uint32_t key0, uint32_t key1)
    {
        Philox q;
        uint32_t lo, hi;
        mulhilo32(kPhiloxM1, w2, lo, hi);               // round 0, word 2
        const uint32_t A = hi ^ w1 ^ key0;              // round 0 output word 0
        q.C = w3 ^ key1;                                // xored into round 0 output word 2
        uint32_t loA, hiA;
        mulhilo32(kPhiloxM0, A, loA, hiA);              // round 1, word 0
        q.D = lo ^ (key0 + kPhiloxW0);                  // round 1 output word 0 = hi(M1 x) ^ D
        q.E = hiA ^ (key1 + kPhiloxW1);                 // round 1 output word 2 = lo0 ^ E
        q.F = loA;                                      // round 1 output word 3
        q.k0 = key0 + 2u * kPhiloxW0;
        q.k1 = key1 + 2u * kPhiloxW1;
        return q;
    }
    __device__ __forceinline__ uint4 operator()(uint32_t ctr) const
    {
        uint32_t lo0, hi0, lo1, hi1;
        mulhilo32(kPhiloxM0, ctr, lo0, hi0);            // round 0, word 0
        mulhilo32(kPhiloxM1, hi0 ^ C, lo1, hi1);        // round 1, word 2
        uint4 c = make_uint4(hi1 ^ D, lo1, lo0 ^ E, F);
        uint32_t a = k0, b = k1;
#pragma unroll
        for (int i = 2; i < 10; ++i) {
            mulhilo32(kPhiloxM0, c.x, lo0, hi0);
            mulhilo32(kPhiloxM1, c.z, lo1, hi1);
            c = make_uint4(hi1 ^ c.y ^ a, lo1, hi0 ^ c.w ^ b, lo0);
            a += kPhiloxW0;
            b += kPhiloxW1;
        }
        return c;
    }
};

__device__ __forceinline__ uint32_t word_of(uint4 v, uint32_t w)
{
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// Gumbel noise -log(-log u) of the uniform u = (2*(x>>9)+1) * 2^-24.
// E = -log(u) needs relative accuracy: for u close to 1 it is computed from
// d = 1 - u (exact, the same lattice read from ~x) by its Taylor series
// d + d^2/2 + ... + d^5/5 (truncation below 2^-25 relative for d < 2^-5);
// elsewhere from the hardware log2.  The outer log only needs absolute
// accuracy.
__device__ __forceinline__ float gumbel_of(uint32_t x)
{
    const float u = __uint_as_float((x >> 9) | 0x3F800000u) - __uint_as_float(0x3F7FFFFFu);
    const float d = __uint_as_float(((~x) >> 9) | 0x3F800000u) - __uint_as_float(0x3F7FFFFFu);
    // both forms evaluated and selected: no divergent branch in a warp
    const float e_series = d * fmaf(d, fmaf(d, fmaf(d, fmaf(d, 0.2f, 0.25f), 1.0f / 3.0f), 0.5f), 1.0f);
    const float e_log = -kLn2 * lg2(u);
    const float e = (d < 0.03125f) ? e_series : e_log;
    return -kLn2 * lg2(e);
}

// ------------------------------------------------------------ misc -----

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits)
{
    if (status && bits) atomicOr(status, bits);
}

}  // namespace specv
