// Shared device helpers for the DSpark kernels (sm_103a): status block,
// bounded mbarrier waits, bulk copies, Philox4x32-10 and the uniform /
// Gumbel draws, and small reductions.  Inline PTX is used where CUDA C++ has
// no spelling for the instruction.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

// ---------------------------------------------------------------- status ---
// Workspace head: {code, detail, pad, pad}.  Written only on error.
struct StatusBlock {
    uint32_t code;
    uint32_t detail;
    uint32_t pad[2];
};
constexpr size_t kStatusBytes = 256;   // keeps what follows 256-byte aligned

__device__ __forceinline__ void set_status(StatusBlock* st, uint32_t code, uint32_t detail) {
    if (st != nullptr && atomicCAS(&st->code, 0u, code) == 0u) st->detail = detail;
}

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16-byte asynchronous global -> shared copy (no register staging); wait with
// cp_async_wait_all before the data is read.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for phase `parity` of `bar`; returns false if kWaitLimitNs passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ------------------------------------------------------------ bulk copy ---
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- Philox ---
constexpr float kLn2f = 0.69314718055994531f;

// Philox4x32-10 (Salmon et al., SC'11): per round, 32x32->64 products of
// c0 and c2 with the two round multipliers, the high halves xored into the
// other words with the round key, key bumped by the Weyl constants.
struct U4 {
    uint32_t x, y, z, w;
};
// The full 64-bit product of two 32-bit words as (lo, hi), one mul.wide.u32.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& lo, uint32_t& hi) {
    uint64_t p;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
    lo = static_cast<uint32_t>(p);
    hi = static_cast<uint32_t>(p >> 32);
}
__device__ __forceinline__ U4 philox4x32_10_inline(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        uint32_t lo0, hi0, lo1, hi1;
        mul_wide(0xD2511F53u, c.x, lo0, hi0);
        mul_wide(0xCD9E8D57u, c.z, lo1, hi1);
        c = U4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}
static __device__ __noinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
    return philox4x32_10_inline(c, k0, k1);
}
enum Stream : uint32_t {
    kStreamDraftToken = 0,    // Gumbel noise of the draft token x_k, one word per vocabulary index
    kStreamAccept = 1,        // acceptance uniform of the rejection test (index 0)
    kStreamVerifyToken = 2,   // Gumbel noise of the token verification emits (residual, bonus or
                              // the draw from p_t when a residual has no mass; one per request)
};
// The 32-bit word keyed by (seed, request b, position k, stream, index).
__device__ __forceinline__ uint32_t draw_word(uint64_t seed, uint32_t b, uint32_t k, uint32_t stream,
                                              uint32_t index) {
    const U4 r = philox4x32_10(U4{index >> 2, k, b, stream}, static_cast<uint32_t>(seed),
                               static_cast<uint32_t>(seed >> 32));
    const uint32_t sel = index & 3u;
    return sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
}

// Philox4x32-10 for the counters (q, k, b, stream) of one row (k, b, stream
// fixed, q varying).  The first round's product of the third counter word (b)
// and the second round's product of the first word (which after round one no
// longer depends on q) are the same for every q: they are formed once here,
// so a call costs eighteen 32x32->64 products instead of twenty.  The result
// is bit-identical to philox4x32_10({q, k, b, stream}, key).
struct PhiloxRow {
    uint32_t k0, k1;     // key
    uint32_t r1_x;       // round 1: word x (constant)
    uint32_t r1_y;       // round 1: word y (constant)
    uint32_t r1_z;       // round 1: word z = hi(M0 q) ^ r1_z
    uint32_t r2_y;       // round 2: word y ^ key (constant part of the new x)
    uint32_t r2_hi0;     // round 2: hi(M0 r1_x) ^ key1 (xored with lo(M0 q) into the new z)
    uint32_t r2_lo0;     // round 2: lo(M0 r1_x) (the new w)
};
__device__ __forceinline__ PhiloxRow philox_row_setup(uint64_t seed, uint32_t k, uint32_t b, uint32_t stream) {
    PhiloxRow r;
    r.k0 = static_cast<uint32_t>(seed);
    r.k1 = static_cast<uint32_t>(seed >> 32);
    uint32_t lo1, hi1;
    mul_wide(0xCD9E8D57u, b, lo1, hi1);
    r.r1_x = hi1 ^ k ^ r.k0;
    r.r1_y = lo1;
    r.r1_z = stream ^ r.k1;
    const uint32_t k0b = r.k0 + 0x9E3779B9u, k1b = r.k1 + 0xBB67AE85u;
    r.r2_y = r.r1_y ^ k0b;
    uint32_t lo0, hi0;
    mul_wide(0xD2511F53u, r.r1_x, lo0, hi0);
    r.r2_hi0 = hi0 ^ k1b;
    r.r2_lo0 = lo0;
    return r;
}
__device__ __forceinline__ U4 philox_row(const PhiloxRow& r, uint32_t q) {
    // round 1: only the product of q varies
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide(0xD2511F53u, q, lo0, hi0);
    const uint32_t z1 = hi0 ^ r.r1_z;
    // round 2: the product of word x is constant, the product of z1 varies
    mul_wide(0xCD9E8D57u, z1, lo1, hi1);
    U4 c{hi1 ^ r.r2_y, lo1, r.r2_hi0 ^ lo0, r.r2_lo0};
    uint32_t k0 = r.k0 + 2u * 0x9E3779B9u, k1 = r.k1 + 2u * 0xBB67AE85u;
#pragma unroll
    for (int i = 2; i < 10; ++i) {
        uint32_t a0, b0, a1, b1;
        mul_wide(0xD2511F53u, c.x, a0, b0);
        mul_wide(0xCD9E8D57u, c.z, a1, b1);
        c = U4{b1 ^ c.y ^ k0, a1, b0 ^ c.w ^ k1, a0};
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}
// The round keys of one seed (the key bumped by the Weyl constants each round),
// formed on the host: kept in a kernel's parameters, they enter the rounds as
// constant operands instead of being re-derived per block.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};
inline PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys K;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        K.k0[i] = k0;
        K.k1[i] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return K;
}
// philox_row with the round keys taken from K (the seed philox_row_setup got).
__device__ __forceinline__ U4 philox_row(const PhiloxRow& r, uint32_t q, const PhiloxKeys& K) {
    uint32_t lo0, hi0, lo1, hi1;
    mul_wide(0xD2511F53u, q, lo0, hi0);
    const uint32_t z1 = hi0 ^ r.r1_z;
    mul_wide(0xCD9E8D57u, z1, lo1, hi1);
    U4 c{hi1 ^ r.r2_y, lo1, r.r2_hi0 ^ lo0, r.r2_lo0};
#pragma unroll
    for (int i = 2; i < 10; ++i) {
        uint32_t a0, b0, a1, b1;
        mul_wide(0xD2511F53u, c.x, a0, b0);
        mul_wide(0xCD9E8D57u, c.z, a1, b1);
        c = U4{b1 ^ c.y ^ K.k0[i], a1, b0 ^ c.w ^ K.k1[i], a0};
    }
    return c;
}
__device__ __forceinline__ uint32_t u4_word(const U4& r, uint32_t sel) {
    return sel == 0 ? r.x : sel == 1 ? r.y : sel == 2 ? r.z : r.w;
}

// u in (0, 1): ((w >> 9) + 1/2) * 2^-23 (exact in float32).
__device__ __forceinline__ float uniform_open(uint32_t w) {
    return (static_cast<float>(w >> 9) + 0.5f) * 1.1920928955078125e-07f;
}
// u in [0, 1): (w >> 8) * 2^-24 (exact in float32).
__device__ __forceinline__ float uniform_accept(uint32_t w) {
    return static_cast<float>(w >> 8) * 5.9604644775390625e-08f;
}

// log2 on the special-function unit (lg2.approx.ftz: absolute error about 2^-22
// for arguments in [1/2, 2]).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The exponential variate E = -ln u of the Gumbel draw G = -ln(-ln u) = -ln E,
// for u = ((w >> 9) + 1/2) 2^-23.  Draws compare e_v / E_v (or lw_v - log2 E_v),
// so E must keep its relative accuracy where it is small, i.e. for u near 1.
// u and s = 1 - u are both exact in float32 (odd multiples of 2^-24).  For
// s < 1/16, E = -ln(1 - s) is its Taylor series s + s^2/2 + s^3/3 + s^4/4 + s^5/5
// (the next term is below 1.7e-7 of the sum); otherwise -ln u >= 0.0645 and the
// special-function log2 (absolute error ~2^-22) keeps the relative error of E
// below ~3e-6.  A GPU test checks every one of the 2^23 values against float64.
__device__ __forceinline__ float exp_draw(uint32_t w) {
    const float f = __uint_as_float((w >> 9) | 0x3F800000u);   // 1 + m 2^-23
    const float u = f - 0.999999940395355225f;                 // (m + 1/2) 2^-23, exact
    const float s = 1.0f - u;                                  // exact
    const float series = s * fmaf(s, fmaf(s, fmaf(s, fmaf(s, 0.2f, 0.25f), 0.333333343f), 0.5f), 1.0f);
    const float viaLog = -kLn2f * fast_log2(u);
    return (s < 0.0625f) ? series : viaLog;
}

// ------------------------------------------------------------ reductions ---
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 2^x on the special-function unit (ex2.approx.ftz: ~2 ulp; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 pair (packed in a 32-bit word) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

}  // namespace dspark
