// dspark_accept_rate_tv: c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 per row
// (DeepSpec walkthrough, section 3.3, paper eq. 8 / `_compute_accept_rate_3d`),
// computed as sum_v exp(min(d_v - L_d, t_v - L_t)) with L = logsumexp of the row;
// and dspark_training_loss (section 7.2, `compute_dspark_loss`), the same sums
// extended to the joint loss and its gradient.
//
// One CTA of 1024 threads per SM takes rows in turn and reads each row's d and t
// once from HBM (pass 1: the two logsumexps) and again from L2, where pass 1 left
// them (pass 2: the sum of min(p_d, p_t); the loss adds a third pass that writes
// dL/dd).  A CTA's row of the Qwen3 vocabulary is 607,744 bytes of bf16, 92 MB
// for one row per SM: it stays in the L2 between the passes.  Every thread
// streams its own 16-byte groups through its own slots of a cp.async ring in
// shared memory, five groups ahead.
#include <type_traits>

#include "common.cuh"
#include "host_common.h"

namespace dspark {
namespace {

template <bool kBF16>
struct TVTraits {
    static constexpr int kEPG = kBF16 ? 8 : 4;   // elements per 16-byte group
    static constexpr int kESZ = kBF16 ? 2 : 4;
};

template <bool kBF16>
__device__ __forceinline__ void unpack(const uint4 v, float* out) {
    if constexpr (kBF16) {
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z); out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
    } else {
        out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
    }
}

// Packed pairs of float32 (Blackwell f32x2 arithmetic): two lanes of work per
// instruction for the element-wise part of the sums.
__device__ __forceinline__ unsigned long long pk(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 upk(unsigned long long v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Two floats -> a bf16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The training loss: per row, with p = softmax,
//   ce = logsumexp(d) - d[target], c* = sum min(p_d, p_t), l1 = 1 - c*,
//   bce = softplus(s) - c* s, row = omega (a_ce ce + a_l1 l1 + a_conf bce),
//   dL/dd_v = omega (a_ce (p_d(v) - [v = target]) + a_l1 / 2 p_d(v) (sgn_v - sum_u p_d(u) sgn_u)),
//   dL/ds = omega a_conf (sigmoid(s) - c*), sgn_v = sign(p_d(v) - p_t(v)).
// sum_u p_d(u) sgn_u = 1 - 2 P_lt - P_eq, with P_lt (P_eq) the p_d mass where
// p_d < p_t (p_d = p_t): pass C's terms there are p_d itself.
struct LossArgs {
    const int32_t* target;  // [rows]
    const float* s;         // [rows] confidence head logits
    const float* omega;     // [rows] row weights
    float a_ce, a_l1, a_conf;
    float* row_out;         // [rows][4] (ce, c*, bce, row)
    void* grad;             // [rows][V] dL/dd (input dtype), or null
    float* grad_s;          // [rows] dL/ds, or null
    float* cl_part;         // [CTAs] each CTA's sum of row totals
    unsigned int* cl_done;  // CTAs finished (starts at 0)
    float* loss;            // [1] sum of row totals
};

// (m, s) with s a sum of 2^((x - m) log2e): merge across a warp (the warp's max of
// the m that carry mass, then the rescaled sum).
__device__ __forceinline__ void warp_lse(float& m, float& s) {
    const float M = warp_max(s > 0.f ? m : -INFINITY);
    const float r = s > 0.f ? s * fast_exp2((m - M) * kLog2e) : 0.f;
    s = warp_sum(r);
    m = M > -INFINITY ? M : 0.f;
}

// log2 on the special-function unit (lg2.approx.ftz: absolute error about 2^-22).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Each CTA of a loss launch leaves its sum of row totals in the workspace: at
// most this many (the grid is one CTA per SM).
constexpr int kMaxLossCtas = 1024;

// ------------------------------------------------------- accept rate, two passes
// dspark_accept_rate_tv's kernel: one CTA of 1024 threads per SM takes rows in
// turn.  Pass 1 streams the row's d and t from HBM (L2 evict-last) and forms each
// thread's online (max, sum of 2^((x - max) log2e)) of both; a block reduction
// gives L_d and L_t; pass 2 streams the same row again -- from L2, where pass 1
// left it (a CTA's row is 607,744 B for bf16 and V = 151936, so one row per SM,
// 92 MB in all, stays within the L2) -- with the evict-first policy, summing
// 2^(min(d - L_d, t - L_t) log2e).  A logit pair costs three exponentials and
// about 24 instructions in all; no shared-memory copy of the row is needed.
//
// Loads: every thread copies its own 16-byte groups into its own slots of a ring
// in shared memory with cp.async (no block barrier guards a slot: only the thread
// that copied it reads it), kTv2Stages - 1 groups of d and of t ahead of the one
// it is summing: 160 KB in flight per SM.  A pass's first groups are issued before
// the block merge that precedes it, so they land while the CTA waits there; a
// row's c* is summed across the block inside the next row's merge.
constexpr int kTv2Threads = 1024;
constexpr int kTv2Stages = 6;
constexpr size_t kTv2Smem = static_cast<size_t>(kTv2Stages) * 2 * kTv2Threads * 16;
// The loss keeps a sign byte per 16-byte group of d beside the ring for rows of up to
// this many groups per thread (V = 270,336 for bf16): 33 KB more shared memory,
// 227 KB per CTA in all with the kernel's static arrays.
constexpr int kLossMaxBitGroups = 33;
// The loss's passes run their group loop unrolled three times (0.6 % faster than
// once; the accept rate's two passes are faster rolled).
constexpr int kLossUnroll = 3;
constexpr size_t kLossSmemMax = kTv2Smem + static_cast<size_t>(kLossMaxBitGroups) * kTv2Threads;

// The group's max (raw units), -inf if it has no finite element.
template <bool kBF16>
__device__ __forceinline__ float group_max(const uint4 v) {
    if constexpr (kBF16) {
        const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
        return fmaxf(bf16lo(m), bf16hi(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}

// (m, s) += the group's elements, s a sum of 2^((x - m) log2e).  m is a running
// reference, not the running max: the group is summed against the current m, and
// only when that sum leaves [0, 2^32] (an element at least 22 above m, or no m
// yet: inf or NaN) is m moved to the group's max, s rescaled and the group summed
// again -- so the max of a group is taken for a thread's first groups of a row and
// rarely after.  Terms up to 2^32 change no relative precision of the float sums.
// For bf16 the exponent is one fused x log2e - (m log2e): every term carries the
// rounding error r of m log2e (|r| <= ulp(m log2e) / 2, a relative 1e-5 at
// |m| = 100, inside the bf16 bound).  For float32, whose bound is tighter, x - m is
// formed first.
template <bool kBF16>
__device__ __forceinline__ void group_lse(const uint4 v, float& m, float& s) {
    constexpr int EPG = TVTraits<kBF16>::kEPG;
    float a[EPG];
    unpack<kBF16>(v, a);
    // the group's sum of 2^((x - mm) log2e)
    auto terms = [&](float mm) -> float {
        const unsigned long long L2E = pk(kLog2e, kLog2e);
        const unsigned long long nm = kBF16 ? pk(-mm * kLog2e, -mm * kLog2e) : pk(-mm, -mm);
        unsigned long long acc = pk(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < EPG; e += 2) {
            const float2 y = kBF16 ? upk(fma2(pk(a[e], a[e + 1]), L2E, nm)) : upk(mul2(add2(pk(a[e], a[e + 1]), nm), L2E));
            acc = add2(acc, pk(fast_exp2(y.x), fast_exp2(y.y)));
        }
        return upk(acc).x + upk(acc).y;
    };
    float g = terms(m);
    if (!(g <= 0x1p32f)) {
        // rare: an element far above m, or no m yet (inf or NaN): rebase on the group's max
        const float gm = group_max<kBF16>(v);
        if (!(gm > -INFINITY)) return;                    // no mass in this group
        if (gm > m) {
            s = (s > 0.f) ? s * fast_exp2((m - gm) * kLog2e) : 0.f;
            m = gm;
        }
        g = terms(m);
    }
    s += g;
}

// Block-wide merge of every thread's (m, s) pair for d and t: all threads get (L_d, L_t)
// in natural units.
__device__ __forceinline__ float2 block_lse2(float md, float sd, float mt, float st, float4* red, float2* fin,
                                             const float* prev = nullptr, float* prev_out = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_lse(md, sd);
    warp_lse(mt, st);
    if (lane == 0) red[warp] = make_float4(md, sd, mt, st);
    __syncthreads();
    if (warp == 0) {
        float4 r = (lane < kTv2Threads / 32) ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        warp_lse(r.x, r.y);
        warp_lse(r.z, r.w);
        // the previous row's per-warp partial sums, left in `prev` before this barrier
        float pv = 0.f;
        if (prev_out != nullptr) pv = warp_sum((lane < kTv2Threads / 32) ? prev[lane] : 0.f);
        if (lane == 0) {
            const float Ld = (r.y > 0.f) ? r.x + fast_log2(r.y) * kLn2 : -INFINITY;
            const float Lt = (r.w > 0.f) ? r.z + fast_log2(r.w) * kLn2 : -INFINITY;
            *fin = make_float2(Ld, Lt);
            if (prev_out != nullptr) *prev_out = pv;
        }
    }
    __syncthreads();
    return *fin;
}

// One 16-byte asynchronous copy global -> shared with an L2 policy (cp.async.cg).
__device__ __forceinline__ void cp16_hint(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One pass over a row: a thread's groups i = 0 .. nmine - 1 (group tid + i T) of d
// and t (of d alone with kT = false; vt is then vd) go through its ring, copied
// kTv2Stages - 1 groups ahead of the one that body(vd, vt, g) sums (g: the group's
// index in the row), d with L2 policy pol and t with polt.  Each issue commits one
// cp.async group, empty past the last, so that "group i has landed" is always
// wait_group(S - 2) after i + S - 1 commits.
// Issues the first kTv2Stages - 1 groups of a pass into the ring (tv2_pass with
// `primed` skips them): lets the next pass's loads fly while the block merges.
template <bool kT = true>
__device__ __forceinline__ void tv2_prime(const uint4* gd, const uint4* gt, int nmine, uint4* ring, uint64_t pol,
                                          uint64_t polt) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < kTv2Stages - 1; ++i) {
        if (i < nmine) {
            const int g = tid + i * kTv2Threads;
            uint4* slot = ring + static_cast<size_t>(i % kTv2Stages) * 2 * kTv2Threads + tid;
            cp16_hint(slot, gd + g, pol);
            if (kT) cp16_hint(slot + kTv2Threads, gt + g, polt);
        }
        cp_commit();
    }
}

template <bool kT = true, int kUnroll = 1, class F>
__device__ __forceinline__ void tv2_pass(const uint4* gd, const uint4* gt, int nmine, uint4* ring, uint64_t pol,
                                         uint64_t polt, F&& body, bool primed = false) {
    const int tid = threadIdx.x;
    auto issue = [&](int i, int slot) {
        if (i < nmine) {
            const int g = tid + i * kTv2Threads;
            uint4* dst = ring + static_cast<size_t>(slot) * 2 * kTv2Threads + tid;
            cp16_hint(dst, gd + g, pol);
            if (kT) cp16_hint(dst + kTv2Threads, gt + g, polt);
        }
        cp_commit();
    };
    if (!primed) {
#pragma unroll
        for (int i = 0; i < kTv2Stages - 1; ++i) issue(i, i);
    }
    int rd = 0, wr = kTv2Stages - 1;
#pragma unroll kUnroll
    for (int i = 0; i < nmine; ++i) {
        cp_wait<kTv2Stages - 2>();
        const uint4* slot = ring + static_cast<size_t>(rd) * 2 * kTv2Threads + tid;
        const uint4 vd = slot[0], vt = kT ? slot[kTv2Threads] : vd;
        issue(i + kTv2Stages - 1, wr);
        wr = rd;
        rd = rd == kTv2Stages - 1 ? 0 : rd + 1;
        body(vd, vt, tid + i * kTv2Threads);
    }
    cp_wait<0>();
}

template <bool kBF16>
__global__ void __launch_bounds__(kTv2Threads, 1)
tv_two_pass(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star, int64_t rows,
            int V) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ;
    extern __shared__ __align__(16) uint8_t tv2_smem[];
    uint4* ring = reinterpret_cast<uint4*>(tv2_smem);
    __shared__ float4 red[kTv2Threads / 32];
    __shared__ float2 fin;
    __shared__ float red2[kTv2Threads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ngroups = V / EPG;
    const int nmine = (ngroups > tid) ? (ngroups - tid + kTv2Threads - 1) / kTv2Threads : 0;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    int64_t prev_row = -1;                                // its per-warp partials wait in red2
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4* gd = reinterpret_cast<const uint4*>(d + static_cast<size_t>(row) * V * ESZ);
        const uint4* gt = reinterpret_cast<const uint4*>(t + static_cast<size_t>(row) * V * ESZ);
        // pass 1: (max, sum) of d and t, from HBM
        float md = -INFINITY, sd = 0.f, mt = -INFINITY, st = 0.f;
        tv2_pass(gd, gt, nmine, ring, keep, keep, [&](const uint4 vd, const uint4 vt, int) {
            group_lse<kBF16>(vd, md, sd);
            group_lse<kBF16>(vt, mt, st);
        });
        if (!(md > -INFINITY)) { md = 0.f; sd = 0.f; }
        if (!(mt > -INFINITY)) { mt = 0.f; st = 0.f; }
        // pass 2's first loads fly while the block merges this row's logsumexps (which
        // also finishes the previous row's c*)
        tv2_prime(gd, gt, nmine, ring, drop, drop);
        const float2 L = block_lse2(md, sd, mt, st, red, &fin, red2, prev_row >= 0 ? c_star + prev_row : nullptr);
        // pass 2: sum of 2^(min(d - L_d, t - L_t) log2e), from L2 (for bf16 the
        // exponents are the fused d log2e - L_d log2e and t log2e - L_t log2e)
        unsigned long long acc = pk(0.f, 0.f);
        if (!(L.x > -INFINITY && L.y > -INFINITY)) cp_wait<0>();   // no mass: the primed loads are dropped
        if (L.x > -INFINITY && L.y > -INFINITY) {
            const unsigned long long L2E = pk(kLog2e, kLog2e);
            const float sc = kBF16 ? kLog2e : 1.f;
            const unsigned long long nLd = pk(-L.x * sc, -L.x * sc), nLt = pk(-L.y * sc, -L.y * sc);
            tv2_pass(gd, gt, nmine, ring, drop, drop, [&](const uint4 vd, const uint4 vt, int) {
                float a[EPG], b[EPG];
                unpack<kBF16>(vd, a);
                unpack<kBF16>(vt, b);
#pragma unroll
                for (int e = 0; e < EPG; e += 2) {
                    if constexpr (kBF16) {
                        const float2 x = upk(fma2(pk(a[e], a[e + 1]), L2E, nLd));
                        const float2 y = upk(fma2(pk(b[e], b[e + 1]), L2E, nLt));
                        acc = add2(acc, pk(fast_exp2(fminf(x.x, y.x)), fast_exp2(fminf(x.y, y.y))));
                    } else {
                        const float2 x = upk(add2(pk(a[e], a[e + 1]), nLd));
                        const float2 y = upk(add2(pk(b[e], b[e + 1]), nLt));
                        const float2 z = upk(mul2(pk(fminf(x.x, y.x), fminf(x.y, y.y)), L2E));
                        acc = add2(acc, pk(fast_exp2(z.x), fast_exp2(z.y)));
                    }
                }
            }, /*primed=*/true);
        }
        float part = upk(acc).x + upk(acc).y;
        part = warp_sum(part);
        if (lane == 0) red2[warp] = part;                 // read after the next row's first barrier
        prev_row = row;
        // red and fin are rewritten by the next row after the first barrier in block_lse2
    }
    if (prev_row >= 0) {
        __syncthreads();
        if (warp == 0) {
            const float v = warp_sum((lane < kTv2Threads / 32) ? red2[lane] : 0.f);
            if (lane == 0) c_star[prev_row] = v;
        }
    }
}

// As block_lse2, but every thread gets the parts (M_d, log S_d, M_t, log S_t) in
// natural units (L = M + log S), so that L_d - L_t can be formed from them.
__device__ __forceinline__ float4 block_lse2_parts(float md, float sd, float mt, float st, float4* red,
                                                   float4* fin) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_lse(md, sd);
    warp_lse(mt, st);
    if (lane == 0) red[warp] = make_float4(md, sd, mt, st);
    __syncthreads();
    if (warp == 0) {
        float4 r = (lane < kTv2Threads / 32) ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        warp_lse(r.x, r.y);
        warp_lse(r.z, r.w);
        if (lane == 0)
            *fin = make_float4(r.y > 0.f ? r.x : 0.f, r.y > 0.f ? fast_log2(r.y) * kLn2 : -INFINITY,
                               r.w > 0.f ? r.z : 0.f, r.w > 0.f ? fast_log2(r.w) * kLn2 : -INFINITY);
    }
    __syncthreads();
    return *fin;
}

// ------------------------------------------------------- training loss, three passes
// dspark_training_loss's kernel: one CTA of 1024 threads per SM takes rows in
// turn, each row in three passes through the per-thread cp.async ring:
//   1. from HBM (evict-last): each tensor's (max, sum) -> L_d, L_t, and
//      L_d - L_t from their parts (it keeps the precision of a small number);
//   2. from L2 (d evict-last again, pass 3 reads it once more; t evict-first when
//      pass 3 does not need it): the terms 2^(min(d - L_d, t - L_t) log2e), their
//      sum c* and the p_d mass where d - t < L_d - L_t (P_lt), the terms being
//      p_d there, and whether any element ties (d - t = L_d - L_t);
//      sum_u p_d(u) sgn_u = 1 - 2 P_lt - P_eq, with P_eq the p_d mass of the ties;
//   3. from L2 (evict-first), only with a gradient: dL/dd written with 16-byte
//      evict-first stores.
// A row without ties (all real logits but a set of measure zero) has P_eq = 0
// and sgn_v = +-1 from the one comparison d_v - t_v < L_d - L_t, which pass 2
// leaves as a bit per element in shared memory (a byte per group, nbits groups
// per thread; 19 KB for V = 151936 in bf16): pass 3 then streams d alone.  Where
// the bytes do not fit (nbits = 0) pass 3 streams t again and compares.  A row
// with a tie (d = t, for one) runs pass 2 once more with the sign's three cases,
// summing P_lt and P_eq, and pass 3 with all three.
// sgn_v compares d_v - t_v (exact for bf16 inputs) with L_d - L_t formed from
// the two logsumexps' parts, so a sign is wrong only where |ln(p_d / p_t)| is
// within float32 rounding of the row's logsumexps; for bf16 the exponents are the
// fused x log2e - L log2e (float32 keeps (x - L) log2e).  Each CTA sums its rows'
// totals in row order and the last CTA to finish adds the CTAs' sums in CTA
// order.
template <bool kBF16>
__global__ void __launch_bounds__(kTv2Threads, 1)
loss_three_pass(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, int64_t rows, int V,
                StatusBlock* status, LossArgs la, int nbits) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ;
    extern __shared__ __align__(16) uint8_t tv2_smem[];
    uint4* ring = reinterpret_cast<uint4*>(tv2_smem);
    uint8_t* sbits = tv2_smem + kTv2Smem;               // [nbits][kTv2Threads] sign bytes, 0 if nbits = 0
    __shared__ float4 red[kTv2Threads / 32];
    __shared__ float4 fin;
    __shared__ float4 red_c[kTv2Threads / 32];
    __shared__ float4 fin_c;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ngroups = V / EPG;
    const int nmine = (ngroups > tid) ? (ngroups - tid + kTv2Threads - 1) / kTv2Threads : 0;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    float cta_sum = 0.f;                                  // this CTA's row totals, in row order
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4* gd = reinterpret_cast<const uint4*>(d + static_cast<size_t>(row) * V * ESZ);
        const uint4* gt = reinterpret_cast<const uint4*>(t + static_cast<size_t>(row) * V * ESZ);
        int tgt = la.target[row];
        float dtgt = -INFINITY;
        if (tgt < 0 || tgt >= V) {
            if (tid == 0) set_status(status, DSPARK_ERR_DEVICE_CHECK, 30);
            tgt = -1;
        } else if (tid == 0) {
            const uint8_t* src = d + (static_cast<size_t>(row) * V + tgt) * ESZ;
            dtgt = kBF16 ? bf16lo(*reinterpret_cast<const uint16_t*>(src)) : *reinterpret_cast<const float*>(src);
        }
        // 1: (max, sum) of d and t, from HBM
        float md = -INFINITY, sd = 0.f, mt = -INFINITY, st = 0.f;
        tv2_pass<true, kLossUnroll>(gd, gt, nmine, ring, keep, keep, [&](const uint4 vd, const uint4 vt, int) {
            group_lse<kBF16>(vd, md, sd);
            group_lse<kBF16>(vt, mt, st);
        });
        if (!(md > -INFINITY)) { md = 0.f; sd = 0.f; }
        if (!(mt > -INFINITY)) { mt = 0.f; st = 0.f; }
        tv2_prime(gd, gt, nmine, ring, keep, keep);             // pass 2's first loads fly during the merge
        const float4 P = block_lse2_parts(md, sd, mt, st, red, &fin);
        const float Ld = P.x + P.y, Lt = P.z + P.w;       // natural-log logsumexp
        const float dL = (P.x - P.z) + (P.y - P.w);       // L_d - L_t from the parts
        const bool mass = Ld > -INFINITY && Lt > -INFINITY;
        if (!mass) cp_wait<0>();                          // no mass: the primed loads are dropped
        // 2: c*, P_lt, P_eq, from L2
        // exponents: for bf16 the fused x log2e - L log2e, for float32 (x - L) log2e
        const float sc = kBF16 ? kLog2e : 1.f;
        const unsigned long long L2E = pk(kLog2e, kLog2e), nLd = pk(-Ld * sc, -Ld * sc),
                                 nLt = pk(-Lt * sc, -Lt * sc);
        auto expo = [&](float a0, float a1, unsigned long long nL) -> float2 {
            return kBF16 ? upk(fma2(pk(a0, a1), L2E, nL)) : upk(mul2(add2(pk(a0, a1), nL), L2E));
        };
        unsigned long long pc = pk(0.f, 0.f);
        float plt0 = 0.f, plt1 = 0.f;
        bool tie = false;                                 // some d_v - t_v == L_d - L_t in this thread's groups
        const bool bits = nbits > 0 && la.grad != nullptr;   // pass 3 takes the signs from sbits
        const uint64_t tpol = bits ? drop : keep;
        tv2_pass<true, kLossUnroll>(gd, gt, mass ? nmine : 0, ring, keep, tpol, [&](const uint4 vd, const uint4 vt, int g) {
            float a[EPG], b[EPG];
            unpack<kBF16>(vd, a);
            unpack<kBF16>(vt, b);
            uint32_t m = 0;                               // bit e: d_e - t_e < L_d - L_t
#pragma unroll
            for (int e = 0; e < EPG; e += 2) {
                const float2 x = expo(a[e], a[e + 1], nLd), y = expo(b[e], b[e + 1], nLt);
                // min(p_d, p_t) is p_d exactly where d - t < L_d - L_t: the comparison that
                // decides the sign picks the smaller exponent too
                const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                const bool l0 = r0 < dL, l1 = r1 < dL;
                const float e0 = fast_exp2(l0 ? x.x : y.x), e1 = fast_exp2(l1 ? x.y : y.y);
                pc = add2(pc, pk(e0, e1));
                if (l0) { plt0 += e0; m |= 1u << e; }
                if (l1) { plt1 += e1; m |= 2u << e; }
                tie |= (r0 == dL) | (r1 == dL);
            }
            if (bits) sbits[g] = static_cast<uint8_t>(m);   // g = tid + i T: slot i of this thread
        }, /*primed=*/mass);
        const bool grad3 = la.grad != nullptr && mass;
        if (grad3) {                                      // pass 3's first loads fly during the merge
            if (bits) tv2_prime<false>(gd, gt, nmine, ring, drop, drop);
            else tv2_prime(gd, gt, nmine, ring, drop, drop);
        }
        {
            const float p = warp_sum(upk(pc).x + upk(pc).y), q1 = warp_sum(plt0 + plt1);
            const bool tw = __any_sync(0xffffffffu, tie);
            if (lane == 0) red_c[warp] = make_float4(p, q1, 0.f, tw ? 1.f : 0.f);
            __syncthreads();
            if (warp == 0) {
                const float4 r = (lane < kTv2Threads / 32) ? red_c[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float c0 = warp_sum(r.x), c1 = warp_sum(r.y), c3 = warp_sum(r.w);
                if (lane == 0) fin_c = make_float4(c0, c1, 0.f, c3);
            }
            __syncthreads();
        }
        float4 C = fin_c;                                 // (c*, P_lt, P_eq, ties): P_eq = 0 without ties
        const bool tie_row = C.w > 0.f;                   // block-uniform
        if (tie_row && la.grad != nullptr) {
            // rare: some d_v - t_v equals L_d - L_t exactly, where sgn_v = 0.  Pass 2
            // again, from L2, with P_lt and P_eq summed per element as in the sign's
            // three-way definition.
            cp_wait<0>();                                 // the primed loads have landed: the ring is free
            float plt = 0.f, peq = 0.f;
            tv2_pass<true, kLossUnroll>(gd, gt, nmine, ring, keep, keep, [&](const uint4 vd, const uint4 vt, int) {
                float a[EPG], b[EPG];
                unpack<kBF16>(vd, a);
                unpack<kBF16>(vt, b);
#pragma unroll
                for (int e = 0; e < EPG; e += 2) {
                    const float2 x = expo(a[e], a[e + 1], nLd), y = expo(b[e], b[e + 1], nLt);
                    const float e0 = fast_exp2(fminf(x.x, y.x)), e1 = fast_exp2(fminf(x.y, y.y));
                    const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                    plt += (r0 < dL ? e0 : 0.f) + (r1 < dL ? e1 : 0.f);
                    peq += (r0 == dL ? e0 : 0.f) + (r1 == dL ? e1 : 0.f);
                }
            });
            const float q1 = warp_sum(plt), q2 = warp_sum(peq);
            if (lane == 0) red_c[warp] = make_float4(0.f, q1, q2, 0.f);
            __syncthreads();
            if (warp == 0) {
                const float4 r = (lane < kTv2Threads / 32) ? red_c[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float c1 = warp_sum(r.y), c2 = warp_sum(r.z);
                if (lane == 0) fin_c = make_float4(C.x, c1, c2, C.w);
            }
            __syncthreads();
            C = fin_c;
            tv2_prime(gd, gt, nmine, ring, drop, drop);
        }
        const float sbar = 1.f - 2.f * C.y - C.z;         // sum_u p_d(u) sign(p_d(u) - p_t(u))
        const float om = la.omega[row];
        // 3: dL/dd, from L2, written once
        if (la.grad != nullptr) {
            // dL/dd_v = p_d(v) (ka + kl (sgn_v - sbar)) - ka [v = target]
            const float ka = om * la.a_ce, kl = 0.5f * om * la.a_l1;
            const float c0 = ka - kl * sbar, cp = c0 + kl, cm = c0 - kl;
            const int tg = tgt >= 0 ? tgt / EPG : -1;     // the target's group
            uint8_t* grow = static_cast<uint8_t*>(la.grad) + static_cast<size_t>(row) * V * ESZ;
            // kMode 0: the sign's three cases; 1 (no tie in the row): two; 2 (no tie, signs
            // kept by pass 2): two, read from sbits, d alone streamed
            auto grad_pass = [&](auto mode) {
                constexpr int kMode = decltype(mode)::value;
                const int n3 = mass ? nmine : 0;
                tv2_pass<kMode != 2, kLossUnroll>(gd, gt, n3, ring, drop, drop, [&](const uint4 vd, const uint4 vt, int g) {
                    float a[EPG], b[EPG], gv[EPG];
                    unpack<kBF16>(vd, a);
                    uint32_t m = 0;
                    if constexpr (kMode == 2) m = sbits[g];
                    else unpack<kBF16>(vt, b);
#pragma unroll
                    for (int e = 0; e < EPG; e += 2) {
                        const float2 z = expo(a[e], a[e + 1], nLd);
                        const float p0 = fast_exp2(z.x), p1 = fast_exp2(z.y);
                        if constexpr (kMode == 0) {
                            const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                            gv[e] = p0 * (r0 > dL ? cp : (r0 < dL ? cm : c0));
                            gv[e + 1] = p1 * (r1 > dL ? cp : (r1 < dL ? cm : c0));
                        } else if constexpr (kMode == 1) {
                            const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                            gv[e] = p0 * (r0 < dL ? cm : cp);
                            gv[e + 1] = p1 * (r1 < dL ? cm : cp);
                        } else {
                            gv[e] = p0 * ((m >> e) & 1u ? cm : cp);
                            gv[e + 1] = p1 * ((m >> (e + 1)) & 1u ? cm : cp);
                        }
                    }
                    if (g == tg) {
#pragma unroll
                        for (int e = 0; e < EPG; ++e)
                            if (g * EPG + e == tgt) gv[e] -= ka;
                    }
                    uint4 o;
                    if constexpr (kBF16) {
                        o.x = pack_bf16(gv[0], gv[1]); o.y = pack_bf16(gv[2], gv[3]);
                        o.z = pack_bf16(gv[4], gv[5]); o.w = pack_bf16(gv[6], gv[7]);
                    } else {
                        o = make_uint4(__float_as_uint(gv[0]), __float_as_uint(gv[1]), __float_as_uint(gv[2]),
                                       __float_as_uint(gv[3]));
                    }
                    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(grow + g * 16),
                                 "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w), "l"(drop)
                                 : "memory");
                }, /*primed=*/grad3);
            };
            if (tie_row) grad_pass(std::integral_constant<int, 0>{});
            else if (bits) grad_pass(std::integral_constant<int, 2>{});
            else grad_pass(std::integral_constant<int, 1>{});
        }
        if (tid == 0) {
            const float sv = la.s[row];
            const float ce = Ld - dtgt;
            const float sp = fmaxf(sv, 0.f) + log1pf(expf(-fabsf(sv)));   // softplus
            const float bce = sp - C.x * sv;
            const float tot = om * (la.a_ce * ce + la.a_l1 * (1.f - C.x) + la.a_conf * bce);
            reinterpret_cast<float4*>(la.row_out)[row] = make_float4(ce, C.x, bce, tot);
            if (la.grad_s != nullptr) la.grad_s[row] = om * la.a_conf * (1.f / (1.f + expf(-sv)) - C.x);
            cta_sum += tot;
        }
        // red, fin, red_c and fin_c are rewritten by the next row after barriers
    }
    if (tid == 0) {
        la.cl_part[blockIdx.x] = cta_sum;
        __threadfence();
        if (atomicAdd(la.cl_done, 1u) == gridDim.x - 1u) {
            __threadfence();
            float tot = 0.f;
            for (unsigned int c = 0; c < gridDim.x; ++c) tot += __ldcg(la.cl_part + c);
            *la.loss = tot;
        }
    }
}

template <bool kBF16>
dspark_status_t launch_loss_three_pass(int64_t rows, int V, const void* d, const void* t, StatusBlock* status,
                                       const LossArgs& la, cudaStream_t stream) {
    const int dev = current_device();
    static OncePerDevice once;
    if (once.run(dev, [] {
            return cudaFuncSetAttribute(loss_three_pass<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kLossSmemMax));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    int sms = sm_count(dev);
    if (sms > kMaxLossCtas) sms = kMaxLossCtas;
    const int64_t grid = rows < sms ? rows : sms;
    // a sign byte per group for every thread's groups, when they fit beside the ring
    const int ngroups = V / TVTraits<kBF16>::kEPG;
    const int per_thread = (ngroups + kTv2Threads - 1) / kTv2Threads;
    const int nbits = (la.grad != nullptr && per_thread <= kLossMaxBitGroups) ? per_thread : 0;
    const size_t smem = kTv2Smem + static_cast<size_t>(nbits) * kTv2Threads;
    loss_three_pass<kBF16><<<static_cast<unsigned>(grid), kTv2Threads, smem, stream>>>(
        static_cast<const uint8_t*>(d), static_cast<const uint8_t*>(t), rows, V, status, la, nbits);
    return launch_status();
}

template <bool kBF16>
dspark_status_t launch_tv_two_pass(int64_t rows, int V, const void* d, const void* t, float* c_star,
                                   cudaStream_t stream) {
    const int dev = current_device();
    static OncePerDevice once;
    if (once.run(dev, [] {
            return cudaFuncSetAttribute(tv_two_pass<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kTv2Smem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int sms = sm_count(dev);
    const int64_t grid = rows < sms ? rows : sms;
    tv_two_pass<kBF16><<<static_cast<unsigned>(grid), kTv2Threads, kTv2Smem, stream>>>(
        static_cast<const uint8_t*>(d), static_cast<const uint8_t*>(t), c_star, rows, V);
    return launch_status();
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_accept_rate_tv_workspace_size(int64_t rows, int V) {
    (void)rows;
    (void)V;
    return kStatusBytes;
}

extern "C" dspark_status_t dspark_accept_rate_tv(int64_t rows, int V, dspark_dtype_t dt, const void* d,
                                                 const void* t, float* c_star, void* workspace,
                                                 size_t workspace_bytes, dspark_stream_t stream) {
    if (rows < 0 || V <= 0 || (dt != DSPARK_F32 && dt != DSPARK_BF16)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_accept_rate_tv_workspace_size(rows, V)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    if (rows == 0) return DSPARK_OK;
    if (d == nullptr || t == nullptr || c_star == nullptr) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!aligned16(d) || !aligned16(t)) return DSPARK_ERR_INVALID_ARGUMENT;
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_status(workspace, s) != DSPARK_OK) return DSPARK_ERR_CUDA;
    return dt == DSPARK_BF16 ? launch_tv_two_pass<true>(rows, V, d, t, c_star, s)
                             : launch_tv_two_pass<false>(rows, V, d, t, c_star, s);
}

// Workspace of the loss: status block | CTA counter (own 256 bytes) | one
// float per CTA.
extern "C" size_t dspark_training_loss_workspace_size(int64_t rows, int V) {
    (void)rows;
    (void)V;
    return kStatusBytes + 256 + static_cast<size_t>(kMaxLossCtas) * sizeof(float);
}

extern "C" dspark_status_t dspark_training_loss(int64_t rows, int V, dspark_dtype_t dt, const void* d,
                                                const void* t, const int32_t* target, const float* conf_logit,
                                                const float* omega, float alpha_ce, float alpha_l1,
                                                float alpha_conf, float* row_out, float* loss, void* grad_d,
                                                float* grad_conf, void* workspace, size_t workspace_bytes,
                                                dspark_stream_t stream) {
    if (rows < 0 || V <= 0 || (dt != DSPARK_F32 && dt != DSPARK_BF16)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_training_loss_workspace_size(rows, V)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    if (loss == nullptr) return DSPARK_ERR_INVALID_ARGUMENT;
    if (rows > 0) {
        if (d == nullptr || t == nullptr || target == nullptr || conf_logit == nullptr || omega == nullptr ||
            row_out == nullptr)
            return DSPARK_ERR_INVALID_ARGUMENT;
        if (!aligned16(d) || !aligned16(t) || !aligned16(row_out)) return DSPARK_ERR_INVALID_ARGUMENT;
        if (grad_d != nullptr && !aligned16(grad_d)) return DSPARK_ERR_INVALID_ARGUMENT;
    }
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // status and the CTA counter
    if (cudaMemsetAsync(workspace, 0, kStatusBytes + 256, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (rows == 0) return cudaMemsetAsync(loss, 0, sizeof(float), s) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
    StatusBlock* st = static_cast<StatusBlock*>(workspace);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    LossArgs la{};
    la.target = target;
    la.s = conf_logit;
    la.omega = omega;
    la.a_ce = alpha_ce;
    la.a_l1 = alpha_l1;
    la.a_conf = alpha_conf;
    la.row_out = row_out;
    la.grad = grad_d;
    la.grad_s = grad_conf;
    la.cl_done = reinterpret_cast<unsigned int*>(base + kStatusBytes);
    la.cl_part = reinterpret_cast<float*>(base + kStatusBytes + 256);
    la.loss = loss;
    return dt == DSPARK_BF16 ? launch_loss_three_pass<true>(rows, V, d, t, st, la, s)
                             : launch_loss_three_pass<false>(rows, V, d, t, st, la, s);
}
