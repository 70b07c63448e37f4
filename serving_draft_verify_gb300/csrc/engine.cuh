// The bias engine shared by dspark_draft_block and dspark_verify: for a set of
// request rows, each with a position k_b, it forms the draft logits
//   z_b = U[b][k_b-1] + W2 . W1[x_{k_b-1}]       (VanillaMarkovHead, eq. 5;
//                                                 DeepSpec walkthrough 3.2)
// tile by tile on the tensor cores and reduces them in its epilogue:
//   kDraft     the running (max, sum) of 2^y, y = z log2e / T (the draft's
//              log-normaliser), and the Gumbel-max draw over the vocabulary:
//              the token maximising y_v - log2 E_v, E_v = -ln u_v with u_v
//              from the Philox word of (request, position, index v, stream 0);
//              greedy: the running argmax of z;
//   kResidual  the Gumbel-max draw from the residual max(0, p_t - p_d)
//              (section 8.2): the token maximising q_v / E_v, stream 2.
// Inside a 32-token sub-block the draw is an exponential race with an exact
// filter: with e_v = 2^(y_v - m) (already formed for the sum) and R = 2^(m - best)
// for the thread's running best key, token v can win only if E_v < e_v R, and
// since E_v >= s_v = 1 - u_v (exact from the word) a token with s_v >= e_v R is
// skipped; only the rare others take E_v and the exact key y_v - log2 E_v, each
// lane walking its own candidate bits in ascending order.
// Each CTA publishes its best token per row with a 64-bit atomicMax of
// (key, ~token) and, for kDraft, its (max, sum) partial and the y of its best
// token (for log p_d of the token that wins overall).
//
// Layout of one CTA (512 threads, one CTA per SM; 128 registers a thread at
// launch, then 56 for warpgroup 0 and 152 for the epilogue warpgroups):
//   warp 0      TMA producer: W2 tiles [128 tokens x 64 K] into a slab ring
//               (128-byte swizzle, L2 evict-last so W2 stays resident);
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M = 128 request rows, N = 128 tokens, K = r, fp32 in TMEM;
//   warps 4-15  three epilogue warpgroups sharing four TMEM accumulators in
//               rotation (a position's tile i: warpgroup i mod 3; the launch's
//               tile g: accumulator g mod 4), so the MMA of the next tile
//               overlaps the epilogues of the others.
// The A operand (rows W1[x_{k_b-1}], or the rows E[b][k_b] of a gated or
// recurrent head, gathered into shared memory with the same swizzle) is built
// by warps 1-15 at the start of every position.
//
// Draft launches may cover positions k .. k_last (a cooperative launch, all
// CTAs resident, TMEM and barriers set up once, the producer streaming W2
// straight through all positions).  Between positions the grid meets at a
// bounded counter barrier; the published word of each request then names
// x_{k} directly, and every CTA reads the tokens of its own M-tile.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "tc.cuh"

namespace dspark {
namespace eng {

constexpr int kMaxChunks = 160;   // partial slots per (position, request): at least the SM count

struct Ws {
    StatusBlock* status;
    unsigned long long* words;   // [positions][B] best (key, ~token)
    float2* part;                // [positions][B][kMaxChunks] (max, sum) of y = z log2e / T
    float* ybest;                // [positions][B][kMaxChunks] y of each chunk's best token
    unsigned int* gbar;          // grid-barrier counter of the multi-position draft launch (starts at 0)
};

// ------------------------------------------------------------ helpers ---
__device__ __forceinline__ uint32_t f2ord(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ unsigned long long pack_key(float key, uint32_t idx) {
    return (static_cast<unsigned long long>(f2ord(key)) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ uint32_t unpack_idx(unsigned long long w) { return ~static_cast<uint32_t>(w); }

// Chunk c of `nchunk` that covers unit u when `nunits` units are split into
// the contiguous ranges [c nunits / nchunk, (c + 1) nunits / nchunk).
__host__ __device__ __forceinline__ int chunk_of(int u, int nunits, int nchunk) {
    return static_cast<int>(((static_cast<long long>(u) + 1) * nchunk - 1) / nunits);
}

template <bool kBF16>
__device__ __forceinline__ float ld_elem(const void* p, size_t i) {
    if constexpr (kBF16) {
        return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16);
    } else {
        return static_cast<const float*>(p)[i];
    }
}

__device__ __forceinline__ void ld_u32x4(const void* p, uint32_t* o, uint64_t pol) {
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
                 : "l"(p), "l"(pol));
}

// Token x_{k-1} of request b (the anchor for k = 1), checked against [0, V).
// x may have been written by other CTAs of a running grid: read it from L2.
__device__ __forceinline__ int prev_token(const int32_t* x0, const int32_t* x, int b, int gamma, int k, int V,
                                          StatusBlock* st) {
    const int t = (k == 1) ? x0[b] : __ldcg(x + b * gamma + k - 2);
    if (t < 0 || t >= V) {
        set_status(st, DSPARK_ERR_DEVICE_CHECK, 2);
        return 0;
    }
    return t;
}

// Combine (m1, s1) += (m2, s2) for sums of 2^(y - m).
__device__ __forceinline__ void lse_merge(float& m1, float& s1, float m2, float s2) {
    if (s2 <= 0.f) return;
    if (s1 <= 0.f) { m1 = m2; s1 = s2; return; }
    const float M = fmaxf(m1, m2);
    s1 = s1 * exp2f(m1 - M) + s2 * exp2f(m2 - M);
    m1 = M;
}

// The rank-r row behind the bias of position k of request b: W1[x_{k-1}] for the
// Markov head (E null), else row (b, k) of the rows E [B][gamma][r] that a
// gated or recurrent head produced.
template <bool kBF16>
__device__ __forceinline__ const void* bias_row(const void* E, const void* W1, int b, int gamma, int k, int r,
                                                int prev) {
    const size_t row = E ? static_cast<size_t>(b) * gamma + (k - 1) : static_cast<size_t>(prev);
    return static_cast<const uint8_t*>(E ? E : W1) + row * r * (kBF16 ? 2 : 4);
}

// Running Gumbel-max state of one thread: the best key so far (log2 units),
// its token and its y.  Tokens reach a thread in ascending order, so a strict
// comparison keeps the lowest index on ties.
struct Best {
    float key;
    int idx;
    float y;
};
__device__ __forceinline__ void best_take(Best& b, float key, int idx, float y) {
    if (key > b.key || (key == b.key && idx < b.idx)) { b.key = key; b.idx = idx; b.y = y; }
}

// The draws' candidate test: s = 1 - u for u = ((w >> 9) + 1/2) 2^-23 is a lower
// bound of E = -ln u (since -ln(1 - s) >= s), so a token whose s already exceeds the
// bound on E that could beat the running best cannot win.
// f = 1 + m 2^-23 for m = w >> 9 (one funnel shift puts the exponent bits above m).
// Then s = 1 - u = 2 - f - 2^-24 exactly, so s < X  <=>  f > 2 - 2^-24 - X; callers test
// f > fma(X, -1, kTopU): kTopU = 2 - 2^-22 sits 3 2^-24 below 2 - 2^-24, more than the
// fma's rounding (at most 2^-24 at these magnitudes), so no candidate is dropped.
constexpr float kTopU = 1.99999976158142089844f;   // 2 - 2^-22
__device__ __forceinline__ float one_plus_m(uint32_t w) { return __uint_as_float(__funnelshift_r(w, 0x7Fu, 9)); }

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// lo += float(low bf16 of w), hi += float(high bf16 of w): the bf16 -> float32 widening
// is exact, so each result is the float32 sum rounded once, as with an explicit widening.
__device__ __forceinline__ void add_bf16_pair(uint32_t w, float& lo, float& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.f32.bf16 %0, l, %0;\n\tadd.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w));
}

// Two float32 lanes in one 64-bit register (Blackwell f32x2 arithmetic); each lane
// of an f32x2 operation is rounded once, exactly as its float32 counterpart.
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// The flat Gumbel-max draw over 32 consecutive tokens v0 .. v0+31 (v0 a
// multiple of 4), given their raw logits s (-inf: no mass) and the scale c > 0
// (y = s c in log2 units), and their (max, sum) of 2^y.
// Token v beats the running best iff y_v - log2 E_v > best.key, i.e. iff
// E_v < 2^(y_v - best.key) = e_v R with e_v = 2^(y_v - m) (formed for the sum
// anyway) and R = 2^(m - best.key).  Since E_v >= s_v = 1 - u_v, a token with
// s_v >= e_v R (R raised by 2^-10 to cover the rounding of e_v, R and E_v)
// cannot win, and only the rare others (a warp enters the branch when any lane
// has one) take E_v and the exact comparison of keys.  Tokens are visited in
// ascending order and a key must be strictly larger to win: ties keep the
// lowest index.  `pr` holds the row's Philox constants; word v & 3 of block
// v >> 2 keys index v.
__device__ __forceinline__ void draw32(const float* s, float c, int v0, const PhiloxRow& pr, const PhiloxKeys& K,
                                       Best& best, float& M, float& S) {
    // the sub-block's max by three-input maxima (max is exact: any grouping gives the same value)
    float m3[11];
#pragma unroll
    for (int w = 0; w < 10; ++w) m3[w] = fmax3(s[w], s[w + 10], s[w + 20]);
    m3[10] = fmaxf(s[30], s[31]);
    const float mraw = fmax3(fmax3(m3[0], m3[1], m3[2]), fmax3(m3[3], m3[4], m3[5]),
                             fmax3(fmax3(m3[6], m3[7], m3[8]), m3[9], m3[10]));
    const bool live = mraw > -INFINITY;                   // no finite logit: no mass, no candidate
    const float mb = mraw * c;                            // the sub-block's max of y
    const float mref = live ? mb : 0.f;
    constexpr float kSlack = 1.0009765625f;               // 1 + 2^-10
    // s_v < e_v R  <=>  f_v > 2 - 2^-24 - e_v R (f_v = one_plus_m(w_v)), tested against kTopU
    const float nR = live ? -(fast_exp2(mb - best.key) * kSlack) : 0.f;   // -inf while nothing is drawn yet
    const unsigned long long c2 = f2pack(c, c), nm2 = f2pack(-mref, -mref);
    unsigned long long sum2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};   // two chains of partial sums
    const uint32_t q0 = static_cast<uint32_t>(v0) >> 2;
    // per half of 16 tokens: its four Philox blocks first (independent chains the scheduler
    // can overlap), then the sum (e = 2^(s c - m), two tokens per f32x2 operation) and the
    // candidates (a bit per token), then -- rare -- E_v and the exact comparison for the
    // candidates, in ascending order
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t wv[16];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const U4 pw = philox_row(pr, q0 + 4 * hh + qq, K);
            wv[4 * qq] = pw.x;
            wv[4 * qq + 1] = pw.y;
            wv[4 * qq + 2] = pw.z;
            wv[4 * qq + 3] = pw.w;
        }
        uint32_t cm[4] = {0u, 0u, 0u, 0u};                // four independent chains of candidate bits
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            float a0, a1;
            f2unpack(f2fma(f2pack(s[16 * hh + i], s[16 * hh + i + 1]), c2, nm2), a0, a1);
            const float e0 = fast_exp2(a0), e1 = fast_exp2(a1);
            sum2[(i >> 1) & 1] = f2add(sum2[(i >> 1) & 1], f2pack(e0, e1));
            if (one_plus_m(wv[i]) > fmaf(e0, nR, kTopU)) cm[(i >> 1) & 3] |= 1u << i;   // 0 * -inf = NaN: false
            if (one_plus_m(wv[i + 1]) > fmaf(e1, nR, kTopU)) cm[(i >> 1) & 3] |= 2u << i;
        }
        const uint32_t cmask = (cm[0] | cm[1]) | (cm[2] | cm[3]);
        if (__any_sync(0xffffffffu, cmask != 0u)) {
            // each lane walks its own candidates of each group of four, lowest first (the
            // warp runs as many steps as its busiest lane, not one per bit position)
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t bits = (cmask >> (4 * qq)) & 0xFu;
                const int g = 16 * hh + 4 * qq;
                while (bits != 0u) {
                    const int j = __ffs(bits) - 1;
                    bits &= bits - 1u;
                    const float sj = j == 0 ? s[g] : j == 1 ? s[g + 1] : j == 2 ? s[g + 2] : s[g + 3];
                    const uint32_t wj = j == 0 ? wv[4 * qq] : j == 1 ? wv[4 * qq + 1]
                                                   : j == 2 ? wv[4 * qq + 2] : wv[4 * qq + 3];
                    const float yj = sj * c;
                    const float key = yj - fast_log2(exp_draw(wj));
                    if (key > best.key) {
                        best.key = key;
                        best.idx = v0 + g + j;
                        best.y = yj;
                    }
                }
            }
        }
    }
    float sl, sh;
    f2unpack(f2add(sum2[0], sum2[1]), sl, sh);
    if (live) lse_merge(M, S, mb, sl + sh);
}

// Grid barrier of the multi-position draft launch (cooperative launch: every CTA
// is resident).  Epoch e is complete once the counter reaches e * gridDim.x;
// every CTA arrives once per epoch.  Waits are bounded (kWaitLimitNs).
__device__ __forceinline__ void grid_arrive(unsigned int* ctr) {
    __threadfence();
    atomicAdd(ctr, 1u);
}
__device__ __forceinline__ bool grid_wait(const unsigned int* ctr, unsigned int target,
                                          uint64_t limit_ns = kWaitLimitNs) {
    auto load = [&]() {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        return v;
    };
    if (load() >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (load() < target) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Warp dot product of n elements of a[a_off..] and b[b_off..] (16-byte chunks
// when both are aligned); lane partial sums, reduced by the caller.
template <bool kBF16>
__device__ __forceinline__ float dot_row(const void* a, size_t a_off, const void* b, size_t b_off, int n, int lane) {
    constexpr int EPC = kBF16 ? 8 : 4;
    constexpr size_t ESZ = kBF16 ? 2 : 4;
    float acc = 0.f;
    const bool vec = ((a_off * ESZ) % 16 == 0) && ((b_off * ESZ) % 16 == 0) && (n % EPC == 0);
    if (vec) {
        const uint4* pa = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a) + a_off * ESZ);
        const uint4* pb = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(b) + b_off * ESZ);
        // four chunks of each operand in flight per lane, accumulated in chunk order
        const int nc = n / EPC;
        for (int c0 = lane; c0 < nc; c0 += 4 * 32) {
            uint4 xs[4], ys[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * 32;
                xs[u] = (c < nc) ? pa[c] : make_uint4(0, 0, 0, 0);
                ys[u] = (c < nc) ? pb[c] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (c0 + u * 32 >= nc) break;
                const uint32_t xv[4] = {xs[u].x, xs[u].y, xs[u].z, xs[u].w};
                const uint32_t yv[4] = {ys[u].x, ys[u].y, ys[u].z, ys[u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (kBF16) {
                        acc = fmaf(bf16lo(xv[q]), bf16lo(yv[q]), acc);
                        acc = fmaf(bf16hi(xv[q]), bf16hi(yv[q]), acc);
                    } else {
                        acc = fmaf(__uint_as_float(xv[q]), __uint_as_float(yv[q]), acc);
                    }
                }
            }
        }
    } else {
        for (int i = lane; i < n; i += 32) acc = fmaf(ld_elem<kBF16>(a, a_off + i), ld_elem<kBF16>(b, b_off + i), acc);
    }
    return acc;
}

// One warp finalizes position k of request b (DeepSpec walkthrough 3.3,
// AcceptRatePredictor): lse_d = logsumexp(z / T) from the nchunk (max, sum)
// partials, logp_d = y(x_k) - lse_d with y(x_k) taken from the chunk that
// covers x_k (its best token is x_k: the overall winner is the best of the
// chunk it lies in), and the confidence c = sigmoid(w . [h_k ; W1[x_{k-1}]] + bias),
// written by lane 0.  Chunk c covers units [c nunits / nchunk, (c+1) nunits /
// nchunk) of `unit` tokens each.
template <bool kBF16>
__device__ __forceinline__ void finalize_position(int b, int k, int B, int gamma, int V, int H, int r, const void* h,
                                                  const void* W1, const void* w, float bias, const int32_t* x0,
                                                  const int32_t* x, int greedy, int nchunk, int unit, int nunits,
                                                  const float2* part, const float* ybest, float* lse_d,
                                                  float* logp_d, float* c, StatusBlock* st) {
    const int lane = threadIdx.x & 31;
    const size_t slot = static_cast<size_t>(k - 1) * B + b;
    const size_t o = static_cast<size_t>(b) * gamma + (k - 1);
    float L = 0.f, lp = 0.f;
    if (!greedy) {
        float m = -INFINITY, s = 0.f;
        constexpr int kPer = (kMaxChunks + 31) / 32;
        float2 pr[kPer];                                  // every partial of this lane in flight at once
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int ch = lane + 32 * u;
            pr[u] = (ch < nchunk) ? __ldcg(part + slot * kMaxChunks + ch) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            if (lane + 32 * u < nchunk) lse_merge(m, s, pr[u].x, pr[u].y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, off);
            const float os = __shfl_xor_sync(0xffffffffu, s, off);
            lse_merge(m, s, om, os);
        }
        const float L2 = m + log2f(s);
        int tok = __ldcg(x + o);
        if (tok < 0 || tok >= V) tok = 0;                 // reported where x was written
        const float ytok = __ldcg(ybest + slot * kMaxChunks + chunk_of(tok / unit, nunits, nchunk));
        L = L2 * kLn2;
        lp = (ytok - L2) * kLn2;
    }
    const int prev = prev_token(x0, x, b, gamma, k, V, st);
    float acc = dot_row<kBF16>(w, 0, h, o * H, H, lane);
    acc += dot_row<kBF16>(w, H, W1, static_cast<size_t>(prev) * r, r, lane);
    const float logit = warp_sum(acc) + bias;
    if (lane == 0) {
        c[o] = 1.f / (1.f + expf(-logit));
        lse_d[o] = L;
        logp_d[o] = lp;
    }
}

// ===================================================== tcgen05 engine ====
constexpr int kBM = 128;              // request rows per M-tile (TMEM lanes)
constexpr int kBN = 128;              // vocabulary columns per tile
constexpr int kBK = 64;               // K per smem slab (128 bytes of bf16)
constexpr int kStages = 8;            // W2 slab ring
constexpr int kEpiWG = 3;             // epilogue warpgroups
constexpr int kTmemBufs = 4;          // TMEM accumulators of kBN columns (all 512), used in rotation
constexpr int kTcThreads = 128 * (1 + kEpiWG);
// Registers a thread: 128 at launch (512 threads, the whole register file), then
// warpgroup 0 drops to kCtlRegs and the three epilogue warpgroups rise to kEpiRegs
// (per scheduler: one warp of the first and three of the others, 56 + 3 x 152 = 4 x 128).
constexpr uint32_t kLaunchRegs = 65536 / kTcThreads;
constexpr uint32_t kCtlRegs = 56;
constexpr uint32_t kEpiRegs = 152;
static_assert(kCtlRegs + kEpiWG * kEpiRegs <= (1 + kEpiWG) * kLaunchRegs, "register split over the launch's total");
template <int R>
struct RoleTag {
    static constexpr int value = R;
};
// setmaxnreg: the warpgroup's registers a thread (every warp of the warpgroup executes it)
template <uint32_t N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
constexpr int kPairs = (kTcThreads / 32 - 2) / 2;   // warp pairs of the residual launch's final step
constexpr int kSlabBytes = kBN * kBK * 2;     // 16 KB
constexpr int kASlabBytes = kBM * kBK * 2;    // 16 KB

enum Mode : int { kDraft = 0, kResidual = 1 };

// What the final-token step of verification reads and writes (section 8.2):
// a request rejected at k takes the residual's winner, or, when the residual
// has no mass, a draw from p_t at row k (stream 2 at (b, k)).  Requests with
// no rejection got their bonus token from the rows pass.
struct FinishArgs {
    const uint16_t* T;               // t_logits [B][gamma+1][V] (bf16, or fp32 read through Tf)
    const float* Tf;                 // the same rows when they are fp32 (else null)
    const int32_t* krow;             // [B] rejected position (0: none)
    const unsigned long long* res_word;   // [B] residual winner (key, ~token), 0: no mass
    int32_t* next_token;             // [B]
};

struct TcParams {
    int B, gamma, V, r, k;           // k: the position of every row (kDraft)
    const uint16_t* U;               // [B][gamma][V]
    const uint16_t* W1;              // [V][r]
    const uint16_t* E;               // [B][gamma][r] bias rows of a gated / recurrent head, or null (W1[x_{k-1}])
    const uint16_t* W2;              // [V][r]
    const int32_t* x0;               // [B]
    int32_t* x;                      // [B][gamma]; kDraft writes x_{k-1} here (CTA 0 of each M-tile)
    float cscale;                    // log2e / T (1 for greedy)
    int greedy;
    uint64_t seed;
    PhiloxKeys keys;                 // the round keys of `seed`
    int P;                           // CTAs per M-tile
    Ws ws;
    float* debug_z;                  // kDraft: write y to [B][V] instead of reducing
    int k_last;                      // kDraft: positions k .. k_last in one (cooperative) launch
    // kDraft with fuse_tail: the launch also writes x_gamma and finalizes
    // (lse_d, logp_d, confidence c and survival a), as draft_finalize does
    int fuse_tail;
    int H;
    const uint16_t* h;               // [B][gamma][H]
    const uint16_t* w;               // [H + r]
    float bias;
    float* lse_d;
    float* logp_d;
    float* c;
    float* a;
    // kResidual with fuse_tail: the launch also writes the final tokens
    FinishArgs fin;
    // kResidual
    const int32_t* krow;             // [B] rejected position k_b (0: row inactive)
    const uint16_t* T;               // t_logits [B][gamma+1][V]
    const float* lt2;                // [B] log2-sum-exp2 of t / T at row k_b (log2 units)
    const float* ld2;                // [B] lse_d[b][k_b-1] * log2e
    const int32_t* rej_list;         // [B] the rejected requests (first *rej_count entries, any order)
    const int32_t* rej_count;        // [1]
};

struct RowRes {
    Best best;
    float m, s;
};

// OR of `v` over the 64 threads of named barrier `bar`.
__device__ __forceinline__ bool pair_any(bool v, int bar) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 64, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(bar)
        : "memory");
    return r != 0;
}

// The final token of request b (two warps, named barrier `bar`; xch/xchi: a
// 2-entry exchange) when its draft was rejected at k = krow[b]: the residual's
// winner, or -- if the residual has no mass after rounding -- a Gumbel-max draw
// from p_t = softmax(t_k / T) over the whole row (stream 2 at (b, k)), taken
// by the two warps together.  Requests with no rejection are left alone: the
// rows pass wrote their bonus token.
template <bool kBF16>
__device__ __forceinline__ void finish_pair(const FinishArgs& f, int b, int gamma, int V, float cscale, uint64_t seed,
                                            StatusBlock* st, int bar, float* xch, int* xchi) {
    const int lane = threadIdx.x & 31, wp = (threadIdx.x >> 5) & 1, pt = threadIdx.x & 63;
    const int kr = f.krow[b];
    if (kr <= 0) return;
    const unsigned long long rw = __ldcg(f.res_word + b);
    if (rw != 0ull && unpack_idx(rw) < static_cast<uint32_t>(V)) {
        if (pt == 0) f.next_token[b] = static_cast<int>(unpack_idx(rw));
        return;
    }
    // no residual mass: the draw from p_t at row kr, four consecutive tokens per thread and step
    const PhiloxRow pr = philox_row_setup(seed, static_cast<uint32_t>(kr), static_cast<uint32_t>(b), kStreamVerifyToken);
    const size_t row = (static_cast<size_t>(b) * (gamma + 1) + (kr - 1)) * V;
    Best best{-INFINITY, 0x7FFFFFFF, 0.f};
    for (int q = pt; q * 4 < V; q += 64) {
        const U4 pw = philox_row(pr, static_cast<uint32_t>(q));
        const uint32_t wv[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int v = 4 * q + j;
            if (v < V) {
                const float y = (kBF16 ? ld_elem<true>(f.T, row + v) : f.Tf[row + v]) * cscale;
                best_take(best, y - fast_log2(exp_draw(wv[j])), v, y);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, best.key, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best.idx, o);
        best_take(best, ok, oi, 0.f);
    }
    if (lane == 0) { xch[wp] = best.key; xchi[wp] = best.idx; }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
    if (pt == 0) {
        int w = 0;
        if (xch[1] > xch[0] || (xch[1] == xch[0] && xchi[1] < xchi[0])) w = 1;
        int tok = xchi[w];
        if (tok < 0 || tok >= V) { set_status(st, DSPARK_ERR_DEVICE_CHECK, 7); tok = 0; }
        f.next_token[b] = tok;
    }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
}

template <int kMode>
__global__ void __launch_bounds__(kTcThreads, 1)
bias_engine_tc(const __grid_constant__ CUtensorMap tmW2, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int nslab = p.r / kBK;
    uint8_t* sA = smem;                                   // nslab x 16 KB
    uint8_t* sB = smem + 4 * kASlabBytes;                 // kStages x 16 KB
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kSlabBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;                    // [kTmemBufs]
    uint64_t* tempty = tfull + kTmemBufs;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + kTmemBufs);
    RowRes* rowres = reinterpret_cast<RowRes*>(tmem_slot + 4);   // [kEpiWG][128]
    int* s_prev = reinterpret_cast<int*>(rowres + kEpiWG * kBM);   // [128] x_{k-1} per request row
    float* xch = reinterpret_cast<float*>(s_prev + kBM);          // [2 kPairs] pair exchange
    int* xchi = reinterpret_cast<int*>(xch + 2 * kPairs);         // [2 kPairs]
    int* s_fail = xchi + 2 * kPairs;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The rows of the launch: every request (kDraft), or the rejected ones, listed on
    // the device by verification's rows pass (kResidual): nact of them, rows
    // compacted so that the whole grid works on the M-tiles that exist.
    const int nact = (kMode == kResidual) ? min(max(__ldcg(p.rej_count), 0), p.B) : p.B;
    // Row replication: with at most 64 rows the A tile holds every row twice (TMEM
    // lanes 0-63 and 64-127), with at most 32 four times (lanes 32 c .. 32 c + 31 for
    // copy c), and the copies reduce different parts (halves, quarters) of each tile,
    // so more epilogue lanes have work at small batches.
    const int R = (nact <= 32) ? 4 : (nact <= 64) ? 2 : 1;
    const int rpc = kBM / R;                              // request rows per copy
    const int nM = max(1, (nact + kBM - 1) / kBM);        // M-tiles (one when R = 2)
    const int NT = (p.V + kBN - 1) / kBN;
    // CTAs per M-tile: the host's P for the draft; for the residual, as many as the
    // grid gives each existing M-tile (CTAs past them stay idle)
    const int P = (kMode == kResidual) ? max(1, min(static_cast<int>(gridDim.x) / nM, NT)) : p.P;
    const int g = blockIdx.x / P, pc = blockIdx.x % P;
    const int m0 = g * kBM;
    const bool idle = g >= nM;
    const int t_lo = idle ? 0 : static_cast<int>(static_cast<long long>(pc) * NT / P);
    const int t_hi = idle ? 0 : static_cast<int>(static_cast<long long>(pc + 1) * NT / P);
    const int ntiles = t_hi - t_lo;
    StatusBlock* st = p.ws.status;
    const int nrows = idle ? 0 : max(0, min(rpc, nact - m0));   // rows of this M-tile
    // the request behind row m0 + rr
    auto req = [&](int rr) -> int { return (kMode == kResidual) ? __ldcg(p.rej_list + m0 + rr) : m0 + rr; };
    const int k0 = p.k;
    const int k1 = (kMode == kDraft && p.k_last > p.k) ? p.k_last : p.k;
    const bool multi = k1 > k0;                           // positions k0..k1, grid barriers between
    auto row_k = [&](int b, int k) -> int { return (kMode == kResidual) ? p.krow[b] : k; };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int e = 0; e < kTmemBufs; ++e) { mbar_init(&tfull[e], 1); mbar_init(&tempty[e], 4); }
        *s_fail = 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tmW2);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    {
        constexpr int kPro = kTcThreads - 32;             // warps 1.. : prologue, MMA, epilogue
        const int ptid = tid - 32;
        auto pro_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kPro) : "memory"); };
        unsigned int epoch = 0;                           // grid-barrier epochs this CTA has arrived at
        auto arrive = [&] {
            pro_sync();                                   // this CTA's writes of the step are done
            if (ptid == 0) grid_arrive(p.ws.gbar);
            ++epoch;
        };
        auto wait_all = [&] {
            if (ptid == 0 && *s_fail == 0 && !grid_wait(p.ws.gbar, epoch * gridDim.x)) {
                set_status(st, DSPARK_ERR_TIMEOUT, 13);
                *s_fail = 1;
            }
            pro_sync();
        };
        // the published winner of request b at position k: its token
        auto winner = [&](int b, int k) -> int {
            const unsigned long long w = __ldcg(p.ws.words + static_cast<size_t>(k - 1) * p.B + b);
            const uint32_t idx = unpack_idx(w);
            if (w == 0ull || idx >= static_cast<uint32_t>(p.V)) {
                set_status(st, DSPARK_ERR_DEVICE_CHECK, 3);
                return 0;
            }
            return static_cast<int>(idx);
        };
        // per-thread pipeline state that continues across positions
        int mma_stage = 0;
        uint32_t mma_phase = 0;
        bool failed = false;

        // The position loop, compiled once per register budget: warps 1-3 (kRole 0: the
        // prologue share and the MMA issuer) and the epilogue warpgroups (kRole 1: the
        // prologue share, the draws and the publish) meet at the same barriers.
        auto positions = [&](auto role) {
            constexpr int kRole = decltype(role)::value;
            for (int k = k0; k <= k1; ++k) {
                const int base = (k - k0) * ntiles;           // running index of this position's first tile
                // ---------------------------------------------- prologue: x_{k-1}
                if (kMode == kDraft && multi && k > k0) {
                    wait_all();                               // every CTA published position k-1
                    for (int rr = ptid; rr < nrows; rr += kPro) {
                        const int b = req(rr);
                        const int tok = (*s_fail == 0) ? winner(b, k - 1) : 0;
                        s_prev[rr] = tok;
                        if (pc == 0) p.x[b * p.gamma + k - 2] = tok;
                    }
                } else {
                    for (int rr = ptid; rr < nrows; rr += kPro) {
                        const int b = req(rr);
                        const int kb = row_k(b, k);
                        s_prev[rr] = (kb > 0) ? prev_token(p.x0, p.x, b, p.gamma, kb, p.V, st) : -1;
                    }
                }
                pro_sync();
                failed = failed || (*s_fail != 0);

                // A operand: rows W1[x_{k_b-1}] of this M-tile, K-major, 128-byte swizzle
                {
                    // one warp per A row, one lane per 16-byte chunk (r / 8 <= 32 chunks)
                    const int cpr = p.r / 8;
                    for (int row = ptid >> 5; row < kBM; row += kPro / 32) {
                        const int rr = row & (rpc - 1);       // rpc is 32, 64 or 128
                        const int prev = (rr < nrows) ? s_prev[rr] : -1;
                        if (lane < cpr) {
                            const int slab = lane >> 3, c = lane & 7;
                            uint8_t* dst = sA + slab * kASlabBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
                            if (prev >= 0) {
                                const uint16_t* src = p.E ? p.E + (static_cast<size_t>(req(rr)) * p.gamma + (row_k(req(rr), k) - 1)) * p.r
                                                          : p.W1 + static_cast<size_t>(prev) * p.r;
                                cp_async16(dst, src + lane * 8);
                            }
                            else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    cp_async_wait_all();
                    fence_proxy_async_smem();
                    tc::fence_before_sync();
                    pro_sync();
                    tc::fence_after_sync();
                }

                if (kRole == 0 && warp == 1) {
                    // -------------------------------------------------- MMA issuer
                    if (lane == 0) {
                        constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
                        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
                        for (int i = 0; i < ntiles && !failed; ++i) {
                            // the position's tile i, the launch's tile gi, goes to accumulator
                            // gi mod kTmemBufs and is reduced by warpgroup i mod kEpiWG (the same
                            // warpgroup whichever launch runs the position, so that every path
                            // sums in the same order)
                            const int gi = base + i;
                            const int buf = gi % kTmemBufs;
                            const uint32_t par = static_cast<uint32_t>(gi / kTmemBufs) & 1u;
                            if (!mbar_wait(&tempty[buf], par ^ 1u)) { failed = true; break; }
                            tc::fence_after_sync();
                            const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kBN);
                            for (int s = 0; s < nslab; ++s) {
                                if (!mbar_wait(&full[mma_stage], mma_phase)) { failed = true; break; }
                                tc::fence_after_sync();
#pragma unroll
                                for (int kk = 0; kk < kBK / 16; ++kk) {
                                    const uint64_t ad = tc::smem_desc_sw128(a0 + s * kASlabBytes + kk * 32);
                                    const uint64_t bd = tc::smem_desc_sw128(b0 + mma_stage * kSlabBytes + kk * 32);
                                    tc::mma_bf16(d, ad, bd, idesc, (s | kk) != 0);
                                }
                                tc::commit(&empty[mma_stage]);
                                if (++mma_stage == kStages) { mma_stage = 0; mma_phase ^= 1u; }
                            }
                            tc::commit(&tfull[buf]);
                        }
                        if (failed) set_status(st, DSPARK_ERR_TIMEOUT, 11);
                    }
                    __syncwarp();
                } else if (kRole == 1) {
                    // ---------------------------------------------------- epilogue
                    const int eg = (warp - 4) >> 2;           // warpgroup 0..kEpiWG-1
                    const int q = warp & 3;                   // TMEM lane quarter
                    const int lrow = q * 32 + lane;           // TMEM lane = A row
                    const int copy = lrow / rpc;              // which copy of the request rows
                    const int rr = lrow % rpc;                // request row within the M-tile
                    const int b = (rr < nrows) ? req(rr) : 0;
                    const int kb = (rr < nrows) ? row_k(b, k) : 0;
                    const bool valid = rr < nrows && kb > 0;
                    const bool warp_live = ((q * 32) % rpc) < nrows;
                    // U rows with the normal policy for the draft (a thread reads the two halves of
                    // each 128-byte line one sub-block apart), evict-first for the residual
                    const uint64_t pol = (kMode == kDraft) ? policy_evict_normal() : policy_evict_first();
                    const uint16_t* urow = p.U + (static_cast<size_t>(valid ? b : 0) * p.gamma + (valid ? kb - 1 : 0)) * p.V;
                    [[maybe_unused]] float ld2 = 0.f, lt2 = 0.f;   // kResidual
                    [[maybe_unused]] const uint16_t* trow = nullptr;
                    if constexpr (kMode == kResidual) {
                        if (valid) {
                            ld2 = p.ld2[b];
                            lt2 = p.lt2[b];
                            trow = p.T + (static_cast<size_t>(b) * (p.gamma + 1) + (kb - 1)) * p.V;
                        }
                    }
                    const PhiloxRow prow =
                        philox_row_setup(p.seed, static_cast<uint32_t>(kb), static_cast<uint32_t>(b),
                                         (kMode == kDraft) ? kStreamDraftToken : kStreamVerifyToken);
                    Best best{-INFINITY, 0x7FFFFFFF, 0.f};
                    float M = -INFINITY, S = 0.f;
                    float qb = 0.f, Eq = 1.f;                 // kResidual: the running winner's q and E
                    const int i0 = eg;                        // this WG's tiles: eg, eg + kEpiWG, ...

                    // The thread's sub-blocks of 32 tokens: four per tile (two or one per tile and
                    // copy when each request is held twice or four times).  One compact loop body
                    // serves them all; the U words of the next sub-block (this tile's next, or the
                    // next tile's first) are loaded one sub-block ahead, so the load has a
                    // sub-block's work to land.
                    const int nsub = kBN / 32 / R;            // this copy's share of a tile: kBN / R tokens
                    const int soff = copy * (kBN / R);        // token offset of the first sub-block in a tile
                    auto load16 = [&](const uint16_t* src, int v0, uint32_t* dst) {
#pragma unroll
                        for (int g8 = 0; g8 < 4; ++g8) {
                            if (valid && v0 + g8 * 8 < p.V) ld_u32x4(src + v0 + g8 * 8, dst + g8 * 4, pol);
                            else { dst[g8 * 4] = dst[g8 * 4 + 1] = dst[g8 * 4 + 2] = dst[g8 * 4 + 3] = 0u; }
                        }
                    };
                    uint32_t un[16];                          // U words of the next sub-block (kDraft)
                    if (kMode == kDraft && i0 < ntiles) load16(urow, (t_lo + i0) * kBN + soff, un);
                    for (int i = i0; i < ntiles; i += kEpiWG) {
                        const int t = t_lo + i;
                        const int buf = (base + i) % kTmemBufs;
                        const uint32_t par = static_cast<uint32_t>((base + i) / kTmemBufs) & 1u;
                        bool bad = false;
                        if (!failed) bad = !mbar_wait(&tfull[buf], par);
                        // warp-uniform: the draw's warp votes need every lane on the same path
                        bad = __any_sync(0xffffffffu, bad);
                        if (bad) { failed = true; set_status(st, DSPARK_ERR_TIMEOUT, 12); }
                        tc::fence_after_sync();
                        const bool have_next = (i + kEpiWG < ntiles);
                        const int tnext = t + kEpiWG;
#pragma unroll 1
                        for (int j = 0; j < nsub; ++j) {
                            const int off = soff + 32 * j;
                            const int v0 = t * kBN + off;
                            // the next sub-block's U (this tile's next, or the next tile's first)
                            const int vn = (j + 1 < nsub) ? v0 + 32 : (have_next ? tnext * kBN + soff : -1);
                            if (!warp_live || failed || v0 >= p.V) {  // warp-uniform
                                if (kMode == kDraft && vn >= 0) load16(urow, vn, un);
                                continue;
                            }
                            [[maybe_unused]] uint32_t tt[16];   // kResidual: t words
                            if constexpr (kMode == kResidual) {
                                load16(urow, v0, un);
                                load16(trow, v0, tt);
                            }
                            float y[32];
                            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + off;
                            tc::tmem_ld32(taddr, y);
                            tc::tmem_ld_wait();
                            // raw logits z = acc + U (each bf16 U added to its float32 accumulator by one
                            // mixed-precision add); the draw scales by cscale
#pragma unroll
                            for (int w = 0; w < 16; ++w) add_bf16_pair(un[w], y[2 * w], y[2 * w + 1]);
                            // this sub-block's U words are consumed: fetch the next one's, in flight
                            // while this sub-block is reduced
                            if (kMode == kDraft && vn >= 0) load16(urow, vn, un);
                            if (v0 + 32 > p.V) {
#pragma unroll
                                for (int w = 0; w < 32; ++w)
                                    if (v0 + w >= p.V) y[w] = -INFINITY;
                            }
                            if constexpr (kMode == kDraft) {
                                if (p.debug_z != nullptr) {
                                    if (valid)                // copies own disjoint halves
                                        for (int w = 0; w < 32; ++w)
                                            if (v0 + w < p.V) p.debug_z[static_cast<size_t>(b) * p.V + v0 + w] = y[w] * p.cscale;
                                    continue;
                                }
                                if (p.greedy) {                // cscale = 1
#pragma unroll
                                    for (int w = 0; w < 32; ++w)
                                        if (y[w] > best.key) { best.key = y[w]; best.idx = v0 + w; }
                                } else {
                                    draw32(y, p.cscale, v0, prow, p.keys, best, M, S);
                                }
                            } else {
                                // residual q = max(0, p_t - p_d), p_d = 2^(y - ld2), p_t = 2^(t c - lt2);
                                // the winner maximises q_v / E_v over the thread's tokens
                                const uint32_t qbase = static_cast<uint32_t>(v0) >> 2;
#pragma unroll
                                for (int qq = 0; qq < 8; ++qq) {
                                    const U4 pw = philox_row(prow, qbase + qq, p.keys);
                                    const uint32_t wv[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                                    for (int jj = 0; jj < 4; ++jj) {
                                        const int w = 4 * qq + jj;
                                        const float tv = (w & 1) ? bf16hi(tt[w >> 1]) : bf16lo(tt[w >> 1]);
                                        const float pd = fast_exp2(fmaf(y[w], p.cscale, -ld2));
                                        const float ptv = fast_exp2(tv * p.cscale - lt2);
                                        const float qv = (v0 + w < p.V) ? fmaxf(ptv - pd, 0.f) : 0.f;
                                        const float E = exp_draw(wv[jj]);
                                        if (qv * Eq > qb * E) { qb = qv; Eq = E; best.idx = v0 + w; }
                                    }
                                }
                            }
                        }
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[buf]);
                    }
                    if (kMode == kResidual && qb > 0.f) best.key = fast_log2(qb) - fast_log2(Eq);
                    // the next position's first U tile of this lane does not depend on x_k:
                    // bring it into L2 while the grid hands over
                    if (kMode == kDraft && k < k1 && valid && warp_live) {
                        const int inext = eg;                 // its first tile of the next position
                        if (inext < ntiles) {
                            const uint16_t* unx = p.U + (static_cast<size_t>(b) * p.gamma + k) * p.V;
                            for (int off = soff; off < soff + 32 * nsub; off += 64) {
                                const int v0 = (t_lo + inext) * kBN + off;
                                if (v0 < p.V) prefetch_l2(unx + v0);
                            }
                        }
                    }
                    rowres[eg * kBM + lrow] = RowRes{best, M, S};
                }
                pro_sync();

                // --------------------------------------- publish this position
                if (kRole == 1 && warp < 8 && p.debug_z == nullptr) {
                    const int rr = (warp - 4) * 32 + lane;
                    const int b = (rr < nrows) ? req(rr) : 0;
                    if (rr < nrows && row_k(b, k) > 0) {
                        Best b0{-INFINITY, 0x7FFFFFFF, 0.f};
                        float m = -INFINITY, s = 0.f;
                        for (int e = 0; e < kEpiWG; ++e)
                            for (int c = 0; c < R; ++c) {
                                const RowRes r1 = rowres[e * kBM + c * rpc + rr];
                                best_take(b0, r1.best.key, r1.best.idx, r1.best.y);
                                lse_merge(m, s, r1.m, r1.s);
                            }
                        const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
                        if (kMode == kDraft && !p.greedy) {
                            p.ws.part[slot * kMaxChunks + pc] = make_float2(m, s);
                            p.ws.ybest[slot * kMaxChunks + pc] = b0.y;
                        }
                        if (b0.key > -INFINITY) atomicMax(&p.ws.words[slot], pack_key(b0.key, static_cast<uint32_t>(b0.idx)));
                        // the next A row is one of the CTAs' best tokens; bring ours into L2
                        if (kMode == kDraft && k < k1 && b0.idx >= 0 && b0.idx < p.V)
                            for (int off = 0; off < p.r * 2; off += 128)
                                prefetch_l2(reinterpret_cast<const uint8_t*>(p.W1) + static_cast<size_t>(b0.idx) * p.r * 2 + off);
                    }
                }
                if (kMode == kDraft && multi && k < k1) arrive();
                else pro_sync();                              // rowres is rewritten by the next position
            }

        };
        if (warp < 4) {
            // warpgroup 0 (producer, MMA issuer, two helpers) hands registers to the epilogue
            reg_dealloc<kCtlRegs>();
            if (warp == 0) {
                // ---------------------------------------------------- TMA producer
                // streams W2 for every position without waiting for the prologues
                if (lane == 0) {
                    const uint64_t pol = policy_evict_last();
                    int stage = 0;
                    uint32_t phase = 0;
                    bool failed = false;
                    for (int k = k0; k <= k1 && !failed; ++k)
                        for (int t = t_lo; t < t_hi && !failed; ++t)
                            for (int s = 0; s < nslab; ++s) {
                                if (!mbar_wait(&empty[stage], phase ^ 1u)) { failed = true; break; }
                                mbar_arrive_expect_tx(&full[stage], kSlabBytes);
                                tc::tma_load_2d(sB + stage * kSlabBytes, &tmW2, s * kBK, t * kBN, &full[stage], pol);
                                if (++stage == kStages) { stage = 0; phase ^= 1u; }
                            }
                    if (failed) set_status(st, DSPARK_ERR_TIMEOUT, 10);
                }
                __syncwarp();
            } else {
                positions(RoleTag<0>{});
            }
            reg_alloc<kLaunchRegs>();
        } else {
            reg_alloc<kEpiRegs>();
            positions(RoleTag<1>{});
            reg_dealloc<kLaunchRegs>();
        }
        if (warp != 0) {
            if (kMode == kResidual && p.fuse_tail) {
                // ------------------------------------------------ final tokens
                arrive();
                wait_all();                                   // every CTA published its residual winners
                if (warp >= 2 && *s_fail == 0) {
                    const int pair = (warp - 2) >> 1;
                    for (int b = blockIdx.x + pair * gridDim.x; b < p.B; b += kPairs * gridDim.x)
                        finish_pair<true>(p.fin, b, p.gamma, p.V, p.cscale, p.seed, st, 2 + pair, xch + 2 * pair,
                                          xchi + 2 * pair);
                }
            }
            if (kMode == kDraft && p.fuse_tail && p.debug_z == nullptr) {
                // ------------------------------------------ x_gamma and finalize
                const int cta = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);
                const int nown = (cta < p.B) ? (p.B - 1 - cta) / ncta + 1 : 0;
                arrive();
                wait_all();                                   // every CTA published the last position
                for (int j = ptid; j < nown; j += kPro) {
                    const int b = cta + j * ncta;
                    p.x[b * p.gamma + k1 - 1] = (*s_fail == 0) ? winner(b, k1) : 0;
                }
                pro_sync();
                // one warp per (owned request, position)
                for (int item = warp - 1; item < nown * p.gamma; item += kPro / 32) {
                    const int b = cta + (item / p.gamma) * ncta, k = item % p.gamma + 1;
                    finalize_position<true>(b, k, p.B, p.gamma, p.V, p.H, p.r, p.h, p.W1, p.w, p.bias, p.x0, p.x,
                                            p.greedy, P, kBN, NT, p.ws.part, p.ws.ybest, p.lse_d, p.logp_d, p.c, st);
                }
                pro_sync();
                for (int j = ptid; j < nown; j += kPro) {     // survival a_k = prod c_1..c_k, in k order
                    const int b = cta + j * ncta;
                    float surv = 1.f;
                    for (int kk = 0; kk < p.gamma; ++kk) {
                        const size_t o = static_cast<size_t>(b) * p.gamma + kk;
                        surv = surv * p.c[o];
                        p.a[o] = surv;
                    }
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, 512);
    }
}

constexpr size_t kTcSmem = 1024 + 4 * kASlabBytes + kStages * kSlabBytes + (2 * kStages + 2 * kTmemBufs) * 8 + 16 +
                           kEpiWG * kBM * sizeof(RowRes) + kBM * 4 + 2 * kPairs * 4 + 2 * kPairs * 4 + 16;

// ------------------------------------------------------------ host side ---
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D map over W2 [V][r] bf16: box {64, 128}, 128-byte swizzle, zero fill.
inline bool encode_w2_map(CUtensorMap* map, const void* W2, int V, int r) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(V)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(r) * 2};
    const cuuint32_t box[2] = {kBK, kBN};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool use_tc_path(dspark_dtype_t dt, int r) { return dt == DSPARK_BF16 && r % kBK == 0 && r <= 256; }

template <int kMode>
dspark_status_t launch_tc(const CUtensorMap& map, const TcParams& p, int grid, cudaStream_t s, bool cooperative) {
    static OncePerDevice once;
    if (once.run(current_device(), [] {
            // the kernel's register split (setmaxnreg) assumes kLaunchRegs a thread at launch:
            // never launch a build that allocated another count
            cudaFuncAttributes fa{};
            cudaError_t e = cudaFuncGetAttributes(&fa, bias_engine_tc<kMode>);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidDeviceFunction;
            return cudaFuncSetAttribute(bias_engine_tc<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kTcSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cooperative) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    if (l2_window(&attr[na], p.W2, static_cast<size_t>(p.V) * p.r * 2)) ++na;   // W2 kept in L2 (opt-in)
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, bias_engine_tc<kMode>, map, p) != cudaSuccess) {
        cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}

// Grid of the tcgen05 engine: nM M-tiles, P CTAs each (P * nM <= SMs).
inline void tc_grid(int B, int V, int* nM, int* P) {
    *nM = (B + kBM - 1) / kBM;
    const int sms = sm_count(current_device());
    int per = sms / *nM;
    if (per < 1) per = 1;
    const int NT = (V + kBN - 1) / kBN;
    if (per > NT) per = NT;
    if (per > kMaxChunks) per = kMaxChunks;
    *P = per;
}

}  // namespace eng
}  // namespace dspark
