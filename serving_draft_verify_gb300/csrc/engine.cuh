// The bias engine shared by dspark_draft_block and dspark_verify: for a set of
// request rows, each with a position k_b, it forms the draft logits
//   z_b = U[b][k_b-1] + W2 . W1[x_{k_b-1}]       (VanillaMarkovHead, eq. 5;
//                                                 DeepSpec walkthrough 3.2)
// tile by tile on the tensor cores and reduces them in its epilogue:
//   kDraft     per 64-token block: logsumexp of z / T and a Gumbel block key
//              (draft sampling), or the running argmax of z (greedy);
//   kResidual  per 64-token block: the mass of max(0, p_t - p_d) and a Gumbel
//              block key (the residual draw of verification, section 8.2).
// Each CTA publishes its best block per row with a 64-bit atomicMax of
// (key, ~block) and, for kDraft, its (max, sum) partial.
//
// Layout of one CTA (384 threads, one CTA per SM):
//   warp 0      TMA producer: W2 tiles [128 tokens x 64 K] into a slab ring
//               (128-byte swizzle, L2 evict-last so W2 stays resident);
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//               M = 128 request rows, N = 128 tokens, K = r, fp32 in TMEM;
//   warps 4-11  two epilogue warpgroups, each with two TMEM accumulators, so
//               the MMA of the next tile overlaps the epilogue of this one.
// The A operand (rows W1[x_{k_b-1}], or the rows E[b][k_b] of a gated or
// recurrent head, gathered into shared memory with the same swizzle) is built
// by warps 1-11 at the start of every position.
//
// Draft launches may cover positions k .. k_last (a cooperative launch, all
// CTAs resident, TMEM and barriers set up once, the producer streaming W2
// straight through all positions).  Between positions the grid meets at a
// bounded counter barrier; then CTA c draws x_{k} for requests b = c (mod
// grid) from the published block winners (pairs of warps rebuild z on the
// winning block from W2 rows), and the grid meets again before x_{k} is read.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "tc.cuh"

namespace dspark {
namespace eng {

constexpr int kMaxChunks = 256;   // partial slots per (position, request)

struct Ws {
    StatusBlock* status;
    unsigned long long* words;   // [positions][B] best (key, ~block) or (value, ~token)
    float2* part;                // [positions][B][kMaxChunks] (max, sum) of y = z log2e / T
    float* ytok;                 // [positions][B] y of the drawn token
    unsigned int* gbar;          // grid-barrier counter of the multi-position draft launch (starts at 0)
    unsigned long long* xw;      // [B] (k << 32) | x_k, the last token drawn in the running launch (starts at 0)
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

// After v[i] (i < 32) is given in every lane, lane l ends with sum over lanes of
// v[l] in v[0] (a butterfly that halves the live values at every stage).
__device__ __forceinline__ void transpose_reduce32(float* v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
}

// N (8, 16 or 32) partial sums v[0..N) per lane, summed over the 32 lanes: lane
// l ends with the total of v[l % N] in v[0].  Lanes pair by the same bits, in
// the same order (16, 8, 4, 2, 1), as in transpose_reduce32, so the totals are
// bit-identical to it; levels above N/2 add without halving.
template <int N>
__device__ __forceinline__ void tree_reduce(float* v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= N; s >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], s);
    }
#pragma unroll
    for (int s = N / 2; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
}

// Two warps per request: z for the 64 tokens of block `blk` of row (b, k):
// warp w rebuilds tokens blk*64 + 32w + (0..31); each lane loads one or two
// 16-byte chunks of every W2 row (coalesced rows) and a transpose-reduce
// leaves token (32w + lane)'s dot product in that lane.  Returns z for the
// lane's token (-inf past V).  erow: the rank-r row behind the bias of (b, k)
// (bias_row).
template <bool kBF16, int kCPL>
__device__ __forceinline__ float block_logit_prev(int b, int gamma, int k, int V, int r, int blk, const void* erow,
                                                  const void* U, const void* W2) {
    constexpr int EPC = kBF16 ? 8 : 4;                    // elements per 16-byte chunk
    const int warp = (threadIdx.x >> 5) & 1, lane = threadIdx.x & 31;
    const int nch = r / EPC;
    const int vbase = blk * 64 + warp * 32;
    const int vl = vbase + lane;
    const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
    const float u = (vl < V) ? ld_elem<kBF16>(U, urow + vl) : 0.f;
    float e[kCPL][EPC];
#pragma unroll
    for (int cc = 0; cc < kCPL; ++cc) {
        const int c = lane + 32 * cc;
#pragma unroll
        for (int q = 0; q < EPC; ++q)
            e[cc][q] = (c < nch) ? ld_elem<kBF16>(erow, static_cast<size_t>(c) * EPC + q) : 0.f;
    }
    const uint64_t pol = policy_evict_last();
    float part[32];
    constexpr int kBatch = 32 / kCPL;
#pragma unroll
    for (int i0 = 0; i0 < 32; i0 += kBatch) {
        uint4 raw[kBatch][kCPL];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int v = vbase + i0 + i;
#pragma unroll
            for (int cc = 0; cc < kCPL; ++cc) {
                const int c = lane + 32 * cc;
                raw[i][cc] = make_uint4(0, 0, 0, 0);
                if (v < V && c < nch)
                    ld_u32x4(static_cast<const uint8_t*>(W2) + (static_cast<size_t>(v) * r + c * EPC) * (kBF16 ? 2 : 4),
                             &raw[i][cc].x, pol);
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int cc = 0; cc < kCPL; ++cc) {
                const uint32_t wv[4] = {raw[i][cc].x, raw[i][cc].y, raw[i][cc].z, raw[i][cc].w};
                if constexpr (kBF16) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc = fmaf(bf16lo(wv[q]), e[cc][2 * q], acc);
                        acc = fmaf(bf16hi(wv[q]), e[cc][2 * q + 1], acc);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc = fmaf(__uint_as_float(wv[q]), e[cc][q], acc);
                }
            }
            part[i0 + i] = acc;
        }
    }
    transpose_reduce32(part);
    if (vl >= V) return -INFINITY;
    return part[0] + u;
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

template <bool kBF16, int kCPL>
__device__ __forceinline__ float block_logit(int b, int gamma, int k, int V, int r, int blk, const void* U,
                                             const void* W1, const void* E, const void* W2, const int32_t* x0,
                                             const int32_t* x, StatusBlock* st) {
    const int prev = prev_token(x0, x, b, gamma, k, V, st);
    return block_logit_prev<kBF16, kCPL>(b, gamma, k, V, r, blk, bias_row<kBF16>(E, W1, b, gamma, k, r, prev), U,
                                         W2);
}

// ===================================================== tcgen05 engine ====
constexpr int kBM = 128;              // request rows per M-tile (TMEM lanes)
constexpr int kBN = 128;              // vocabulary columns per tile
constexpr int kBK = 64;               // K per smem slab (128 bytes of bf16)
constexpr int kStages = 8;            // W2 slab ring
constexpr int kEpiWG = 2;             // epilogue warpgroups, two TMEM buffers each
constexpr int kTcThreads = 128 * (1 + kEpiWG);
constexpr int kSlabBytes = kBN * kBK * 2;     // 16 KB
constexpr int kASlabBytes = kBM * kBK * 2;    // 16 KB

enum Mode : int { kDraft = 0, kResidual = 1 };

// What the final token draw of verification reads and writes (section 8.2:
// the residual draw after a rejection, or a draw from p_t at the stop row).
struct FinishArgs {
    const uint16_t* T;               // t_logits [B][gamma+1][V]
    const int32_t* krow;             // [B] rejected position (0: none)
    const int32_t* stop;             // [B] row of the final draw
    const float* lt2;                // [B]
    const float* ld2;                // [B]
    const unsigned long long* res_word;   // [B] residual block winner
    const unsigned long long* wt;    // [B][gamma+1] target-row block winner
    int32_t* next_token;             // [B]
};

struct TcParams {
    int B, gamma, V, r, k;           // k: the position of every row (kDraft)
    const uint16_t* U;               // [B][gamma][V]
    const uint16_t* W1;              // [V][r]
    const uint16_t* E;               // [B][gamma][r] bias rows of a gated / recurrent head, or null (W1[x_{k-1}])
    const uint16_t* W2;              // [V][r] (the redraw of the winning block reads rows directly)
    const int32_t* x0;               // [B]
    int32_t* x;                      // [B][gamma]; kDraft writes x_{k-1} here (CTA 0 of each M-tile)
    float cscale;                    // log2e / T (1 for greedy)
    int greedy;
    uint64_t seed;
    int P;                           // CTAs per M-tile
    Ws ws;
    float* debug_z;                  // kDraft: write y to [B][V] instead of reducing
    int k_last;                      // kDraft: positions k .. k_last in one (cooperative) launch
    // kDraft with fuse_tail: the launch also draws x_gamma and finalizes
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
    // kResidual with fuse_tail: the launch also draws the final token
    FinishArgs fin;
    // kResidual
    const int32_t* krow;             // [B] rejected position k_b (0: row inactive)
    const uint16_t* T;               // t_logits [B][gamma+1][V]
    const float* lt2;                // [B] log2-sum-exp2 of t / T at row k_b (log2 units)
    const float* ld2;                // [B] lse_d[b][k_b-1] * log2e
};

struct RowRes {
    float key;
    int idx;
    float m, s;
};
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

// Waits (bounded) until the tagged token word of a request carries position k.
__device__ __forceinline__ bool wait_token(const unsigned long long* xw, int k, int* tok) {
    auto load = [&]() {
        unsigned long long v;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(xw) : "memory");
        return v;
    };
    unsigned long long v = load();
    if (static_cast<uint32_t>(v >> 32) != static_cast<uint32_t>(k)) {
        const uint64_t t0 = globaltimer_ns();
        while (static_cast<uint32_t>((v = load()) >> 32) != static_cast<uint32_t>(k)) {
            __nanosleep(32);
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    *tok = static_cast<int>(static_cast<uint32_t>(v));
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
// partials, logp_d = y(x_k) - lse_d, and the confidence
// c = sigmoid(w . [h_k ; W1[x_{k-1}]] + bias), written by lane 0.
template <bool kBF16>
__device__ __forceinline__ void finalize_position(int b, int k, int B, int gamma, int V, int H, int r, const void* h,
                                                  const void* W1, const void* w, float bias, const int32_t* x0,
                                                  const int32_t* x, int greedy, int nchunk, const float2* part,
                                                  const float* ytok, float* lse_d, float* logp_d, float* c,
                                                  StatusBlock* st) {
    const int lane = threadIdx.x & 31;
    const size_t slot = static_cast<size_t>(k - 1) * B + b;
    const size_t o = static_cast<size_t>(b) * gamma + (k - 1);
    float L = 0.f, lp = 0.f;
    if (!greedy) {
        float m = -INFINITY, s = 0.f;
        float2 pr[kMaxChunks / 32];                       // every partial of this lane in flight at once
#pragma unroll
        for (int u = 0; u < kMaxChunks / 32; ++u) {
            const int ch = lane + 32 * u;
            pr[u] = (ch < nchunk) ? __ldcg(part + slot * kMaxChunks + ch) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMaxChunks / 32; ++u)
            if (lane + 32 * u < nchunk) lse_merge(m, s, pr[u].x, pr[u].y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, off);
            const float os = __shfl_xor_sync(0xffffffffu, s, off);
            lse_merge(m, s, om, os);
        }
        const float L2 = m + log2f(s);
        L = L2 * kLn2;
        lp = (__ldcg(ytok + slot) - L2) * kLn2;
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
// 2-entry exchange): if a draft token was rejected at k and the residual
// max(0, p_t - p_d) has mass, the token inside the residual's winning block
// (second Gumbel level, stream 2); otherwise a draw from p_t at the stop row
// (bonus row, stream 5) inside that row's winning block.
template <bool kBF16, int kCPL>
__device__ __forceinline__ void finish_pair(const FinishArgs& f, int b, int gamma, int V, int r, const void* U,
                                            const void* W1, const void* E, const void* W2, const int32_t* x0,
                                            const int32_t* x,
                                            float cscale, uint64_t seed, StatusBlock* st, int bar, float* xch,
                                            int* xchi) {
    const int lane = threadIdx.x & 31, wp = (threadIdx.x >> 5) & 1;
    const int kr = f.krow[b];
    const unsigned long long rw = (kr > 0) ? __ldcg(f.res_word + b) : 0ull;
    const uint32_t nblk = static_cast<uint32_t>((V + 63) / 64);
    bool residual = rw != 0ull && unpack_idx(rw) < nblk;
    float score = -INFINITY;
    int v = 0x7FFFFFFF;
    if (residual) {
        const int blk = static_cast<int>(unpack_idx(rw));
        const float z = block_logit<kBF16, kCPL>(b, gamma, kr, V, r, blk, U, W1, E, W2, x0, x, st);
        v = blk * 64 + wp * 32 + lane;
        if (z > -INFINITY) {
            const float yd = z * cscale;
            const float yt = ld_elem<kBF16>(f.T, (static_cast<size_t>(b) * (gamma + 1) + (kr - 1)) * V + v) * cscale;
            const float qv = fast_exp2(yt - f.lt2[b]) - fast_exp2(yd - f.ld2[b]);
            if (qv > 0.f) {
                const float g =
                    gumbel_of(uniform_open(draw_word(seed, b, kr, kStreamResidualToken, static_cast<uint32_t>(v))));
                score = log2f(qv) * kLn2 + g;
            }
        }
        if (!pair_any(score > -INFINITY, bar)) residual = false;   // no mass left after rounding
    }
    bool bad = false;
    if (!residual) {
        const int srow = (kr > 0) ? kr : f.stop[b];
        const unsigned long long w = __ldcg(f.wt + static_cast<size_t>(b) * (gamma + 1) + srow - 1);
        if (w == 0ull || unpack_idx(w) >= nblk) {
            if (threadIdx.x % 64 == 0) set_status(st, DSPARK_ERR_DEVICE_CHECK, w == 0ull ? 7 : 9);
            bad = true;
        } else {
            const int blk = static_cast<int>(unpack_idx(w));
            v = blk * 64 + wp * 32 + lane;
            score = -INFINITY;
            if (v < V) {
                const float yt = ld_elem<kBF16>(f.T, (static_cast<size_t>(b) * (gamma + 1) + (srow - 1)) * V + v) * cscale;
                const float g =
                    gumbel_of(uniform_open(draw_word(seed, b, srow, kStreamTargetToken, static_cast<uint32_t>(v))));
                score = yt + g * kLog2e;
            }
        }
    }
    int bi = (score > -INFINITY) ? v : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, score, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (os > score || (os == score && oi < bi)) { score = os; bi = oi; }
    }
    if (lane == 0) { xch[wp] = score; xchi[wp] = bi; }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
    if (wp == 0 && lane == 0) {
        int w = 0;
        if (xch[1] > xch[0] || (xch[1] == xch[0] && xchi[1] < xchi[0])) w = 1;
        f.next_token[b] = (bad || xchi[w] == 0x7FFFFFFF) ? 0 : xchi[w];
    }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
}

// Draw x_k for request b with a group of G = 4 or 8 warps (group warp gw,
// named barrier `bar` over 32 G threads).  Each warp rebuilds z on 64 / G
// tokens of the winning block: lane c multiplies the c-th 16-byte chunk of
// each W2 row by the same chunk of e = W1[x_{k-1}], kept in shared memory
// (e_s, float[r]) since this CTA drew x_{k-1}; a butterfly over the lanes sums
// the chunks (the same order as the two-warp draw, so z is bit-identical).
// The second Gumbel level (stream 0) picks the token; the group leader
// publishes it ((k << 32) | x_k word, x, ytok) and the group refills e_s with
// W1[x_k] for the next draw.  g: [3 G] words of exchange space.
template <int G>
__device__ __forceinline__ void group_draw(const TcParams& p, int b, int k, int gw, int bar, float* e_s, float* g) {
    constexpr int NT = 64 / G;                            // tokens per warp
    const int lane = threadIdx.x & 31;
    float* gsc = g;
    float* gy = g + G;
    int* gix = reinterpret_cast<int*>(g + 2 * G);
    const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
    const unsigned long long word = __ldcg(p.ws.words + slot);
    const uint32_t idx = unpack_idx(word);
    const bool ok = word != 0ull && idx < static_cast<uint32_t>((p.V + 63) / 64);
    float score = -INFINITY, yv = 0.f;
    int bi = 0x7FFFFFFF;
    if (ok) {
        const int vbase = static_cast<int>(idx) * 64 + gw * NT;
        const int vl = vbase + (lane & (NT - 1));
        const int nch = p.r / 8;
        const float u = (lane < NT && vl < p.V)
                            ? bf16lo(p.U[(static_cast<size_t>(b) * p.gamma + (k - 1)) * p.V + vl])
                            : 0.f;
        const uint64_t pol = policy_evict_last();
        uint4 raw[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            raw[t] = make_uint4(0, 0, 0, 0);
            if (vbase + t < p.V && lane < nch)
                ld_u32x4(p.W2 + static_cast<size_t>(vbase + t) * p.r + lane * 8, &raw[t].x, pol);
        }
        float e[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) e[q] = (lane < nch) ? e_s[lane * 8 + q] : 0.f;
        float part[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint32_t wv[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(bf16lo(wv[q]), e[2 * q], acc);
                acc = fmaf(bf16hi(wv[q]), e[2 * q + 1], acc);
            }
            part[t] = acc;
        }
        tree_reduce<NT>(part);
        if (lane < NT && vl < p.V) {
            yv = (part[0] + u) * p.cscale;
            const float gum = gumbel_of(uniform_open(draw_word(p.seed, b, k, kStreamDraftToken, static_cast<uint32_t>(vl))));
            score = yv + gum * kLog2e;
            bi = vl;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, score, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const float oy = __shfl_xor_sync(0xffffffffu, yv, o);
        if (os > score || (os == score && oi < bi)) { score = os; bi = oi; yv = oy; }
    }
    if (lane == 0) { gsc[gw] = score; gix[gw] = bi; gy[gw] = yv; }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * G) : "memory");
    if (gw == 0 && lane == 0) {
        int w = 0;
        for (int q = 1; q < G; ++q)
            if (gsc[q] > gsc[w] || (gsc[q] == gsc[w] && gix[q] < gix[w])) w = q;
        int tok = gix[w];
        if (tok == 0x7FFFFFFF) { set_status(p.ws.status, DSPARK_ERR_DEVICE_CHECK, 3); tok = 0; }
        const unsigned long long tagged = (static_cast<unsigned long long>(k) << 32) | static_cast<uint32_t>(tok);
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p.ws.xw + b), "l"(tagged) : "memory");
        p.x[b * p.gamma + k - 1] = tok;
        p.ws.ytok[slot] = gy[w];
        gix[0] = tok;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * G) : "memory");
    // e for the next draw: W1[x_k] (also the next position's A row, so bring it into L2 too)
    const int tok = gix[0];
    for (int j = gw * 32 + lane; j < p.r / 2; j += 32 * G) {
        const uint32_t w2 = reinterpret_cast<const uint32_t*>(p.W1 + static_cast<size_t>(tok) * p.r)[j];
        e_s[2 * j] = bf16lo(w2);
        e_s[2 * j + 1] = bf16hi(w2);
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(32 * G) : "memory");
}

// Draw x_k for request b inside a running multi-position launch: a pair of
// warps (named barrier `bar`, 64 threads) rebuilds z on the winning block from
// W2 rows and takes the second Gumbel level (stream 0); the even warp's lane 0
// writes x and ytok.  xch/xchi: this pair's 2-entry exchange slots.
__device__ __forceinline__ void pair_draw(const TcParams& p, int b, int k, int bar, float2* xch, int* xchi) {
    const int lane = threadIdx.x & 31, wp = (threadIdx.x >> 5) & 1;
    const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
    // independent L2 reads first: the winning block, and x_{k-1} for W1
    const unsigned long long word = __ldcg(p.ws.words + slot);
    const int prev = prev_token(p.x0, p.x, b, p.gamma, k, p.V, p.ws.status);
    const uint32_t idx = unpack_idx(word);
    const bool ok = word != 0ull && idx < static_cast<uint32_t>((p.V + 63) / 64);
    float score = -INFINITY, yv = 0.f;
    int bi = 0x7FFFFFFF;
    if (ok) {
        const int blk = static_cast<int>(idx);
        const float z = block_logit_prev<true, 1>(b, p.gamma, k, p.V, p.r, blk,
                                                  bias_row<true>(p.E, p.W1, b, p.gamma, k, p.r, prev), p.U, p.W2);
        const int v = blk * 64 + wp * 32 + lane;
        if (z > -INFINITY) {
            yv = z * p.cscale;
            const float g = gumbel_of(uniform_open(draw_word(p.seed, b, k, kStreamDraftToken, static_cast<uint32_t>(v))));
            score = yv + g * kLog2e;
            bi = v;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, score, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const float oy = __shfl_xor_sync(0xffffffffu, yv, o);
        if (os > score || (os == score && oi < bi)) { score = os; bi = oi; yv = oy; }
    }
    if (lane == 0) { xch[wp] = make_float2(score, yv); xchi[wp] = bi; }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
    if (wp == 0 && lane == 0) {
        int w = 0;
        if (xch[1].x > xch[0].x || (xch[1].x == xch[0].x && xchi[1] < xchi[0])) w = 1;
        int tok = xchi[w];
        if (tok == 0x7FFFFFFF) { set_status(p.ws.status, DSPARK_ERR_DEVICE_CHECK, 3); tok = 0; }
        // the tagged word carries the token itself: no ordering with other stores is needed
        const unsigned long long tagged = (static_cast<unsigned long long>(k) << 32) | static_cast<uint32_t>(tok);
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p.ws.xw + b), "l"(tagged) : "memory");
        p.x[b * p.gamma + k - 1] = tok;
        p.ws.ytok[slot] = xch[w].y;
        xchi[0] = tok;
    }
    asm volatile("bar.sync %0, 64;" ::"r"(bar) : "memory");
    // W1[x_k] is the next position's A row and the next draw's e: bring it into L2
    if (wp == 0 && lane * 128 < p.r * 2)
        prefetch_l2(reinterpret_cast<const uint8_t*>(p.W1) + static_cast<size_t>(xchi[0]) * p.r * 2 + lane * 128);
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
    uint64_t* tfull = empty + kStages;                    // [2 * kEpiWG]
    uint64_t* tempty = tfull + 2 * kEpiWG;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2 * kEpiWG);
    RowRes* rowres = reinterpret_cast<RowRes*>(tmem_slot + 4);   // [kEpiWG][128]
    int* s_prev = reinterpret_cast<int*>(rowres + kEpiWG * kBM);   // [128] x_{k-1} per request row
    float2* xch = reinterpret_cast<float2*>(s_prev + kBM);        // [10] pair exchange
    int* xchi = reinterpret_cast<int*>(xch + 10);                 // [10]
    int* s_fail = xchi + 10;
    float* e_s = reinterpret_cast<float*>(s_fail + 4);           // [2][256] W1 row of the last token drawn
    float* gx = e_s + 2 * 256;                                     // [2][3 * 8] group-draw exchange

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x / p.P, pc = blockIdx.x % p.P;
    const int m0 = g * kBM;
    const int NT = (p.V + kBN - 1) / kBN;
    const int t_lo = static_cast<int>(static_cast<long long>(pc) * NT / p.P);
    const int t_hi = static_cast<int>(static_cast<long long>(pc + 1) * NT / p.P);
    const int ntiles = t_hi - t_lo;
    StatusBlock* st = p.ws.status;
    // Row replication: with at most 64 requests the A tile holds every request
    // twice (TMEM lanes 0-63 and 64-127) and the two copies reduce different
    // 64-token blocks of each tile, so all epilogue warps have work.
    const int R = (p.B <= 64) ? 2 : 1;
    const int rpc = kBM / R;                              // request rows per copy
    const int nrows = min(rpc, p.B - m0);                 // requests of this M-tile
    const int k0 = p.k;
    const int k1 = (kMode == kDraft && p.k_last > p.k) ? p.k_last : p.k;
    const bool multi = k1 > k0;                           // positions k0..k1, grid barriers between
    auto row_k = [&](int b, int k) -> int { return (kMode == kResidual) ? p.krow[b] : k; };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int e = 0; e < 2 * kEpiWG; ++e) { mbar_init(&tfull[e], 1); mbar_init(&tempty[e], 4); }
        *s_fail = 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tmW2);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

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
        // per-thread pipeline state that continues across positions
        int mma_stage = 0;
        uint32_t mma_phase = 0;
        bool failed = false;
        // requests b = blockIdx.x + j * gridDim.x < B, j < nown, belong to this CTA: it draws their
        // tokens (with one group of 8 or two of 4 warps when it owns at most two, keeping e = W1[x]
        // in shared memory; with pairs of warps otherwise) and finalizes them
        const int cta = static_cast<int>(blockIdx.x), ncta = static_cast<int>(gridDim.x);
        const int nown = (cta < p.B) ? (p.B - 1 - cta) / ncta + 1 : 0;
        const bool grouped = kMode == kDraft && !p.greedy && nown <= 2 && (multi || p.fuse_tail);
        auto draw_owned = [&](int kd) {
            if (*s_fail != 0) return;
            if (grouped) {
                if (warp >= 4) {
                    if (nown == 1)
                        group_draw<8>(p, cta, kd, warp - 4, 2, e_s, gx);
                    else if (nown == 2)
                        group_draw<4>(p, cta + ((warp - 4) >> 2) * ncta, kd, (warp - 4) & 3, 2 + ((warp - 4) >> 2),
                                      e_s + ((warp - 4) >> 2) * 256, gx + ((warp - 4) >> 2) * 24);
                }
            } else if (warp >= 2) {
                const int pair = (warp - 2) >> 1;
                for (int b = cta + pair * ncta; b < p.B; b += 5 * ncta)
                    pair_draw(p, b, kd, 2 + pair, xch + 2 * pair, xchi + 2 * pair);
            }
        };

        for (int k = k0; k <= k1; ++k) {
            const int base = (k - k0) * ntiles;           // running index of this position's first tile
            // ---------------------------------------------- prologue: x_{k-1}
            if (kMode == kDraft && multi && k > k0) {
                wait_all();                               // every CTA published position k-1
                if (!p.greedy) {
                    // second Gumbel level for x_{k-1}, spread over the grid (owned requests)
                    draw_owned(k - 1);
                    // x_{k-1} of this M-tile's requests, as their drawers publish them
                    for (int rr = ptid; rr < nrows; rr += kPro) {
                        int tok = 0;
                        if (*s_fail == 0 && !wait_token(p.ws.xw + m0 + rr, k - 1, &tok)) {
                            set_status(st, DSPARK_ERR_TIMEOUT, 14);
                            *s_fail = 1;
                        }
                        if (tok < 0 || tok >= p.V) { set_status(st, DSPARK_ERR_DEVICE_CHECK, 2); tok = 0; }
                        s_prev[rr] = tok;
                    }
                } else {
                    for (int rr = ptid; rr < nrows; rr += kPro) {
                        const int b = m0 + rr;
                        const unsigned long long w = __ldcg(p.ws.words + static_cast<size_t>(k - 2) * p.B + b);
                        const uint32_t idx = unpack_idx(w);
                        int tok = static_cast<int>(idx);
                        if (w == 0ull || idx >= static_cast<uint32_t>(p.V)) {
                            set_status(st, DSPARK_ERR_DEVICE_CHECK, 3);
                            tok = 0;
                        }
                        s_prev[rr] = tok;
                        if (pc == 0) p.x[b * p.gamma + k - 2] = tok;
                    }
                }
            } else {
                for (int rr = ptid; rr < nrows; rr += kPro) {
                    const int b = m0 + rr;
                    const int kb = row_k(b, k);
                    s_prev[rr] = (kb > 0) ? prev_token(p.x0, p.x, b, p.gamma, kb, p.V, st) : -1;
                }
                if (grouped && warp >= 4) {                // e of the first draw: W1[x_{k0-1}]
                    for (int j = 0; j < nown; ++j) {
                        const int prev = prev_token(p.x0, p.x, cta + j * ncta, p.gamma, k, p.V, st);
                        for (int i = tid - 128; i < p.r / 2; i += kTcThreads - 128) {
                            const uint32_t w2 = reinterpret_cast<const uint32_t*>(p.W1 + static_cast<size_t>(prev) * p.r)[i];
                            e_s[j * 256 + 2 * i] = bf16lo(w2);
                            e_s[j * 256 + 2 * i + 1] = bf16hi(w2);
                        }
                    }
                }
            }
            pro_sync();
            failed = failed || (*s_fail != 0);

            // A operand: rows W1[x_{k_b-1}] of this M-tile, K-major, 128-byte swizzle
            {
                // one warp per A row, one lane per 16-byte chunk (r / 8 <= 32 chunks)
                const int cpr = p.r / 8;
                for (int row = ptid >> 5; row < kBM; row += kPro / 32) {
                    const int rr = row & (rpc - 1);       // rpc is 64 or 128
                    const int prev = (rr < nrows) ? s_prev[rr] : -1;
                    if (lane < cpr) {
                        const int slab = lane >> 3, c = lane & 7;
                        uint8_t* dst = sA + slab * kASlabBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
                        if (prev >= 0) {
                            const uint16_t* src = p.E ? p.E + (static_cast<size_t>(m0 + rr) * p.gamma + (row_k(m0 + rr, k) - 1)) * p.r
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

            if (warp == 1) {
                // -------------------------------------------------- MMA issuer
                if (lane == 0) {
                    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
                    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
                    for (int i = 0; i < ntiles && !failed; ++i) {
                        const int gi = base + i;
                        const int eg = gi % kEpiWG, use = gi / kEpiWG;
                        const int buf = eg * 2 + (use & 1);
                        const uint32_t par = static_cast<uint32_t>(use >> 1) & 1u;
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
            } else if (warp >= 4) {
                // ---------------------------------------------------- epilogue
                const int eg = (warp - 4) >> 2;           // warpgroup 0..kEpiWG-1
                const int q = warp & 3;                   // TMEM lane quarter
                const int lrow = q * 32 + lane;           // TMEM lane = A row
                const int copy = lrow / rpc;              // which copy of the request rows
                const int rr = lrow % rpc;                // request row within the M-tile
                const int b = m0 + rr;
                const int kb = (rr < nrows) ? row_k(b, k) : 0;
                const bool valid = rr < nrows && kb > 0;
                const bool warp_live = ((q * 32) % rpc) < nrows;
                // U rows stay in L2 (normal policy): the token draw after this position
                // re-reads the 64 values of each winning block
                const uint64_t pol = (kMode == kDraft) ? policy_evict_normal() : policy_evict_first();
                const uint16_t* urow = p.U + (static_cast<size_t>(valid ? b : 0) * p.gamma + (valid ? kb - 1 : 0)) * p.V;
                float ld2 = 0.f, lt2 = 0.f;
                const uint16_t* trow = nullptr;
                if constexpr (kMode == kResidual) {
                    if (valid) {
                        ld2 = p.ld2[b];
                        lt2 = p.lt2[b];
                        trow = p.T + (static_cast<size_t>(b) * (p.gamma + 1) + (kb - 1)) * p.V;
                    }
                }
                float best = -INFINITY, M = -INFINITY, S = 0.f;
                int best_i = 0x7FFFFFFF;
                const int i0 = ((eg - base) % kEpiWG + kEpiWG) % kEpiWG;   // this WG's first local tile

                uint32_t u[2][32];                        // U of the two 64-token blocks of one tile
                auto load_blk = [&](const uint16_t* src, int t, int hb, uint32_t* dst) {
                    const int v0 = t * kBN + hb * 64;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        if (valid && v0 + g8 * 8 < p.V) ld_u32x4(src + v0 + g8 * 8, dst + g8 * 4, pol);
                        else { dst[g8 * 4] = dst[g8 * 4 + 1] = dst[g8 * 4 + 2] = dst[g8 * 4 + 3] = 0u; }
                    }
                };
                auto mine = [&](int hb) -> bool { return R == 1 || hb == copy; };
                if (kMode == kDraft && i0 < ntiles && warp_live) {
                    if (mine(0)) load_blk(urow, t_lo + i0, 0, u[0]);
                    if (mine(1)) load_blk(urow, t_lo + i0, 1, u[1]);
                }
                const uint32_t stream = (kMode == kDraft) ? kStreamDraftBlock : kStreamResidualBlock;
                for (int i = i0; i < ntiles; i += kEpiWG) {
                    const int t = t_lo + i;
                    const int use = (base + i) / kEpiWG;
                    const int buf = eg * 2 + (use & 1);
                    const uint32_t par = static_cast<uint32_t>(use >> 1) & 1u;
                    bool bad = false;
                    if (!failed) bad = !mbar_wait(&tfull[buf], par);
                    if (bad) { failed = true; set_status(st, DSPARK_ERR_TIMEOUT, 12); }
                    tc::fence_after_sync();
                    const bool have_next = (i + kEpiWG < ntiles);
                    const int tnext = t + kEpiWG;
                    // the two blocks 2t and 2t+1 share one Philox counter (index >> 2)
                    U4 pw{0, 0, 0, 0};
                    if (!p.greedy && warp_live)
                        pw = philox4x32_10(U4{static_cast<uint32_t>(t >> 1), static_cast<uint32_t>(kb),
                                              static_cast<uint32_t>(b), stream},
                                           static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
#pragma unroll
                    for (int hb = 0; hb < 2; ++hb) {
                        const int v0 = t * kBN + hb * 64;
                        if (!mine(hb) || !warp_live || failed || v0 >= p.V) continue;   // warp-uniform
                        float y[64];
                        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + hb * 64;
                        uint32_t tt[32];
                        if constexpr (kMode == kResidual) {
                            load_blk(urow, t, hb, u[hb]);
                            load_blk(trow, t, hb, tt);
                        }
                        tc::tmem_ld32(taddr, y);
                        tc::tmem_ld32(taddr + 32, y + 32);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int w = 0; w < 32; ++w) {
                            y[2 * w] = (y[2 * w] + bf16lo(u[hb][w])) * p.cscale;
                            y[2 * w + 1] = (y[2 * w + 1] + bf16hi(u[hb][w])) * p.cscale;
                        }
                        if (kMode == kDraft && have_next) load_blk(urow, tnext, hb, u[hb]);
                        const int blk = 2 * t + hb;
                        const uint32_t wsel = static_cast<uint32_t>(blk) & 3u;
                        const uint32_t rword = wsel == 0 ? pw.x : wsel == 1 ? pw.y : wsel == 2 ? pw.z : pw.w;
                        if constexpr (kMode == kDraft) {
                            if (v0 + 64 > p.V) {
#pragma unroll
                                for (int w = 0; w < 64; ++w)
                                    if (v0 + w >= p.V) y[w] = -INFINITY;
                            }
                            if (p.debug_z != nullptr) {
                                if (valid)                // copies own disjoint blocks
                                    for (int w = 0; w < 64; ++w)
                                        if (v0 + w < p.V) p.debug_z[static_cast<size_t>(b) * p.V + v0 + w] = y[w];
                                continue;
                            }
                            if (p.greedy) {
#pragma unroll
                                for (int w = 0; w < 64; ++w)
                                    if (y[w] > best) { best = y[w]; best_i = v0 + w; }
                            } else {
                                float m4[4] = {y[0], y[1], y[2], y[3]};
#pragma unroll
                                for (int w = 4; w < 64; ++w) m4[w & 3] = fmaxf(m4[w & 3], y[w]);
                                const float mb = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                                if (!(mb > -INFINITY)) continue;   // a block without a finite logit has no mass
                                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                                for (int w = 0; w < 64; ++w) s4[w & 3] += fast_exp2(y[w] - mb);
                                const float sb = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                                const float key = (mb + log2f(sb)) * kLn2 + gumbel_of(uniform_open(rword));
                                if (key > best || (key == best && blk < best_i)) { best = key; best_i = blk; }
                                lse_merge(M, S, mb, sb);
                            }
                        } else {
                            // residual mass q = max(0, p_t - p_d), p_d = 2^(y - ld2), p_t = 2^(t c - lt2)
                            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int w = 0; w < 32; ++w) {
                                const float pd0 = fast_exp2(y[2 * w] - ld2), pd1 = fast_exp2(y[2 * w + 1] - ld2);
                                const float pt0 = fast_exp2(bf16lo(tt[w]) * p.cscale - lt2);
                                const float pt1 = fast_exp2(bf16hi(tt[w]) * p.cscale - lt2);
                                float q0 = fmaxf(pt0 - pd0, 0.f), q1 = fmaxf(pt1 - pd1, 0.f);
                                if (v0 + 2 * w >= p.V) q0 = 0.f;
                                if (v0 + 2 * w + 1 >= p.V) q1 = 0.f;
                                s4[(2 * w) & 3] += q0;
                                s4[(2 * w + 1) & 3] += q1;
                            }
                            const float Q = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                            if (Q > 0.f) {
                                const float key = log2f(Q) * kLn2 + gumbel_of(uniform_open(rword));
                                if (key > best || (key == best && blk < best_i)) { best = key; best_i = blk; }
                            }
                        }
                    }
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[buf]);
                }
                // the next position's first U tile of this lane does not depend on x_k:
                // bring it into L2 while the grid hands over
                if (kMode == kDraft && k < k1 && valid && warp_live) {
                    const int inext = ((eg - (base + ntiles)) % kEpiWG + kEpiWG) % kEpiWG;
                    if (inext < ntiles) {
                        const uint16_t* un = p.U + (static_cast<size_t>(b) * p.gamma + k) * p.V;
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
                            const int v0 = (t_lo + inext) * kBN + hb * 64;
                            if (mine(hb) && v0 < p.V) prefetch_l2(un + v0);
                        }
                    }
                }
                rowres[eg * kBM + lrow] = RowRes{best, best_i, M, S};
            }
            pro_sync();

            // --------------------------------------- publish this position
            if (warp >= 4 && warp < 8 && p.debug_z == nullptr) {
                const int rr = (warp - 4) * 32 + lane;
                const int b = m0 + rr;
                if (rr < nrows && row_k(b, k) > 0) {
                    RowRes r0{-INFINITY, 0x7FFFFFFF, -INFINITY, 0.f};
                    for (int e = 0; e < kEpiWG; ++e)
                        for (int c = 0; c < R; ++c) {
                            const RowRes r1 = rowres[e * kBM + c * rpc + rr];
                            if (r1.key > r0.key || (r1.key == r0.key && r1.idx < r0.idx)) { r0.key = r1.key; r0.idx = r1.idx; }
                            lse_merge(r0.m, r0.s, r1.m, r1.s);
                        }
                    const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
                    if (kMode == kDraft && !p.greedy) p.ws.part[slot * kMaxChunks + pc] = make_float2(r0.m, r0.s);
                    if (r0.key > -INFINITY) atomicMax(&p.ws.words[slot], pack_key(r0.key, static_cast<uint32_t>(r0.idx)));
                    // greedy: the next A row is one of the CTAs' best tokens; bring ours into L2
                    if (kMode == kDraft && p.greedy && k < k1 && r0.idx >= 0 && r0.idx < p.V)
                        for (int off = 0; off < p.r * 2; off += 128)
                            prefetch_l2(reinterpret_cast<const uint8_t*>(p.W1) + static_cast<size_t>(r0.idx) * p.r * 2 + off);
                }
            }
            if (kMode == kDraft && multi && k < k1) arrive();
            else pro_sync();                              // rowres is rewritten by the next position
        }

        if (kMode == kResidual && p.fuse_tail) {
            // ------------------------------------------------ final tokens
            arrive();
            wait_all();                                   // every CTA published its residual blocks
            if (warp >= 2 && *s_fail == 0) {
                const int pair = (warp - 2) >> 1;
                for (int b = blockIdx.x + pair * gridDim.x; b < p.B; b += 5 * gridDim.x)
                    finish_pair<true, 1>(p.fin, b, p.gamma, p.V, p.r, p.U, p.W1, p.E, p.W2, p.x0, p.x, p.cscale, p.seed,
                                         st, 2 + pair, reinterpret_cast<float*>(xch + 2 * pair), xchi + 2 * pair);
            }
        }
        if (kMode == kDraft && p.fuse_tail && p.debug_z == nullptr) {
            // ------------------------------------------ x_gamma and finalize
            arrive();
            wait_all();                                   // every CTA published the last position
            if (!p.greedy) {
                draw_owned(k1);
            } else {
                for (int j = ptid; j < nown; j += kPro) {
                    const int b = blockIdx.x + j * gridDim.x;
                    const unsigned long long w = __ldcg(p.ws.words + static_cast<size_t>(k1 - 1) * p.B + b);
                    const uint32_t idx = unpack_idx(w);
                    int tok = static_cast<int>(idx);
                    if (w == 0ull || idx >= static_cast<uint32_t>(p.V)) {
                        set_status(st, DSPARK_ERR_DEVICE_CHECK, 3);
                        tok = 0;
                    }
                    p.x[b * p.gamma + k1 - 1] = tok;
                }
            }
            pro_sync();
            // one warp per (owned request, position)
            for (int item = warp - 1; item < nown * p.gamma; item += kPro / 32) {
                const int b = blockIdx.x + (item / p.gamma) * gridDim.x, k = item % p.gamma + 1;
                finalize_position<true>(b, k, p.B, p.gamma, p.V, p.H, p.r, p.h, p.W1, p.w, p.bias, p.x0, p.x,
                                        p.greedy, p.P, p.ws.part, p.ws.ytok, p.lse_d, p.logp_d, p.c, st);
            }
            pro_sync();
            for (int j = ptid; j < nown; j += kPro) {     // survival a_k = prod c_1..c_k, in k order
                const int b = blockIdx.x + j * gridDim.x;
                float surv = 1.f;
                for (int kk = 0; kk < p.gamma; ++kk) {
                    const size_t o = static_cast<size_t>(b) * p.gamma + kk;
                    surv = surv * p.c[o];
                    p.a[o] = surv;
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

constexpr size_t kTcSmem = 1024 + 4 * kASlabBytes + kStages * kSlabBytes + (2 * kStages + 4 * kEpiWG) * 8 + 16 +
                           kEpiWG * kBM * sizeof(RowRes) + kBM * 4 + 10 * 8 + 10 * 4 + 16 + 2 * 256 * 4 +
                           2 * 24 * 4 + 16;

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
            return cudaFuncSetAttribute(bias_engine_tc<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kTcSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 1 : 0;
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
