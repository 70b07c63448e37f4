// dspark_draft_block: the semi-autoregressive draft block of DSpark
// (DeepSpec walkthrough, section 3.2 stage two, `sample_block_tokens`):
//   for k = 1..gamma:  z_k = U_k + W2 . W1[x_{k-1}]   (VanillaMarkovHead, eq. 5)
//                      x_k ~ softmax(z_k / T)          (two-level Gumbel-max)
// plus the confidence head and survival product (section 3.3).
//
// Per phase k (x_k needs a vocabulary-wide reduction before phase k+1 starts):
//   phase kernel   streams U_k, forms the bias tile by tile, and per request
//                  reduces every 64-token sampling block to its logsumexp and
//                  Gumbel key; each CTA publishes its best block (64-bit
//                  atomicMax of (key, ~block)) and its (max, sum) partial;
//   winner kernel  one warp per request: rebuilds z on the winning block only
//                  and draws the token inside it (second Gumbel level).
// After the last phase a finalize kernel forms lse_d / logp_d from the
// partials, and the confidence c_k and survival a_k.
//
// Two phase kernels: a tcgen05 one (bf16, r % 64 == 0, r <= 256): the bias is
// a [128 requests x 128 vocab x r] MMA per tile with W2 tiles streamed by TMA
// (L2 evict-last, reused across phases) and the accumulator in TMEM; and a
// CUDA-core one for fp32 inputs or other ranks.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "host_common.h"
#include "tc.cuh"
#include "../../include/dspark_debug.h"

namespace dspark {

constexpr int kMaxChunks = 256;   // partial slots per (phase, request)

struct DraftWs {
    StatusBlock* status;
    unsigned long long* words;   // [gamma][B] best (key, ~block) or (value, ~token)
    float2* part;                // [gamma][B][kMaxChunks] (max, sum) of y = z log2e / T
    float* ytok;                 // [gamma][B] y of the drawn token
};

inline size_t draft_ws_layout(int B, int gamma, size_t* o_words, size_t* o_part, size_t* o_ytok) {
    size_t o = kStatusBytes;
    *o_words = o;
    o += round_up(static_cast<size_t>(gamma) * B * 8, 256);
    *o_part = o;
    o += round_up(static_cast<size_t>(gamma) * B * kMaxChunks * 8, 256);
    *o_ytok = o;
    o += round_up(static_cast<size_t>(gamma) * B * 4, 256);
    return o;
}

namespace {

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

// Token x_{k-1} of request b (the anchor for k = 1), checked against [0, V).
__device__ __forceinline__ int prev_token(const int32_t* x0, const int32_t* x, int b, int gamma, int k, int V,
                                          StatusBlock* st) {
    const int t = (k == 1) ? x0[b] : x[b * gamma + k - 2];
    if (t < 0 || t >= V) {
        set_status(st, DSPARK_ERR_DEVICE_CHECK, 2);
        return 0;
    }
    return t;
}

__device__ __forceinline__ void ld_u32x4(const void* p, uint32_t* o, uint64_t pol) {
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
                 : "l"(p), "l"(pol));
}

// Combine (m1, s1) += (m2, s2) for sums of 2^(y - m).
__device__ __forceinline__ void lse_merge(float& m1, float& s1, float m2, float s2) {
    if (s2 <= 0.f) return;
    if (s1 <= 0.f) { m1 = m2; s1 = s2; return; }
    const float M = fmaxf(m1, m2);
    s1 = s1 * exp2f(m1 - M) + s2 * exp2f(m2 - M);
    m1 = M;
}

// Block key: logsumexp of the block in natural units plus a Gumbel draw.
__device__ __forceinline__ float block_key(float m, float s, uint64_t seed, int b, int k, int blk) {
    const float u = uniform_open(draw_word(seed, b, k, kStreamDraftBlock, static_cast<uint32_t>(blk)));
    return (m + log2f(s)) * kLn2 + gumbel_of(u);
}

// ==================================================== CUDA-core phase ====
constexpr int kSimtThreads = 256;

template <bool kBF16>
__global__ void __launch_bounds__(kSimtThreads)
draft_phase_simt(int B, int gamma, int V, int r, int k, const void* __restrict__ U,
                 const void* __restrict__ W1, const void* __restrict__ W2, const int32_t* __restrict__ x0,
                 const int32_t* __restrict__ x, float cscale, int greedy, uint64_t seed, int nchunk,
                 DraftWs ws) {
    __shared__ float e[256];
    __shared__ float rk[kSimtThreads / 32], rm[kSimtThreads / 32], rs[kSimtThreads / 32];
    __shared__ int ri[kSimtThreads / 32];
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
    for (int j = threadIdx.x; j < r; j += blockDim.x) e[j] = ld_elem<kBF16>(W1, static_cast<size_t>(prev) * r + j);
    __syncthreads();
    const int nblk = (V + 63) / 64;
    const int lo = static_cast<int>(static_cast<long long>(chunk) * nblk / nchunk);
    const int hi = static_cast<int>(static_cast<long long>(chunk + 1) * nblk / nchunk);
    const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
    float best = -INFINITY, M = -INFINITY, S = 0.f;
    int best_i = 0x7FFFFFFF;
    for (int blk = lo + warp; blk < hi; blk += kSimtThreads / 32) {
        float y[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = blk * 64 + h * 32 + lane;
            if (v < V) {
                float acc = 0.f;
                for (int j = 0; j < r; ++j) acc = fmaf(ld_elem<kBF16>(W2, static_cast<size_t>(v) * r + j), e[j], acc);
                y[h] = (ld_elem<kBF16>(U, urow + v) + acc) * cscale;
            } else {
                y[h] = -INFINITY;
            }
        }
        if (greedy) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = blk * 64 + h * 32 + lane;
                if (y[h] > best || (y[h] == best && v < best_i)) { best = y[h]; best_i = v; }
            }
        } else {
            const float mb = warp_max(fmaxf(y[0], y[1]));
            const float sb = warp_sum(exp2f(y[0] - mb) + exp2f(y[1] - mb));
            const float key = block_key(mb, sb, seed, b, k, blk);
            if (key > best) { best = key; best_i = blk; }   // blocks ascend per warp
            lse_merge(M, S, mb, sb);
        }
    }
    if (greedy) {
        // warp argmax, lowest index on ties
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
            if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
        }
    }
    if (lane == 0) { rk[warp] = best; ri[warp] = best_i; rm[warp] = M; rs[warp] = S; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bk = -INFINITY, m = -INFINITY, s = 0.f;
        int bi = 0x7FFFFFFF;
        for (int w = 0; w < kSimtThreads / 32; ++w) {
            if (rk[w] > bk || (rk[w] == bk && ri[w] < bi)) { bk = rk[w]; bi = ri[w]; }
            lse_merge(m, s, rm[w], rs[w]);
        }
        const size_t slot = static_cast<size_t>(k - 1) * B + b;
        if (!greedy) ws.part[slot * kMaxChunks + chunk] = make_float2(m, s);
        if (bk > -INFINITY) atomicMax(&ws.words[slot], pack_key(bk, static_cast<uint32_t>(bi)));
    }
}

// ===================================================== tcgen05 phase ====
constexpr int kBM = 128;              // requests per M-tile (TMEM lanes)
constexpr int kBN = 128;              // vocabulary columns per tile
constexpr int kBK = 64;               // K per smem slab (128 bytes of bf16)
constexpr int kStages = 6;            // W2 slab ring
constexpr int kEpiWG = 2;             // epilogue warpgroups, two TMEM buffers each
constexpr int kTcThreads = 128 * (1 + kEpiWG);
constexpr int kSlabBytes = kBN * kBK * 2;     // 16 KB
constexpr int kASlabBytes = kBM * kBK * 2;    // 16 KB

struct TcParams {
    int B, gamma, V, r, k;
    const uint16_t* U;
    const uint16_t* W1;
    const int32_t* x0;
    const int32_t* x;
    float cscale;
    int greedy;
    uint64_t seed;
    int P;               // CTAs per M-tile
    DraftWs ws;
    float* debug_z;      // if set: write y = (acc + U) * cscale to [B][V] instead of reducing
};

struct RowRes {
    float key;
    int idx;
    float m, s;
};


__global__ void __launch_bounds__(kTcThreads, 1)
draft_phase_tc(const __grid_constant__ CUtensorMap tmW2, const TcParams p) {
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

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x / p.P, pc = blockIdx.x % p.P;
    const int m0 = g * kBM;
    const int NT = (p.V + kBN - 1) / kBN;
    const int t_lo = static_cast<int>(static_cast<long long>(pc) * NT / p.P);
    const int t_hi = static_cast<int>(static_cast<long long>(pc + 1) * NT / p.P);
    const int ntiles = t_hi - t_lo;
    StatusBlock* st = p.ws.status;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int e = 0; e < 2 * kEpiWG; ++e) { mbar_init(&tfull[e], 1); mbar_init(&tempty[e], 4); }
        fence_mbar_init();
        tc::prefetch_tmap(&tmW2);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);

    // A operand: rows W1[x_{k-1}] of this M-tile, K-major, 128-byte swizzle
    {
        const int cpr = p.r / 8;                          // 16-byte chunks per row
        for (int idx = tid; idx < kBM * cpr; idx += kTcThreads) {
            const int row = idx / cpr, c16 = idx % cpr;
            const int slab = c16 >> 3, c = c16 & 7;
            const int b = m0 + row;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (b < p.B) {
                const int prev = prev_token(p.x0, p.x, b, p.gamma, p.k, p.V, st);
                v = *reinterpret_cast<const uint4*>(p.W1 + static_cast<size_t>(prev) * p.r + c16 * 8);
            }
            uint8_t* dst = sA + slab * kASlabBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = v;
        }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    bool failed = false;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            for (int t = t_lo; t < t_hi && !failed; ++t) {
                for (int s = 0; s < nslab; ++s) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u)) { failed = true; break; }
                    mbar_arrive_expect_tx(&full[stage], kSlabBytes);
                    tc::tma_load_2d(sB + stage * kSlabBytes, &tmW2, s * kBK, t * kBN, &full[stage], pol);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (failed) set_status(st, DSPARK_ERR_TIMEOUT, 10);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < ntiles && !failed; ++i) {
                const int eg = i % kEpiWG, use = i / kEpiWG;
                const int buf = eg * 2 + (use & 1);
                const uint32_t par = static_cast<uint32_t>(use >> 1) & 1u;
                if (!mbar_wait(&tempty[buf], par ^ 1u)) { failed = true; break; }
                tc::fence_after_sync();
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kBN);
                for (int s = 0; s < nslab; ++s) {
                    if (!mbar_wait(&full[stage], phase)) { failed = true; break; }
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t ad = tc::smem_desc_sw128(a0 + s * kASlabBytes + kk * 32);
                        const uint64_t bd = tc::smem_desc_sw128(b0 + stage * kSlabBytes + kk * 32);
                        tc::mma_bf16(d, ad, bd, idesc, (s | kk) != 0);
                    }
                    tc::commit(&empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                tc::commit(&tfull[buf]);
            }
            if (failed) set_status(st, DSPARK_ERR_TIMEOUT, 11);
        }
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue
        const int eg = (warp - 4) >> 2;                   // warpgroup 0..kEpiWG-1
        const int q = warp & 3;                           // TMEM lane quarter
        const int row = q * 32 + lane;
        const int b = m0 + row;
        const bool valid = b < p.B;
        const bool warp_live = (m0 + q * 32) < p.B;
        const uint64_t pol = policy_evict_first();
        const uint16_t* urow = p.U + (static_cast<size_t>(valid ? b : 0) * p.gamma + (p.k - 1)) * p.V;
        float best = -INFINITY, M = -INFINITY, S = 0.f;
        int best_i = 0x7FFFFFFF;
        const int nmine = (ntiles > eg) ? (ntiles - eg + kEpiWG - 1) / kEpiWG : 0;

        uint32_t u[4][16];                                // U of the 4 chunks of one tile
        auto load_u = [&](int t, int j, uint32_t* dst) {
            const int v0 = t * kBN + j * 32;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                if (valid && v0 + g4 * 8 < p.V) ld_u32x4(urow + v0 + g4 * 8, dst + g4 * 4, pol);
                else { dst[g4 * 4] = dst[g4 * 4 + 1] = dst[g4 * 4 + 2] = dst[g4 * 4 + 3] = 0u; }
            }
        };
        if (nmine > 0 && warp_live) {
#pragma unroll
            for (int j = 0; j < 4; ++j) load_u(t_lo + eg, j, u[j]);
        }
        for (int n = 0; n < nmine; ++n) {
            const int i = eg + n * kEpiWG;
            const int t = t_lo + i;
            const int use = n;
            const int buf = eg * 2 + (use & 1);
            const uint32_t par = static_cast<uint32_t>(use >> 1) & 1u;
            bool bad = false;
            if (!failed) bad = !mbar_wait(&tfull[buf], par);
            if (bad) { failed = true; set_status(st, DSPARK_ERR_TIMEOUT, 12); }
            tc::fence_after_sync();
            const bool have_next = (n + 1 < nmine);
            const int tnext = t + kEpiWG;
            float mb = -INFINITY, sb = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!warp_live || failed) continue;
                const int v0 = t * kBN + j * 32;
                float acc[32];
                tc::tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + j * 32, acc);
                tc::tmem_ld_wait();
                float y[32];
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    y[2 * w] = (acc[2 * w] + bf16lo(u[j][w])) * p.cscale;
                    y[2 * w + 1] = (acc[2 * w + 1] + bf16hi(u[j][w])) * p.cscale;
                }
                if (have_next) load_u(tnext, j, u[j]);
#pragma unroll
                for (int w = 0; w < 32; ++w)
                    if (v0 + w >= p.V) y[w] = -INFINITY;
                if (p.debug_z != nullptr) {
                    if (valid)
                        for (int w = 0; w < 32; ++w)
                            if (v0 + w < p.V) p.debug_z[static_cast<size_t>(b) * p.V + v0 + w] = y[w];
                    continue;
                }
                if (p.greedy) {
#pragma unroll
                    for (int w = 0; w < 32; ++w)
                        if (y[w] > best) { best = y[w]; best_i = v0 + w; }
                } else {
                    float mc = y[0];
#pragma unroll
                    for (int w = 1; w < 32; ++w) mc = fmaxf(mc, y[w]);
                    if (mc > -INFINITY) {
                        const float mn = fmaxf(mb, mc);
                        float sc = 0.f;
#pragma unroll
                        for (int w = 0; w < 32; ++w) sc += exp2f(y[w] - mn);
                        sb = (sb > 0.f ? sb * exp2f(mb - mn) : 0.f) + sc;
                        mb = mn;
                    }
                    if (j & 1) {                          // a 64-token block is complete
                        const int blk = (t * kBN + (j - 1) * 32) / 64;
                        if (sb > 0.f) {
                            const float key = block_key(mb, sb, p.seed, b, p.k, blk);
                            if (key > best || (key == best && blk < best_i)) { best = key; best_i = blk; }
                            lse_merge(M, S, mb, sb);
                        }
                        mb = -INFINITY;
                        sb = 0.f;
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        rowres[eg * kBM + row] = RowRes{best, best_i, M, S};
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp >= 4 && warp < 8 && p.debug_z == nullptr) {
        const int row = (warp - 4) * 32 + lane;
        const int b = m0 + row;
        if (b < p.B) {
            RowRes r0 = rowres[row];
            for (int e = 1; e < kEpiWG; ++e) {
                const RowRes r1 = rowres[e * kBM + row];
                if (r1.key > r0.key || (r1.key == r0.key && r1.idx < r0.idx)) { r0.key = r1.key; r0.idx = r1.idx; }
                lse_merge(r0.m, r0.s, r1.m, r1.s);
            }
            const size_t slot = static_cast<size_t>(p.k - 1) * p.B + b;
            if (!p.greedy) p.ws.part[slot * kMaxChunks + pc] = make_float2(r0.m, r0.s);
            if (r0.key > -INFINITY) atomicMax(&p.ws.words[slot], pack_key(r0.key, static_cast<uint32_t>(r0.idx)));
        }
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, 512);
    }
}

constexpr size_t kTcSmem = 1024 + 4 * kASlabBytes + kStages * kSlabBytes + (4 * kStages + 8) * 8 + 16 +
                           kEpiWG * kBM * sizeof(RowRes);

// ============================================================ winner ====
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

// Two warps per request: the token inside the winning 64-token block (greedy:
// the argmax token itself) and y at that token.  Warp w rebuilds z for tokens
// blk*64 + 32w + (0..31): every lane loads one 16-byte chunk of each W2 row
// (coalesced rows), forms its partial dot products, and a transpose-reduce
// leaves token (32w + lane)'s dot product in lane `lane`.
template <bool kBF16, int kCPL>
__global__ void __launch_bounds__(64)
draft_winner(int B, int gamma, int V, int r, int k, const void* __restrict__ U, const void* __restrict__ W1,
             const void* __restrict__ W2, const int32_t* __restrict__ x0, int32_t* __restrict__ x,
             float cscale, int greedy, uint64_t seed, DraftWs ws) {
    constexpr int EPC = kBF16 ? 8 : 4;                    // elements per 16-byte chunk
    __shared__ float sbest[2], sy[2];
    __shared__ int sidx[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const size_t slot = static_cast<size_t>(k - 1) * B + b;
    const unsigned long long word = ws.words[slot];
    if (word == 0ull) {
        if (threadIdx.x == 0) { set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 3); x[b * gamma + k - 1] = 0; }
        return;
    }
    const uint32_t idx = unpack_idx(word);
    if (greedy) {
        if (threadIdx.x == 0) { x[b * gamma + k - 1] = static_cast<int>(idx); ws.ytok[slot] = 0.f; }
        return;
    }
    const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
    const int nch = r / EPC;                              // 16-byte chunks per row
    float e[kCPL][EPC];
#pragma unroll
    for (int cc = 0; cc < kCPL; ++cc) {
        const int c = lane + 32 * cc;
#pragma unroll
        for (int q = 0; q < EPC; ++q)
            e[cc][q] = (c < nch) ? ld_elem<kBF16>(W1, static_cast<size_t>(prev) * r + c * EPC + q) : 0.f;
    }
    const int vbase = static_cast<int>(idx) * 64 + warp * 32;
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
                if (v < V && c < nch)   // volatile loads: all issue before the first use
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
    const int v = vbase + lane;
    float score = -INFINITY, yv = 0.f;
    if (v < V) {
        const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
        yv = (part[0] + ld_elem<kBF16>(U, urow + v)) * cscale;
        const float g = gumbel_of(uniform_open(draw_word(seed, b, k, kStreamDraftToken, static_cast<uint32_t>(v))));
        score = yv + g * kLog2e;
    }
    int bi = (v < V) ? v : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, score, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const float oy = __shfl_xor_sync(0xffffffffu, yv, o);
        if (os > score || (os == score && oi < bi)) { score = os; bi = oi; yv = oy; }
    }
    if (lane == 0) { sbest[warp] = score; sidx[warp] = bi; sy[warp] = yv; }
    __syncthreads();
    if (threadIdx.x == 0) {
        int w = 0;
        if (sbest[1] > sbest[0] || (sbest[1] == sbest[0] && sidx[1] < sidx[0])) w = 1;
        x[b * gamma + k - 1] = (sidx[w] == 0x7FFFFFFF) ? 0 : sidx[w];
        ws.ytok[slot] = sy[w];
    }
}

// ========================================================== finalize ====
template <bool kBF16>
__global__ void __launch_bounds__(256)
draft_finalize(int B, int gamma, int V, int H, int r, const void* __restrict__ h, const void* __restrict__ W1,
               const void* __restrict__ w, float bias, const int32_t* __restrict__ x0,
               const int32_t* __restrict__ x, int greedy, int nchunk, float* __restrict__ lse_d,
               float* __restrict__ logp_d, float* __restrict__ c, float* __restrict__ a, DraftWs ws) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 8 + warp;
    if (b >= B) return;
    float surv = 1.f;
    for (int k = 1; k <= gamma; ++k) {
        const size_t slot = static_cast<size_t>(k - 1) * B + b;
        float L = 0.f, lp = 0.f;
        if (!greedy) {
            float m = -INFINITY, s = 0.f;
            for (int ch = lane; ch < nchunk; ch += 32) {
                const float2 pr = ws.part[slot * kMaxChunks + ch];
                lse_merge(m, s, pr.x, pr.y);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float om = __shfl_xor_sync(0xffffffffu, m, o);
                const float os = __shfl_xor_sync(0xffffffffu, s, o);
                lse_merge(m, s, om, os);
            }
            const float L2 = m + log2f(s);
            L = L2 * kLn2;
            lp = (ws.ytok[slot] - L2) * kLn2;
        }
        const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
        const size_t hrow = (static_cast<size_t>(b) * gamma + (k - 1)) * H;
        float acc = 0.f;
        for (int i = lane; i < H; i += 32) acc = fmaf(ld_elem<kBF16>(w, i), ld_elem<kBF16>(h, hrow + i), acc);
        for (int j = lane; j < r; j += 32)
            acc = fmaf(ld_elem<kBF16>(w, H + j), ld_elem<kBF16>(W1, static_cast<size_t>(prev) * r + j), acc);
        const float logit = warp_sum(acc) + bias;
        const float ck = 1.f / (1.f + expf(-logit));
        surv = surv * ck;
        if (lane == 0) {
            const size_t o = static_cast<size_t>(b) * gamma + (k - 1);
            lse_d[o] = L;
            logp_d[o] = lp;
            c[o] = ck;
            a[o] = surv;
        }
    }
}

// ====================================================== host launch ====
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
bool encode_w2_map(CUtensorMap* map, const void* W2, int V, int r) {
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

bool use_tc_path(dspark_dtype_t dt, int r) { return dt == DSPARK_BF16 && r % kBK == 0 && r <= 256; }

dspark_status_t launch_phase_tc(const CUtensorMap& map, const TcParams& p, int grid, cudaStream_t s) {
    static OncePerDevice once;
    if (once.run(current_device(), [] {
            return cudaFuncSetAttribute(draft_phase_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kTcSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    draft_phase_tc<<<grid, kTcThreads, kTcSmem, s>>>(map, p);
    return launch_status();
}

// Grid of the tcgen05 phase: nM M-tiles, P CTAs each (P * nM <= SMs).
void tc_grid(int B, int V, int* nM, int* P) {
    *nM = (B + kBM - 1) / kBM;
    const int sms = sm_count(current_device());
    int per = sms / *nM;
    if (per < 1) per = 1;
    const int NT = (V + kBN - 1) / kBN;
    if (per > NT) per = NT;
    if (per > kMaxChunks) per = kMaxChunks;
    *P = per;
}

int simt_chunks(int V) {
    const int nblk = (V + 63) / 64;
    int n = (nblk + 7) / 8;
    if (n > kMaxChunks) n = kMaxChunks;
    return n < 1 ? 1 : n;
}

}  // namespace

// Full draft block on `s`.
dspark_status_t draft_block_impl(int B, int gamma, int V, int H, int r, dspark_dtype_t dt, const void* U,
                                 const void* h, const void* W1, const void* W2, const void* w, float bias,
                                 const int32_t* x0, float temperature, uint64_t seed, int32_t* x, float* lse_d,
                                 float* logp_d, float* c, float* a, void* workspace, cudaStream_t s) {
    size_t ow, op, oy;
    draft_ws_layout(B, gamma, &ow, &op, &oy);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    DraftWs ws{reinterpret_cast<StatusBlock*>(wsb), reinterpret_cast<unsigned long long*>(wsb + ow),
               reinterpret_cast<float2*>(wsb + op), reinterpret_cast<float*>(wsb + oy)};
    if (cudaMemsetAsync(wsb, 0, op, s) != cudaSuccess) return DSPARK_ERR_CUDA;   // status + words
    const int greedy = (temperature == 0.f);
    const float cscale = greedy ? 1.f : kLog2e / temperature;
    const bool tcp = use_tc_path(dt, r);
    CUtensorMap map;
    int nM = 1, P = 1, nchunk = 1;
    if (tcp) {
        if (!encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
        tc_grid(B, V, &nM, &P);
        nchunk = P;
    } else {
        nchunk = simt_chunks(V);
    }
    const bool bf = (dt == DSPARK_BF16);
    for (int k = 1; k <= gamma; ++k) {
        dspark_status_t stt;
        if (tcp) {
            TcParams p{B, gamma, V, r, k, static_cast<const uint16_t*>(U), static_cast<const uint16_t*>(W1), x0, x,
                       cscale, greedy, seed, P, ws, nullptr};
            stt = launch_phase_tc(map, p, nM * P, s);
        } else {
            dim3 grid(nchunk, B);
            if (bf)
                draft_phase_simt<true><<<grid, kSimtThreads, 0, s>>>(B, gamma, V, r, k, U, W1, W2, x0, x, cscale,
                                                                     greedy, seed, nchunk, ws);
            else
                draft_phase_simt<false><<<grid, kSimtThreads, 0, s>>>(B, gamma, V, r, k, U, W1, W2, x0, x, cscale,
                                                                      greedy, seed, nchunk, ws);
            stt = launch_status();
        }
        if (stt != DSPARK_OK) return stt;
        // chunks of 16 bytes per W2 row: up to 32 (bf16, r <= 256) or 64 (f32) -> 1 or 2 per lane
        if (bf)
            draft_winner<true, 1><<<B, 64, 0, s>>>(B, gamma, V, r, k, U, W1, W2, x0, x, cscale, greedy, seed, ws);
        else if (r <= 128)
            draft_winner<false, 1><<<B, 64, 0, s>>>(B, gamma, V, r, k, U, W1, W2, x0, x, cscale, greedy, seed, ws);
        else
            draft_winner<false, 2><<<B, 64, 0, s>>>(B, gamma, V, r, k, U, W1, W2, x0, x, cscale, greedy, seed, ws);
        if ((stt = launch_status()) != DSPARK_OK) return stt;
    }
    const int fgrid = (B + 7) / 8;
    if (bf)
        draft_finalize<true><<<fgrid, 256, 0, s>>>(B, gamma, V, H, r, h, W1, w, bias, x0, x, greedy, nchunk, lse_d,
                                                   logp_d, c, a, ws);
    else
        draft_finalize<false><<<fgrid, 256, 0, s>>>(B, gamma, V, H, r, h, W1, w, bias, x0, x, greedy, nchunk, lse_d,
                                                    logp_d, c, a, ws);
    return launch_status();
}

// Debug: z = (U_k + W2 . W1[prev]) for one phase through the tcgen05 path,
// written as float [B][V].  `prev` plays the role of x0 (k = 1).
dspark_status_t debug_tc_logits(int B, int V, int r, const void* U, const void* W1, const void* W2,
                                const int32_t* prev, float* z, void* workspace, cudaStream_t s) {
    if (!use_tc_path(DSPARK_BF16, r)) return DSPARK_ERR_UNSUPPORTED;
    CUtensorMap map;
    if (!encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
    int nM, P;
    tc_grid(B, V, &nM, &P);
    size_t ow, op, oy;
    draft_ws_layout(B, 1, &ow, &op, &oy);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    DraftWs ws{reinterpret_cast<StatusBlock*>(wsb), reinterpret_cast<unsigned long long*>(wsb + ow),
               reinterpret_cast<float2*>(wsb + op), reinterpret_cast<float*>(wsb + oy)};
    if (cudaMemsetAsync(wsb, 0, 16, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    TcParams p{B, 1, V, r, 1, static_cast<const uint16_t*>(U), static_cast<const uint16_t*>(W1), prev, nullptr,
               1.f, 1, 0, P, ws, z};
    return launch_phase_tc(map, p, nM * P, s);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_draft_block_workspace_size(int B, int gamma, int V, int r) {
    (void)V;
    (void)r;
    if (B <= 0 || gamma <= 0) return kStatusBytes;
    size_t ow, op, oy;
    return draft_ws_layout(B, gamma, &ow, &op, &oy);
}

extern "C" dspark_status_t dspark_draft_block(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                              const void* U, const void* h, const void* W1, const void* W2,
                                              const void* w, float bias, const int32_t* x0, float temperature,
                                              uint64_t seed, int32_t* x, float* lse_d, float* logp_d, float* c,
                                              float* a, void* workspace, size_t workspace_bytes,
                                              dspark_stream_t stream) {
    if (B <= 0 || B > 65535 || gamma <= 0 || gamma > DSPARK_MAX_GAMMA || V <= 0 || H < 0 || r <= 0 || r > 256)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (dt != DSPARK_F32 && dt != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!(temperature >= 0.f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0 || r % 8 != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!U || !W1 || !W2 || !w || !x0 || !x || !lse_d || !logp_d || !c || !a || (H > 0 && !h))
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (!aligned16(U) || !aligned16(W1) || !aligned16(W2)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_draft_block_workspace_size(B, gamma, V, r)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    return draft_block_impl(B, gamma, V, H, r, dt, U, h, W1, W2, w, bias, x0, temperature, seed, x, lse_d, logp_d,
                            c, a, workspace, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dspark_status_t dspark_debug_draft_logits(int B, int V, int r, const void* U_k, const void* W1,
                                                     const void* W2, const int32_t* prev, float* z,
                                                     void* workspace, size_t workspace_bytes,
                                                     dspark_stream_t stream) {
    if (B <= 0 || V <= 0 || V % 8 != 0 || r <= 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!U_k || !W1 || !W2 || !prev || !z || !workspace || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_draft_block_workspace_size(B, 1, V, r)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    return debug_tc_logits(B, V, r, U_k, W1, W2, prev, z, workspace, reinterpret_cast<cudaStream_t>(stream));
}
