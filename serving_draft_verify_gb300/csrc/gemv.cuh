// The draft block's CUDA-core path for small batches (DeepSpec walkthrough,
// section 3.2 stage two, `sample_block_tokens`; VanillaMarkovHead, eq. 5):
// for k = 1..gamma, z_k[b][v] = U_k[b][v] + W2[v] . W1[x_{k-1}[b]], then the
// Gumbel-max draw of x_k from softmax(z_k / T) -- the same computation as the
// tcgen05 engine, for batches too small to fill its 128-row tiles.
//
// Below a few dozen requests the rank-r contraction is a matrix-vector product
// per request: each 512-byte row of W2 (r = 256 bf16) meets B rows of W1, so the
// position streams W2 once (78 MB for the Qwen3 vocabulary, kept in L2 with the
// evict-last policy so that the next position reads it from there) and the work
// per byte is B r / 512 MACs.  One cooperative launch covers every position:
//   * one CTA per SM owns a contiguous range of 64-token tiles (the partition
//     the finalize maps tokens to, as for the other paths); a producer warp
//     bulk-copies each tile's W2 rows (32 KB) and the B rows of U_k over it into
//     a ring of four slots, running ahead across positions (neither depends
//     on x);
//   * each of 16 warps takes four tokens of a tile, eight lanes per token, each
//     lane holding r / 8 of the row's weights in registers and reading the B
//     rows W1[x_{k-1}] from shared memory, permuted so that the eight lanes of a
//     token read 128 contiguous bytes;
//   * the four tokens' dot products meet in shared memory, and lane b draws them
//     for request b: y = (z + U) * cscale, key = y - log2(-ln u) with u from
//     word v & 3 of Philox(counter (v >> 2, k, b, 0)) -- one Philox block per
//     four tokens -- exactly the engine's draw;
//   * per position every CTA publishes its (max, sum) partials, its best token's
//     y and its winner (atomicMax), then meets the others at a grid barrier;
//     x_{k-1} is the published winner.  After the last position the same launch
//     writes x_gamma and finalizes the requests it owns (lse_d, logp_d, the
//     confidence c_k and the survival a_k).
#pragma once
#include "engine.cuh"

namespace dspark {
namespace gemv {

using eng::Best;
using eng::best_take;
using eng::kMaxChunks;
using eng::lse_merge;
using eng::pack_key;
using eng::unpack_idx;
using eng::ld_u32x4;

constexpr int kWarps = 16;                       // compute warps; warp kWarps is the producer
constexpr int kCompute = kWarps * 32;
constexpr int kThreads = kCompute + 32;
constexpr int kMaxB = 32;                        // one request per lane in the draw
constexpr int kMaxR = 256;
constexpr int kTile = 4 * kWarps;                // tokens per tile (the chunk partition's unit)
constexpr int kStages = 4;                       // W2 tile ring
constexpr size_t kTileBytes = static_cast<size_t>(kTile) * kMaxR * 2;     // W2 rows of a tile
constexpr size_t kStageBytes = kTileBytes + static_cast<size_t>(kMaxB) * kTile * 2;   // + U_k of every request
constexpr size_t kSmem = kStages * kStageBytes + static_cast<size_t>(kMaxB) * kMaxR * 4;   // ring | W1 rows

struct Params {
    int B, gamma, V, H, r;
    const uint16_t* U;              // [B][gamma][V] bf16
    const uint16_t* W1;             // [V][r] bf16
    const uint16_t* W2;             // [V][r] bf16
    const uint16_t* h;              // [B][gamma][H] bf16
    const uint16_t* w;              // [H + r] bf16
    float bias;
    const int32_t* x0;
    int32_t* x;
    float cscale;
    int greedy;
    uint64_t seed;
    float* lse_d;
    float* logp_d;
    float* c;
    float* a;
    eng::Ws ws;
};

// Element j = 64 i + 8 s + 4 hh + q of a W1 row (i < r / 64, s < 8, hh < 2,
// q < 4) sits at float ((2 i + hh) 8 + s) 4 + q of its shared-memory row: lane s
// of a token reads its two 16-byte halves at (2 i + hh) 128 + 16 s bytes.
__device__ __forceinline__ int eperm(int j) {
    const int i = j >> 6, s = (j >> 3) & 7, hh = (j >> 2) & 1, q = j & 3;
    return (((2 * i + hh) << 3) + s) * 4 + q;
}

__global__ void __launch_bounds__(kThreads, 1)
draft_gemv(Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;                                  // [kStages]: W2 [kTile][r] | U_k [B][kTile], bf16
    float* es = reinterpret_cast<float*>(smem + kStages * kStageBytes);   // [B][r] float32, permuted rows
    __shared__ __align__(16) float zt[kWarps][kMaxB][4];  // a warp's four tokens' dot products
    __shared__ float rm[kWarps][kMaxB], rs[kWarps][kMaxB], rk[kWarps][kMaxB], ry[kWarps][kMaxB];
    __shared__ int ri[kWarps][kMaxB];
    __shared__ int s_prev[kMaxB];
    __shared__ int s_fail;
    __shared__ int s_ring_dead;                           // a tile wait timed out: the producer stopped
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    StatusBlock* st = p.ws.status;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = lane >> 3, s = lane & 7;                // token of the warp's four, r-slice of the lane
    const int nq = p.r / 64;                              // 16-byte pieces per lane (1..4)
    const int chunk = blockIdx.x, nchunk = gridDim.x;
    const int ntiles = (p.V + kTile - 1) / kTile;
    const int j_lo = static_cast<int>(static_cast<long long>(chunk) * ntiles / nchunk);
    const int j_hi = static_cast<int>(static_cast<long long>(chunk + 1) * ntiles / nchunk);
    const size_t row_bytes = static_cast<size_t>(p.r) * 2;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    if (tid == 0) {
        s_fail = 0;
        s_ring_dead = 0;
        for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kWarps); }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------------------------ producer: W2 tiles
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool failed = false;
            for (int k = 1; k <= p.gamma && !failed; ++k)
                for (int j = j_lo; j < j_hi; ++j) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u)) { failed = true; break; }
                    const int rows = min(kTile, p.V - j * kTile);   // a multiple of 8 (V % 8 == 0)
                    const uint32_t wbytes = static_cast<uint32_t>(rows * row_bytes), ubytes = rows * 2u;
                    uint8_t* dst = ring + stage * kStageBytes;
                    mbar_arrive_expect_tx(&full[stage], wbytes + p.B * ubytes);
                    bulk_g2s(dst, reinterpret_cast<const uint8_t*>(p.W2) + j * kTile * row_bytes, wbytes,
                             &full[stage], keep);
                    for (int b = 0; b < p.B; ++b)             // U_k[b] over the tile's tokens
                        bulk_g2s(dst + kTileBytes + b * (kTile * 2),
                                 p.U + (static_cast<size_t>(b) * p.gamma + (k - 1)) * p.V + j * kTile, ubytes,
                                 &full[stage], drop);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            if (failed) set_status(st, DSPARK_ERR_TIMEOUT, 15);
        }
        return;                                           // no block-wide barrier follows
    }

    // ---------------------------------------------------- compute warps
    auto csync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory"); };
    unsigned int epoch = 0;
    auto arrive = [&] {
        csync();                                          // this CTA's writes of the step are done
        if (tid == 0) eng::grid_arrive(p.ws.gbar);
        ++epoch;
    };
    auto wait_all = [&] {
        if (tid == 0 && s_fail == 0 && !eng::grid_wait(p.ws.gbar, epoch * gridDim.x)) {
            set_status(st, DSPARK_ERR_TIMEOUT, 14);
            s_fail = 1;
        }
        csync();
    };
    auto winner = [&](int b, int k) -> int {
        const unsigned long long wd = __ldcg(p.ws.words + static_cast<size_t>(k - 1) * p.B + b);
        const uint32_t idx = unpack_idx(wd);
        if (wd == 0ull || idx >= static_cast<uint32_t>(p.V)) {
            set_status(st, DSPARK_ERR_DEVICE_CHECK, 3);
            return 0;
        }
        return static_cast<int>(idx);
    };
    int cstage = 0;
    uint32_t cphase = 0;

    for (int k = 1; k <= p.gamma; ++k) {
        // ------------------------------------------------ x_{k-1} and its W1 rows
        if (k > 1) wait_all();                            // every CTA published position k-1
        if (tid < p.B) {
            const int b = tid;
            int tok;
            if (k == 1) {
                tok = eng::prev_token(p.x0, p.x, b, p.gamma, 1, p.V, st);
            } else {
                tok = (s_fail == 0) ? winner(b, k - 1) : 0;
                if (chunk == 0) p.x[b * p.gamma + k - 2] = tok;
            }
            s_prev[b] = tok;
        }
        csync();
        for (int item = tid; item < p.B * (p.r / 8); item += kCompute) {
            const int b = item / (p.r / 8), j8 = item % (p.r / 8);
            uint32_t wv[4];
            ld_u32x4(p.W1 + static_cast<size_t>(s_prev[b]) * p.r + j8 * 8, wv, keep);
            float* dst = es + b * p.r;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dst[eperm(j8 * 8 + 2 * q)] = bf16lo(wv[q]);
                dst[eperm(j8 * 8 + 2 * q + 1)] = bf16hi(wv[q]);
            }
        }
        csync();

        // ------------------------------------------------ this CTA's tiles
        const PhiloxRow pr = philox_row_setup(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(lane),
                                              kStreamDraftToken);
        Best best{-INFINITY, 0x7FFFFFFF, 0.f};
        float M = -INFINITY, S = 0.f;
        for (int j = j_lo; j < j_hi; ++j) {
            const int v0 = j * kTile + 4 * warp;          // this warp's four tokens
            // every issued tile is waited for (no copy may be left in flight at exit),
            // after a failed grid barrier too; only a ring that stopped is skipped
            bool bad = false;
            if (s_ring_dead == 0) bad = !mbar_wait(&full[cstage], cphase);
            bad = __any_sync(0xffffffffu, bad);
            if (bad && lane == 0) {
                set_status(st, DSPARK_ERR_TIMEOUT, 16);
                s_ring_dead = 1;
                s_fail = 1;
            }
            // this lane's r / 8 weights of token v0 + t, as float32 pairs
            unsigned long long wf[16];
            {
                const uint8_t* row = ring + cstage * kStageBytes + (4 * warp + t) * row_bytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 q4 = make_uint4(0u, 0u, 0u, 0u);
                    if (i < nq) q4 = *reinterpret_cast<const uint4*>(row + i * 128 + s * 16);
                    wf[4 * i] = eng::f2pack(bf16lo(q4.x), bf16hi(q4.x));
                    wf[4 * i + 1] = eng::f2pack(bf16lo(q4.y), bf16hi(q4.y));
                    wf[4 * i + 2] = eng::f2pack(bf16lo(q4.z), bf16hi(q4.z));
                    wf[4 * i + 3] = eng::f2pack(bf16lo(q4.w), bf16hi(q4.w));
                }
            }
            // U_k of request `lane` at the warp's four tokens
            uint2 u2 = make_uint2(0u, 0u);
            if (lane < p.B)
                u2 = *reinterpret_cast<const uint2*>(ring + cstage * kStageBytes + kTileBytes + lane * (kTile * 2) +
                                                     (4 * warp) * 2);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[cstage]);   // this warp's rows are in registers
            if (++cstage == kStages) { cstage = 0; cphase ^= 1u; }
            if (s_fail != 0) continue;
            // dot products with every request's W1 row; the eight lanes of a token meet by xor
            for (int b = 0; b < p.B; ++b) {
                const float4* er = reinterpret_cast<const float4*>(es + b * p.r);
                unsigned long long acc0 = eng::f2pack(0.f, 0.f), acc1 = acc0;   // two chains
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < nq) {
                        const float4 e0 = er[(2 * i) * 8 + s], e1 = er[(2 * i + 1) * 8 + s];
                        acc0 = eng::f2fma(wf[4 * i], eng::f2pack(e0.x, e0.y), acc0);
                        acc1 = eng::f2fma(wf[4 * i + 1], eng::f2pack(e0.z, e0.w), acc1);
                        acc0 = eng::f2fma(wf[4 * i + 2], eng::f2pack(e1.x, e1.y), acc0);
                        acc1 = eng::f2fma(wf[4 * i + 3], eng::f2pack(e1.z, e1.w), acc1);
                    }
                }
                float lo, hi;
                eng::f2unpack(eng::f2add(acc0, acc1), lo, hi);
                float dot = lo + hi;
                dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                if (s == (b & 7)) zt[warp][b][t] = dot;
            }
            __syncwarp();
            if (lane < p.B) {
                const int b = lane;
                const float4 z4 = *reinterpret_cast<const float4*>(&zt[warp][b][0]);
                float y[4] = {(z4.x + bf16lo(u2.x)) * p.cscale, (z4.y + bf16hi(u2.x)) * p.cscale,
                              (z4.z + bf16lo(u2.y)) * p.cscale, (z4.w + bf16hi(u2.y)) * p.cscale};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (v0 + q >= p.V) y[q] = -INFINITY;
                if (p.greedy) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) best_take(best, y[q], v0 + q, y[q]);
                } else {
                    const float m4 = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
                    if (m4 > -INFINITY) {
                        const float s4 = fast_exp2(y[0] - m4) + fast_exp2(y[1] - m4) + fast_exp2(y[2] - m4) +
                                         fast_exp2(y[3] - m4);
                        lse_merge(M, S, m4, s4);
                        const U4 pw = philox_row(pr, static_cast<uint32_t>(v0) >> 2);
                        const uint32_t wd[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (y[q] > -INFINITY) best_take(best, y[q] - fast_log2(exp_draw(wd[q])), v0 + q, y[q]);
                    }
                }
            }
            __syncwarp();                                 // zt is rewritten by the next tile
        }

        // ------------------------------------------------ this CTA's partials
        if (lane < p.B) {
            rm[warp][lane] = M;
            rs[warp][lane] = S;
            rk[warp][lane] = best.key;
            ri[warp][lane] = best.idx;
            ry[warp][lane] = best.y;
        }
        csync();
        if (tid < p.B && s_fail == 0) {
            const int b = tid;
            Best cb{-INFINITY, 0x7FFFFFFF, 0.f};
            float m = -INFINITY, sum = 0.f;
            for (int wi = 0; wi < kWarps; ++wi) {
                best_take(cb, rk[wi][b], ri[wi][b], ry[wi][b]);
                lse_merge(m, sum, rm[wi][b], rs[wi][b]);
            }
            const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
            if (!p.greedy) {
                p.ws.part[slot * kMaxChunks + chunk] = make_float2(m, sum);
                p.ws.ybest[slot * kMaxChunks + chunk] = cb.y;
            }
            if (cb.key > -INFINITY) atomicMax(&p.ws.words[slot], pack_key(cb.key, static_cast<uint32_t>(cb.idx)));
        }
        arrive();                                         // position k published (rm .. ri are reused after a barrier)
    }

    // ---------------------------------------------------- x_gamma and finalize
    const int nown = (chunk < p.B) ? (p.B - 1 - chunk) / nchunk + 1 : 0;
    wait_all();                                           // every CTA published the last position
    for (int j = tid; j < nown; j += kCompute) {
        const int b = chunk + j * nchunk;
        p.x[b * p.gamma + p.gamma - 1] = (s_fail == 0) ? winner(b, p.gamma) : 0;
    }
    csync();
    for (int item = warp; item < nown * p.gamma; item += kWarps) {   // one warp per (owned request, position)
        const int b = chunk + (item / p.gamma) * nchunk, k = item % p.gamma + 1;
        eng::finalize_position<true>(b, k, p.B, p.gamma, p.V, p.H, p.r, p.h, p.W1, p.w, p.bias, p.x0, p.x,
                                     p.greedy, nchunk, kTile, ntiles, p.ws.part, p.ws.ybest, p.lse_d, p.logp_d,
                                     p.c, st);
    }
    csync();
    for (int j = tid; j < nown; j += kCompute) {          // survival a_k = prod c_1..c_k, in k order
        const int b = chunk + j * nchunk;
        float surv = 1.f;
        for (int kk = 0; kk < p.gamma; ++kk) {
            const size_t o = static_cast<size_t>(b) * p.gamma + kk;
            surv = surv * p.c[o];
            p.a[o] = surv;
        }
    }
}

// The path applies to bf16 weights with r a multiple of 64 up to 256 (the
// engine's ranks) and B up to kMaxB.
inline bool supported(dspark_dtype_t dt, int B, int r) {
    return dt == DSPARK_BF16 && r % 64 == 0 && r <= kMaxR && B >= 1 && B <= kMaxB;
}

// One CTA per SM (at most kMaxChunks, at most one per tile), all co-resident.
inline int grid_for(int V) {
    int g = sm_count(current_device());
    const int nunits = (V + kTile - 1) / kTile;
    if (g > kMaxChunks) g = kMaxChunks;
    if (g > nunits) g = nunits;
    return g < 1 ? 1 : g;
}

inline dspark_status_t launch(const Params& p, int grid, cudaStream_t s) {
    static OncePerDevice once;
    if (once.run(current_device(), [] {
            return cudaFuncSetAttribute(draft_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kStages * kStageBytes + static_cast<size_t>(p.B) * p.r * 4;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, draft_gemv, p) != cudaSuccess) {
        cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}

}  // namespace gemv
}  // namespace dspark
