// The draft block's path for small batches (DeepSpec walkthrough, section 3.2
// stage two, `sample_block_tokens`; VanillaMarkovHead, eq. 5): for k = 1..gamma,
// z_k[b][v] = U_k[b][v] + W2[v] . W1[x_{k-1}[b]], then the Gumbel-max draw of x_k
// from softmax(z_k / T) -- the same computation as the tcgen05 engine, for
// batches too small to fill its 128-row tiles.
//
// Below a few dozen requests the rank-r contraction is a matrix-vector product
// per request: each 512-byte row of W2 (r = 256 bf16) meets B rows of W1, so a
// position streams W2 once (78 MB for the Qwen3 vocabulary; it stays in L2 from
// one position to the next) and does B r MACs per row.  One cooperative launch
// covers every position:
//   * one CTA per SM owns a contiguous range of 64-token tiles (the partition the
//     finalize maps tokens to, as for the other paths); a producer warp loads
//     each tile's W2 rows with TMA (4 boxes of 64 rows x 64 k, 128-byte swizzle)
//     and bulk-copies U_k of every request over the tile, into a four-slot ring,
//     running ahead across positions (neither depends on x);
//   * the product runs as warp-level bf16 MMAs with float32 accumulation
//     (m16n8k16: 16 tokens x 8 requests x 16 k): warp w takes the tile's 16-token
//     block w mod 4 and the 8-request blocks w / 4, w / 4 + 4, its A fragments
//     read from the swizzled tile with ldmatrix, its B fragments (the requests'
//     W1 rows, in fragment order) from shared memory, built once per position;
//   * s = z + U_k goes to shared memory, and the CTA's threads then draw: thread
//     (b, g) takes four consecutive tokens of request b, y = s * cscale, key =
//     y - log2(-ln u) with u from word v & 3 of Philox(counter (v >> 2, k, b, 0))
//     -- exactly the engine's draw -- and the 16 threads of a request merge
//     their (max, sum) and best token at the end of the position;
//   * per position every CTA publishes its (max, sum) partials, its best token's
//     y and its winner (atomicMax), then meets the others at a grid barrier;
//     x_{k-1} is the published winner.  After the last position the same launch
//     writes x_gamma and finalizes the requests it owns (lse_d, logp_d, the
//     confidence c_k and the survival a_k).
#pragma once
#include "engine.cuh"
#include "tc.cuh"

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
constexpr int kGroups = 4;                       // warp groups, each with its own ring slot and tiles
constexpr int kMaxB = 16;                        // 2 request blocks of 8
constexpr int kMaxNB = kMaxB / 8;
constexpr int kMaxR = 256;
constexpr int kTile = 64;                        // tokens per tile (the chunk partition's unit)
constexpr int kStages = 4;                       // tile ring
constexpr size_t kBoxBytes = 64 * 128;           // one TMA box: 64 rows x 64 k of bf16, swizzled
constexpr size_t kW2Bytes = kMaxR / 64 * kBoxBytes;                 // a tile's W2 rows (32 KB)
constexpr size_t kStageBytes = kW2Bytes + static_cast<size_t>(kMaxB) * kTile * 2;   // + U_k of every request
constexpr size_t kFragBytes = static_cast<size_t>(kMaxNB) * (kMaxR / 16) * 32 * 8;  // B fragments
constexpr size_t kZBytes = static_cast<size_t>(kGroups) * kMaxB * kTile * 4;   // s = z + U, a tile per group
constexpr size_t kSmem = 1024 + kStages * kStageBytes + kFragBytes + kZBytes;

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
    PhiloxKeys keys;                // the round keys of `seed`
    float* lse_d;
    float* logp_d;
    float* c;
    float* a;
    eng::Ws ws;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                            uint32_t& a3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                 : "r"(addr));
}
// D += A B for one m16n8k16 bf16 tile, float32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// kUHost: U in page-locked host memory, read with loads (bulk copies read device
// memory only).
template <bool kUHost>
__global__ void __launch_bounds__(kThreads, 1)
draft_gemv(const __grid_constant__ CUtensorMap tmW2, Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);   // 1024-byte aligned for the swizzle
    uint8_t* ring = smem;                                 // [kStages]: W2 boxes | U_k [B][kTile] bf16
    uint2* frag = reinterpret_cast<uint2*>(smem + kStages * kStageBytes);   // [nb][k16][lane]
    float* zs = reinterpret_cast<float*>(smem + kStages * kStageBytes + kFragBytes);   // [group][B][kTile]
    __shared__ int s_prev[kMaxB];
    __shared__ float pm[kGroups][kMaxB], ps[kGroups][kMaxB], pk[kGroups][kMaxB], py[kGroups][kMaxB];
    __shared__ int pi[kGroups][kMaxB];
    __shared__ int s_fail;
    __shared__ int s_ring_dead;                           // a tile wait timed out: the producer stopped
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    StatusBlock* st = p.ws.status;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nk16 = p.r / 16;                            // k steps of 16
    const int nslab = p.r / 64;                           // TMA boxes per tile
    const int NB = (p.B + 7) / 8;
    const int chunk = blockIdx.x, nchunk = gridDim.x;
    const int ntiles = (p.V + kTile - 1) / kTile;
    const int j_lo = static_cast<int>(static_cast<long long>(chunk) * ntiles / nchunk);
    const int j_hi = static_cast<int>(static_cast<long long>(chunk + 1) * ntiles / nchunk);
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    if (tid == 0) {
        s_fail = 0;
        s_ring_dead = 0;
        for (int i = 0; i < kStages; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kWarps / kGroups); }
        fence_mbar_init();
        tc::prefetch_tmap(&tmW2);
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------------------------ producer: W2 and U tiles
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool failed = false;
            for (int k = 1; k <= p.gamma && !failed; ++k)
                for (int j = j_lo; j < j_hi; ++j) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u)) { failed = true; break; }
                    const int rows = min(kTile, p.V - j * kTile);   // a multiple of 8 (V % 8 == 0)
                    const uint32_t ubytes = rows * 2u;
                    uint8_t* dst = ring + stage * kStageBytes;
                    // TMA counts the whole box (rows past V are zero-filled)
                    const uint32_t utx = kUHost ? 0u : p.B * ubytes;
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nslab * kBoxBytes) + utx);
                    for (int sl = 0; sl < nslab; ++sl)
                        tc::tma_load_2d(dst + sl * kBoxBytes, &tmW2, sl * 64, j * kTile, &full[stage], keep);
                    for (int b = 0; b < (kUHost ? 0 : p.B); ++b)   // U_k[b] over the tile's tokens
                        bulk_g2s(dst + kW2Bytes + b * (kTile * 2),
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
    // warp group grp (warps 4 grp .. 4 grp + 3) owns ring slot grp: tile i of a
    // position is the (n0 + i)-th tile the producer loads (n0 = (k - 1) T), so it
    // lands in slot (n0 + i) mod 4 and the group of that slot takes it
    const int grp = warp >> 2, w4 = warp & 3, t128 = tid & 127;
    auto gsync = [grp] { asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "n"(kCompute / kGroups) : "memory"); };
    // the draw's items in the group: thread (b, g) takes request b (and b + 8),
    // tokens 4 g .. 4 g + 3 of the tile
    const int gq = t128 & 15, bq = t128 >> 4;
    const int nreq = bq + 8 < p.B ? 2 : (bq < p.B ? 1 : 0);
    const int T = j_hi - j_lo;
    uint32_t cphase = 0;                                  // parity of this group's next wait on its slot
    float* zsg = zs + grp * (kMaxB * kTile);
    const uint8_t* stg = ring + grp * kStageBytes;

    for (int k = 1; k <= p.gamma; ++k) {
        // ------------------------------------------------ x_{k-1}; the B fragments
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
        // fragment (nb, kk, lane): request n = 8 nb + lane / 4, k = 16 kk + 2 (lane % 4) (+ 8)
        for (int item = tid; item < NB * nk16 * 32; item += kCompute) {
            const int ln = item & 31, kk = (item >> 5) % nk16, nb = (item >> 5) / nk16;
            const int n = nb * 8 + (ln >> 2), kq = kk * 16 + 2 * (ln & 3);
            uint2 f = make_uint2(0u, 0u);
            if (n < p.B) {
                const uint32_t* row = reinterpret_cast<const uint32_t*>(p.W1 + static_cast<size_t>(s_prev[n]) * p.r);
                f = make_uint2(__ldg(row + kq / 2), __ldg(row + kq / 2 + 4));
            }
            frag[(nb * (kMaxR / 16) + kk) * 32 + ln] = f;
        }
        csync();

        PhiloxRow pr[2];
        Best best[2];
        float M[2], S[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            pr[q] = philox_row_setup(p.seed, static_cast<uint32_t>(k), static_cast<uint32_t>(bq + 8 * q),
                                     kStreamDraftToken);
            best[q] = Best{-INFINITY, 0x7FFFFFFF, 0.f};
            M[q] = -INFINITY;
            S[q] = 0.f;
        }
        const int n0 = static_cast<int>((static_cast<long long>(k - 1) * T) % kGroups);
        for (int i = (grp - n0 + kGroups) % kGroups; i < T; i += kGroups) {
            const int j = j_lo + i;
            // every issued tile is waited for (no copy may be left in flight at exit),
            // after a failed grid barrier too; only a ring that stopped is skipped
            bool bad = false;
            if (s_ring_dead == 0) bad = !mbar_wait(&full[grp], cphase);
            cphase ^= 1u;
            bad = __any_sync(0xffffffffu, bad);
            if (bad && lane == 0) {
                set_status(st, DSPARK_ERR_TIMEOUT, 16);
                s_ring_dead = 1;
                s_fail = 1;
            }
            // z for tokens 16 w4 .. + 15 and every request block
            if (s_fail == 0) {
                float c[kMaxNB][4] = {};
                const int arow = w4 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;   // ldmatrix row of this lane
                for (int kk = 0; kk < nk16; ++kk) {
                    const int chk = (kk & 3) * 2 + (lane >> 4);                    // 16-byte chunk in the box row
                    const uint32_t addr = smem_u32(stg + (kk >> 2) * kBoxBytes + arow * 128 +
                                                   ((chk ^ (arow & 7)) << 4));
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int nb = 0; nb < kMaxNB; ++nb) {
                        if (nb < NB) {
                            const uint2 f = frag[(nb * (kMaxR / 16) + kk) * 32 + lane];
                            mma_bf16_16816(c[nb], a0, a1, a2, a3, f.x, f.y);
                        }
                    }
                }
                // s = z + U_k: rows g, g + 8 of the block, requests 2 (lane % 4) (+ 1) of each request block
                const int g = lane >> 2, cq = 2 * (lane & 3);
#pragma unroll
                for (int nb = 0; nb < kMaxNB; ++nb) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int n = nb * 8 + cq + (e & 1), row = w4 * 16 + g + (e >> 1) * 8;
                        if (nb < NB && n < p.B) {
                            const int v = j * kTile + row;
                            uint16_t u;
                            if constexpr (kUHost)
                                u = v < p.V ? p.U[(static_cast<size_t>(n) * p.gamma + (k - 1)) * p.V + v] : uint16_t(0);
                            else
                                u = *reinterpret_cast<const uint16_t*>(stg + kW2Bytes + n * (kTile * 2) + row * 2);
                            zsg[n * kTile + row] = c[nb][e] + __uint_as_float(static_cast<uint32_t>(u) << 16);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[grp]);      // this warp is done with the slot
            gsync();                                      // the tile's s is complete
            if (s_fail == 0) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q >= nreq) break;
                    const int b = bq + 8 * q, v0 = j * kTile + 4 * gq;
                    const float4 s4 = *reinterpret_cast<const float4*>(zsg + b * kTile + 4 * gq);
                    float y[4] = {s4.x * p.cscale, s4.y * p.cscale, s4.z * p.cscale, s4.w * p.cscale};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (v0 + e >= p.V) y[e] = -INFINITY;
                    if (p.greedy) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) best_take(best[q], y[e], v0 + e, y[e]);
                    } else {
                        const float m4 = fmaxf(eng::fmax3(y[0], y[1], y[2]), y[3]);
                        if (m4 > -INFINITY) {
                            const float s4s = fast_exp2(y[0] - m4) + fast_exp2(y[1] - m4) + fast_exp2(y[2] - m4) +
                                              fast_exp2(y[3] - m4);
                            lse_merge(M[q], S[q], m4, s4s);
                            const U4 pw = philox_row(pr[q], static_cast<uint32_t>(v0) >> 2, p.keys);
                            const uint32_t wd[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (y[e] > -INFINITY)
                                    best_take(best[q], y[e] - fast_log2(exp_draw(wd[e])), v0 + e, y[e]);
                        }
                    }
                }
            }
            gsync();                                      // zsg is rewritten by the group's next tile
        }

        // ------------------------------------------------ this CTA's partials
        // the 16 threads of a request in a group (a half warp) merge, then thread b
        // merges the groups in group order
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                const float ok = __shfl_xor_sync(0xffffffffu, best[q].key, o);
                const int oi = __shfl_xor_sync(0xffffffffu, best[q].idx, o);
                const float oy = __shfl_xor_sync(0xffffffffu, best[q].y, o);
                const float om = __shfl_xor_sync(0xffffffffu, M[q], o);
                const float os = __shfl_xor_sync(0xffffffffu, S[q], o);
                best_take(best[q], ok, oi, oy);
                lse_merge(M[q], S[q], om, os);
            }
            if (gq == 0 && q < nreq) {
                const int b = bq + 8 * q;
                pm[grp][b] = M[q];
                ps[grp][b] = S[q];
                pk[grp][b] = best[q].key;
                pi[grp][b] = best[q].idx;
                py[grp][b] = best[q].y;
            }
        }
        csync();
        if (tid < p.B && s_fail == 0) {
            const int b = tid;
            Best cb{-INFINITY, 0x7FFFFFFF, 0.f};
            float m = -INFINITY, sum = 0.f;
            for (int gg = 0; gg < kGroups; ++gg) {
                best_take(cb, pk[gg][b], pi[gg][b], py[gg][b]);
                lse_merge(m, sum, pm[gg][b], ps[gg][b]);
            }
            const size_t slot = static_cast<size_t>(k - 1) * p.B + b;
            if (!p.greedy) {
                p.ws.part[slot * kMaxChunks + chunk] = make_float2(m, sum);
                p.ws.ybest[slot * kMaxChunks + chunk] = cb.y;
            }
            if (cb.key > -INFINITY) atomicMax(&p.ws.words[slot], pack_key(cb.key, static_cast<uint32_t>(cb.idx)));
        }
        arrive();                                         // position k published (pm .. py reused after a barrier)
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

// 2-D map over W2 [V][r] bf16: box {64 k, 64 rows}, 128-byte swizzle, zero fill.
inline bool encode_w2_map(CUtensorMap* map, const void* W2, int V, int r) {
    auto enc = eng::tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(V)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(r) * 2};
    const cuuint32_t box[2] = {64, kTile};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W2), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <bool kUHost>
dspark_status_t launch_as(const Params& p, int grid, cudaStream_t s) {
    static OncePerDevice once;
    if (once.run(current_device(), [] {
            return cudaFuncSetAttribute(draft_gemv<kUHost>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    CUtensorMap map;
    if (!encode_w2_map(&map, p.W2, p.V, p.r)) return DSPARK_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1 + (l2_window(&attr[1], p.W2, static_cast<size_t>(p.V) * p.r * 2) ? 1 : 0);   // opt-in
    if (cudaLaunchKernelEx(&cfg, draft_gemv<kUHost>, map, p) != cudaSuccess) {
        cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}

// u_host: U is page-locked host memory (read through its mapping with loads).
inline dspark_status_t launch(const Params& p, int grid, bool u_host, cudaStream_t s) {
    return u_host ? launch_as<true>(p, grid, s) : launch_as<false>(p, grid, s);
}

}  // namespace gemv
}  // namespace dspark
