// dspark_draft_block: the semi-autoregressive draft block of DSpark
// (DeepSpec walkthrough, section 3.2 stage two, `sample_block_tokens`):
//   for k = 1..gamma:  z_k = U_k + W2 . W1[x_{k-1}]   (VanillaMarkovHead, eq. 5;
//                      dspark_draft_block_ex: W2 . e_k of a gated or recurrent head)
//                      x_k ~ softmax(z_k / T)          (Gumbel-max over the vocabulary)
// plus the confidence head and survival product (section 3.3).
//
// Tensor-core path (bf16, r % 64 == 0): one cooperative launch of the bias
// engine (engine.cuh) runs every position; between positions its CTAs meet at
// a grid barrier, after which each request's published winner is x_{k-1}.
// After the last position the same launch writes x_gamma and finalizes the
// requests each CTA owns.
// CUDA-core path (and the tensor-core path when the grid cannot be
// co-resident): per position a phase kernel (the Gumbel-max draw and the
// (max, sum) of each chunk of the vocabulary, the chunk's winner published by
// atomicMax) and a winner kernel that writes x_k.  There, after the last
// position a finalize kernel forms lse_d / logp_d and the confidence c_k and
// survival a_k.
#include "engine.cuh"
#include "gemv.cuh"
#include "../../include/dspark_debug.h"

namespace dspark {

using eng::kMaxChunks;
using eng::lse_merge;
using eng::ld_elem;
using eng::pack_key;
using eng::prev_token;
using eng::unpack_idx;
using eng::Best;
using eng::best_take;
using DraftWs = eng::Ws;

// Workspace: status | grid-barrier counter | words [gamma][B] | partials
// [gamma][B][kMaxChunks] (max, sum) | y of each chunk's best token
// [gamma][B][kMaxChunks].  The first three are cleared by every call; the
// chunk entries are written before they are read.
inline size_t draft_ws_layout(int B, int gamma, size_t* o_bar, size_t* o_words, size_t* o_part, size_t* o_yb) {
    size_t o = kStatusBytes;
    *o_bar = o;
    o += 256;
    *o_words = o;
    o += round_up(static_cast<size_t>(gamma) * B * 8, 256);
    *o_part = o;
    o += round_up(static_cast<size_t>(gamma) * B * kMaxChunks * 8, 256);
    *o_yb = o;
    o += round_up(static_cast<size_t>(gamma) * B * kMaxChunks * 4, 256);
    return o;
}

inline DraftWs draft_ws(void* workspace, int B, int gamma, size_t* clear_bytes) {
    size_t ob, ow, op, oy;
    draft_ws_layout(B, gamma, &ob, &ow, &op, &oy);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    *clear_bytes = op;
    return DraftWs{reinterpret_cast<StatusBlock*>(wsb), reinterpret_cast<unsigned long long*>(wsb + ow),
                   reinterpret_cast<float2*>(wsb + op), reinterpret_cast<float*>(wsb + oy),
                   reinterpret_cast<unsigned int*>(wsb + ob)};
}

namespace {

// ==================================================== CUDA-core phase ====
constexpr int kSimtThreads = 256;

// Position k of request b (blockIdx.y), chunk blockIdx.x of the vocabulary's
// 64-token blocks: y = (U_k + W2 . e) * cscale per token (e = W1[x_{k-1}] or
// the head's row), the chunk's (max, sum) of 2^y and its Gumbel-max winner
// (key y_v - log2 E_v, stream 0; greedy: the largest y).  Lane l of a warp
// takes tokens 64 blk + 2 l and + 1 of each block the warp visits.
template <bool kBF16>
__global__ void __launch_bounds__(kSimtThreads)
draft_phase_simt(int B, int gamma, int V, int r, int k, const void* __restrict__ U,
                 const void* __restrict__ W1, const void* __restrict__ E, const void* __restrict__ W2,
                 const int32_t* __restrict__ x0,
                 const int32_t* __restrict__ x, float cscale, int greedy, uint64_t seed, int nchunk,
                 DraftWs ws) {
    __shared__ float e[256];
    __shared__ float rk[kSimtThreads / 32], rm[kSimtThreads / 32], rs[kSimtThreads / 32], ry[kSimtThreads / 32];
    __shared__ int ri[kSimtThreads / 32];
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
    const void* erow = eng::bias_row<kBF16>(E, W1, b, gamma, k, r, prev);
    for (int j = threadIdx.x; j < r; j += blockDim.x) e[j] = ld_elem<kBF16>(erow, j);
    __syncthreads();
    const int nblk = (V + 63) / 64;
    const int lo = static_cast<int>(static_cast<long long>(chunk) * nblk / nchunk);
    const int hi = static_cast<int>(static_cast<long long>(chunk + 1) * nblk / nchunk);
    const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
    const PhiloxRow pr = philox_row_setup(seed, static_cast<uint32_t>(k), static_cast<uint32_t>(b), kStreamDraftToken);
    Best best{-INFINITY, 0x7FFFFFFF, 0.f};
    float M = -INFINITY, S = 0.f;
    for (int blk = lo + warp; blk < hi; blk += kSimtThreads / 32) {
        const int v = blk * 64 + 2 * lane;
        float y[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (v + h < V) {
                float acc = 0.f;
                for (int j = 0; j < r; ++j)
                    acc = fmaf(ld_elem<kBF16>(W2, static_cast<size_t>(v + h) * r + j), e[j], acc);
                y[h] = (ld_elem<kBF16>(U, urow + v + h) + acc) * cscale;
            } else {
                y[h] = -INFINITY;
            }
        }
        if (greedy) {
#pragma unroll
            for (int h = 0; h < 2; ++h) best_take(best, y[h], v + h, y[h]);
        } else {
            const float mb = warp_max(fmaxf(y[0], y[1]));
            const float sb = warp_sum(fast_exp2(y[0] - mb) + fast_exp2(y[1] - mb));
            lse_merge(M, S, mb, sb);
            // the two tokens share a Philox block (v is even): words (v & 3) and (v & 3) + 1
            const U4 pw = philox_row(pr, static_cast<uint32_t>(v) >> 2);
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (y[h] > -INFINITY)
                    best_take(best, y[h] - fast_log2(exp_draw(u4_word(pw, (v + h) & 3))), v + h, y[h]);
        }
    }
    // warp: best (lowest index on ties)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, best.key, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best.idx, o);
        const float oy = __shfl_xor_sync(0xffffffffu, best.y, o);
        best_take(best, ok, oi, oy);
    }
    if (lane == 0) { rk[warp] = best.key; ri[warp] = best.idx; ry[warp] = best.y; rm[warp] = M; rs[warp] = S; }
    __syncthreads();
    if (threadIdx.x == 0) {
        Best cb{-INFINITY, 0x7FFFFFFF, 0.f};
        float m = -INFINITY, s = 0.f;
        for (int w = 0; w < kSimtThreads / 32; ++w) {
            best_take(cb, rk[w], ri[w], ry[w]);
            lse_merge(m, s, rm[w], rs[w]);
        }
        const size_t slot = static_cast<size_t>(k - 1) * B + b;
        if (!greedy) {
            ws.part[slot * kMaxChunks + chunk] = make_float2(m, s);
            ws.ybest[slot * kMaxChunks + chunk] = cb.y;
        }
        if (cb.key > -INFINITY) atomicMax(&ws.words[slot], pack_key(cb.key, static_cast<uint32_t>(cb.idx)));
    }
}

// ============================================================ winner ====
// x_k of every request: the token of its published winner.
__global__ void __launch_bounds__(256)
draft_winner(int B, int gamma, int V, int k, int32_t* __restrict__ x, DraftWs ws) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const unsigned long long word = ws.words[static_cast<size_t>(k - 1) * B + b];
    const uint32_t idx = unpack_idx(word);
    int tok = static_cast<int>(idx);
    if (word == 0ull || idx >= static_cast<uint32_t>(V)) {   // never produced by the phase kernels
        set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, word == 0ull ? 3 : 8);
        tok = 0;
    }
    x[b * gamma + k - 1] = tok;
}

// ========================================================== finalize ====
// One CTA per request, one warp per position k (eng::finalize_position: lse_d,
// logp_d and the confidence c_k); thread 0 then forms the float32 survival
// product in k order.  Used by the per-position path; the cooperative launch
// does the same work in its tail.  unit / nunits: the tokens per unit and the
// units that the nchunk chunks of the phase launches split.
template <bool kBF16>
__global__ void __launch_bounds__(1024, 1)
draft_finalize(int B, int gamma, int V, int H, int r, const void* __restrict__ h, const void* __restrict__ W1,
               const void* __restrict__ w, float bias, const int32_t* __restrict__ x0,
               const int32_t* __restrict__ x, int greedy, int nchunk, int unit, int nunits,
               float* __restrict__ lse_d, float* __restrict__ logp_d, float* __restrict__ c, float* __restrict__ a,
               DraftWs ws) {
    const int warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    const int k = warp + 1;
    if (k <= gamma)
        eng::finalize_position<kBF16>(b, k, B, gamma, V, H, r, h, W1, w, bias, x0, x, greedy, nchunk, unit, nunits,
                                      ws.part, ws.ybest, lse_d, logp_d, c, ws.status);
    __syncthreads();
    if (threadIdx.x == 0) {
        float surv = 1.f;
        for (int kk = 0; kk < gamma; ++kk) {
            const size_t o = static_cast<size_t>(b) * gamma + kk;
            surv = surv * c[o];
            a[o] = surv;
        }
    }
}

// ============================================================= heads ====
// Gated and recurrent heads (section 3.2, markov_head.py): the rank-r row e_k
// behind position k's bias, written to E [B][gamma][r] before that position's
// phase launch.  The h_k columns of Wg (and Wc) do not depend on the drawn
// tokens, so their products with every h_k are formed once up front.
struct HeadCtx {
    int kind;                        // dspark_head_kind_t
    const void* Wg;
    const void* Wc;
    void* E;                         // [B][gamma][r] in the call's dtype
    float* hg;                       // [kHpSplits][B * gamma][r]: split-K partials of Wg's h columns . h_k
    float* hc;                       // [kHpSplits][B * gamma][r]: the same for Wc (RNN)
    float* state;                    // [B][r]: the RNN state s_{k-1}
};

constexpr int kHpTile = 64, kHpK = 32;   // 64 x 64 outputs per CTA, K in steps of 32
constexpr int kHpSplits = 10;            // split-K partials, summed in order by head_step

// Loads 8 consecutive elements (a 16-byte bf16 group when vec) as floats; elements
// at or past `n` read as 0.
template <bool kBF16>
__device__ __forceinline__ void load8(const void* base, size_t i, int n, bool vec, float* o) {
    if (kBF16 && vec && n >= 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
        o[0] = bf16lo(v.x); o[1] = bf16hi(v.x); o[2] = bf16lo(v.y); o[3] = bf16hi(v.y);
        o[4] = bf16lo(v.z); o[5] = bf16hi(v.z); o[6] = bf16lo(v.w); o[7] = bf16hi(v.w);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (e < n) ? ld_elem<kBF16>(base, i + e) : 0.f;
    }
}

// part[split][m][j] = sum over this split's i of h[m][i] W[j][col + i], m < M, j < r
// (W rows of ldw elements).  Each thread owns 4 x 4 outputs; every output sums its
// i in order, and head_step adds the splits in order.
template <bool kBF16>
__global__ void __launch_bounds__(256)
head_hproj(int M, int H, int r, int ldw, int col, int vec, const void* __restrict__ h, const void* __restrict__ W,
           float* __restrict__ part) {
    __shared__ __align__(16) float As[kHpK][kHpTile];
    __shared__ __align__(16) float Bs[kHpK][kHpTile];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.x * kHpTile, j0 = blockIdx.y * kHpTile, split = blockIdx.z;
    const int nk = (H + kHpK - 1) / kHpK;
    const int c0 = split * nk / kHpSplits, c1 = (split + 1) * nk / kHpSplits;
    const int ty = tid >> 4, tx = tid & 15;
    const int lr = tid >> 2, lk = (tid & 3) * 8;       // loader: row lr of the tile, k offset lk
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int m = m0 + lr, j = j0 + lr;
    // chunk c's operands, loaded one chunk ahead of their use
    auto fetch = [&](int c, float* va, float* vb) {
        const int i0 = c * kHpK + lk;
        const int n = H - i0;
        if (c < c1 && m < M) load8<kBF16>(h, static_cast<size_t>(m) * H + i0, n, vec, va);
        else for (int e = 0; e < 8; ++e) va[e] = 0.f;
        if (c < c1 && j < r) load8<kBF16>(W, static_cast<size_t>(j) * ldw + col + i0, n, vec, vb);
        else for (int e = 0; e < 8; ++e) vb[e] = 0.f;
    };
    float va[8], vb[8];
    fetch(c0, va, vb);
    for (int c = c0; c < c1; ++c) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            As[lk + e][lr] = va[e];
            Bs[lk + e][lr] = vb[e];
        }
        __syncthreads();
        fetch(c + 1, va, vb);
#pragma unroll 8
        for (int kk = 0; kk < kHpK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][4 * ty]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(av[i], bv[jj], acc[i][jj]);
        }
        __syncthreads();
    }
    float* out = part + static_cast<size_t>(split) * M * r;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int m = m0 + 4 * ty + i, j = j0 + 4 * tx + jj;
            if (m < M && j < r) out[static_cast<size_t>(m) * r + j] = acc[i][jj];
        }
}

constexpr int kStepThreads = 512;

// e_k of every request (one CTA each, one warp per output row of Wg / Wc):
//   gated  e = sigmoid(hg + Wg[:, H:H+r] . W1[x_{k-1}]) * W1[x_{k-1}]
//   RNN    g = sigmoid(hg + Wg[:, 0:r] . s + Wg[:, r:2r] . W1[x_{k-1}]),
//          s' = g * s + (1 - g) * tanh(hc + Wc[:, 0:r] . s + Wc[:, r:2r] . W1[x_{k-1}]), e = s'
// with s = s_{k-1} (0 at k = 1) and hg, hc the sums of the split-K partials (in
// split order); e rounded to the dtype into E.
template <bool kBF16>
__global__ void __launch_bounds__(kStepThreads)
head_step(int kind, int B, int gamma, int V, int H, int r, int k, int vec, const void* __restrict__ W1,
          const void* __restrict__ Wg, const void* __restrict__ Wc, const int32_t* __restrict__ x0,
          const int32_t* __restrict__ x, const float* __restrict__ hg, const float* __restrict__ hc,
          float* __restrict__ state, void* __restrict__ E, StatusBlock* st) {
    __shared__ float xr[256], sv[256], pg[256], pc[256], hsum[256], csum[256];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarpsS = kStepThreads / 32;
    const bool rnn = (kind == DSPARK_HEAD_RNN);
    const int prev = prev_token(x0, x, b, gamma, k, V, st);
    const size_t row = static_cast<size_t>(b) * gamma + (k - 1);
    const size_t M = static_cast<size_t>(B) * gamma;
    for (int j = tid; j < r; j += kStepThreads) {
        xr[j] = ld_elem<kBF16>(W1, static_cast<size_t>(prev) * r + j);
        sv[j] = (rnn && k > 1) ? state[static_cast<size_t>(b) * r + j] : 0.f;
        // the h_k products: the split-K partials summed in split order
        float hs = 0.f, cs = 0.f;
        for (int p = 0; p < kHpSplits; ++p) {
            hs += hg[(p * M + row) * r + j];
            if (rnn) cs += hc[(p * M + row) * r + j];
        }
        hsum[j] = hs;
        csum[j] = cs;
    }
    __syncthreads();
    const size_t ldw = rnn ? static_cast<size_t>(2 * r + H) : static_cast<size_t>(H + r);
    if (!rnn) {
        // rows j = warp + 16 i, their loads issued together; each lane takes elements
        // g = 8 lane + 256 t of a row, t < ceil(r / 256)
        constexpr int kRows = 4;
        for (int j0 = warp; j0 < r; j0 += kWarpsS * kRows) {
            float acc[kRows];
#pragma unroll
            for (int q = 0; q < kRows; ++q) acc[q] = 0.f;
            for (int g = lane * 8; g < r; g += 256) {
                float w8[kRows][8];
#pragma unroll
                for (int q = 0; q < kRows; ++q) {
                    const int j = j0 + q * kWarpsS;
                    if (j < r) load8<kBF16>(Wg, static_cast<size_t>(j) * ldw + H + g, r - g, vec, w8[q]);
                }
#pragma unroll
                for (int q = 0; q < kRows; ++q)
                    if (j0 + q * kWarpsS < r)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[q] = fmaf(w8[q][e], (g + e < r) ? xr[g + e] : 0.f, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const int j = j0 + q * kWarpsS;
                const float ag = warp_sum(acc[q]);
                if (lane == 0 && j < r) pg[j] = ag + hsum[j];
            }
        }
    }
    if (rnn) {
        // rows j = warp + 16 i, two at a time: the four segments of each (Wg and Wc over
        // s and over the W1 row) loaded together
        constexpr int kRows = 2;
        for (int j0 = warp; j0 < r; j0 += kWarpsS * kRows) {
            float ag[kRows], ac[kRows];
#pragma unroll
            for (int q = 0; q < kRows; ++q) ag[q] = ac[q] = 0.f;
            for (int g = lane * 8; g < r; g += 256) {
                float w8[kRows][4][8];
#pragma unroll
                for (int q = 0; q < kRows; ++q) {
                    const int j = j0 + q * kWarpsS;
                    if (j < r) {
                        const size_t wr = static_cast<size_t>(j) * ldw;
                        load8<kBF16>(Wg, wr + g, r - g, vec, w8[q][0]);
                        load8<kBF16>(Wg, wr + r + g, r - g, vec, w8[q][1]);
                        load8<kBF16>(Wc, wr + g, r - g, vec, w8[q][2]);
                        load8<kBF16>(Wc, wr + r + g, r - g, vec, w8[q][3]);
                    }
                }
#pragma unroll
                for (int q = 0; q < kRows; ++q)
                    if (j0 + q * kWarpsS < r)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float s_ = (g + e < r) ? sv[g + e] : 0.f, x_ = (g + e < r) ? xr[g + e] : 0.f;
                            ag[q] = fmaf(w8[q][1][e], x_, fmaf(w8[q][0][e], s_, ag[q]));
                            ac[q] = fmaf(w8[q][3][e], x_, fmaf(w8[q][2][e], s_, ac[q]));
                        }
            }
#pragma unroll
            for (int q = 0; q < kRows; ++q) {
                const int j = j0 + q * kWarpsS;
                const float a1 = warp_sum(ag[q]), a2 = warp_sum(ac[q]);
                if (lane == 0 && j < r) {
                    pg[j] = a1 + hsum[j];
                    pc[j] = a2 + csum[j];
                }
            }
        }
    }
    __syncthreads();
    for (int j = tid; j < r; j += kStepThreads) {
        const float g = 1.f / (1.f + expf(-pg[j]));
        float e;
        if (!rnn) {
            e = g * xr[j];
        } else {
            e = g * sv[j] + (1.f - g) * tanhf(pc[j]);
            state[static_cast<size_t>(b) * r + j] = e;
        }
        if constexpr (kBF16)
            static_cast<uint16_t*>(E)[row * r + j] = __bfloat16_as_ushort(__float2bfloat16_rn(e));
        else
            static_cast<float*>(E)[row * r + j] = e;
    }
}

template <bool kBF16>
dspark_status_t launch_hproj(int M, int H, int r, int ldw, int col, int vec, const void* h, const void* W,
                             float* part, cudaStream_t s) {
    const dim3 grid((M + kHpTile - 1) / kHpTile, (r + kHpTile - 1) / kHpTile, kHpSplits);
    head_hproj<kBF16><<<grid, 256, 0, s>>>(M, H, r, ldw, col, vec, h, W, part);
    return launch_status();
}

// ====================================================== host launch ====
// Phase-launch timing hook (see dspark_debug.h).
struct PhaseTiming {
    bool on = false;
    int recorded = 0;
    cudaEvent_t ev[2 * DSPARK_MAX_GAMMA] = {};
};
PhaseTiming g_timing;

int simt_chunks(int V) {
    const int nblk = (V + 63) / 64;
    int n = (nblk + 7) / 8;
    if (n > kMaxChunks) n = kMaxChunks;
    return n < 1 ? 1 : n;
}

bool g_force_phase_launches = false;
// 0: choose by batch size; 1: always the tensor-core path; 2: the CUDA-core GEMV
// path wherever it applies (test hook)
int g_draft_path = 0;
// Up to this many requests the bf16 Markov-head draft runs on the small-batch
// GEMV path.  Measured on the Qwen3 shape (V 151936, r 256, gamma 7, T 0.7):
//   B            1     4     8     9    12    16
//   GEMV path  118   131   147   168   184   206 us
//   tcgen05    151   153   155   155   156   159 us
constexpr int kGemvMaxBatch = 8;

dspark_status_t launch_winner(int B, int gamma, int V, int k, int32_t* x, DraftWs ws, cudaStream_t s) {
    draft_winner<<<(B + 255) / 256, 256, 0, s>>>(B, gamma, V, k, x, ws);
    return launch_status();
}

}  // namespace

// Full draft block on `s`.
// hd: a gated or recurrent head (null: the Markov head).
dspark_status_t draft_block_impl(int B, int gamma, int V, int H, int r, dspark_dtype_t dt, const void* U,
                                 const void* h, const void* W1, const void* W2, const void* w, float bias,
                                 const int32_t* x0, float temperature, uint64_t seed, int32_t* x, float* lse_d,
                                 float* logp_d, float* c, float* a, void* workspace, cudaStream_t s,
                                 const HeadCtx* hd) {
    size_t clear = 0;
    const DraftWs ws = draft_ws(workspace, B, gamma, &clear);
    if (cudaMemsetAsync(workspace, 0, clear, s) != cudaSuccess) return DSPARK_ERR_CUDA;   // status .. words
    const int greedy = (temperature == 0.f);
    const float cscale = greedy ? 1.f : kLog2e / temperature;
    const bool tcp = eng::use_tc_path(dt, r);
    const bool bf = (dt == DSPARK_BF16);
    const void* E = hd ? hd->E : nullptr;
    // 16-byte loads of h and of the head's weight rows (bf16) when every row segment is aligned
    const int hd_vec = hd && bf && H % 8 == 0 && r % 8 == 0 && aligned16(h) && aligned16(hd->Wg) &&
                       (hd->Wc == nullptr || aligned16(hd->Wc));
    if (hd) {
        // the h_k products of the head's gate (and candidate) matrices, once
        const int M = B * gamma;
        const bool rnn = hd->kind == DSPARK_HEAD_RNN;
        const int ldw = rnn ? 2 * r + H : H + r, col = rnn ? 2 * r : 0;
        dspark_status_t st = bf ? launch_hproj<true>(M, H, r, ldw, col, hd_vec, h, hd->Wg, hd->hg, s)
                                : launch_hproj<false>(M, H, r, ldw, col, hd_vec, h, hd->Wg, hd->hg, s);
        if (st == DSPARK_OK && rnn)
            st = bf ? launch_hproj<true>(M, H, r, ldw, col, hd_vec, h, hd->Wc, hd->hc, s)
                    : launch_hproj<false>(M, H, r, ldw, col, hd_vec, h, hd->Wc, hd->hc, s);
        if (st != DSPARK_OK) return st;
    }
    const bool gemv_ok = tcp && !hd && gemv::supported(dt, B, r);
    if (gemv_ok && (g_draft_path == 2 || (g_draft_path == 0 && B <= kGemvMaxBatch))) {
        // every position, x_gamma and the finalize in one cooperative launch
        gemv::Params gp{};
        gp.B = B; gp.gamma = gamma; gp.V = V; gp.H = H; gp.r = r;
        gp.U = static_cast<const uint16_t*>(U); gp.W1 = static_cast<const uint16_t*>(W1);
        gp.W2 = static_cast<const uint16_t*>(W2); gp.h = static_cast<const uint16_t*>(h);
        gp.w = static_cast<const uint16_t*>(w); gp.bias = bias; gp.x0 = x0; gp.x = x;
        gp.cscale = cscale; gp.greedy = greedy; gp.seed = seed; gp.keys = philox_keys(seed);
        gp.lse_d = lse_d; gp.logp_d = logp_d; gp.c = c; gp.a = a; gp.ws = ws;
        if (g_timing.on) cudaEventRecord(g_timing.ev[0], s);
        const dspark_status_t stg = gemv::launch(gp, gemv::grid_for(V), in_host_memory(U), s);
        if (g_timing.on) {
            cudaEventRecord(g_timing.ev[1], s);
            g_timing.recorded = 1;
        }
        return stg;
    }
    if (g_draft_path == 2) return DSPARK_ERR_UNSUPPORTED;
    CUtensorMap map;
    int nM = 1, P = 1, nchunk = 1;
    eng::TcParams p{};
    if (tcp) {
        if (!eng::encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
        eng::tc_grid(B, V, &nM, &P);
        nchunk = P;
        p.B = B; p.gamma = gamma; p.V = V; p.r = r;
        p.U = static_cast<const uint16_t*>(U); p.W1 = static_cast<const uint16_t*>(W1);
        p.E = static_cast<const uint16_t*>(E);
        p.W2 = static_cast<const uint16_t*>(W2);
        p.x0 = x0; p.x = x; p.cscale = cscale; p.greedy = greedy; p.seed = seed; p.keys = philox_keys(seed);
        p.P = P; p.ws = ws;
    } else {
        nchunk = simt_chunks(V);
    }
    // a head kernel runs between positions: one launch per position
    const bool one_launch = tcp && !hd && !g_force_phase_launches && nM * P <= sm_count(current_device());
    dspark_status_t stt = DSPARK_OK;
    if (one_launch) {
        // every position, x_gamma and the finalize in one cooperative launch
        if (g_timing.on) cudaEventRecord(g_timing.ev[0], s);
        p.k = 1;
        p.k_last = gamma;
        p.fuse_tail = 1;
        p.H = H; p.h = static_cast<const uint16_t*>(h); p.w = static_cast<const uint16_t*>(w); p.bias = bias;
        p.lse_d = lse_d; p.logp_d = logp_d; p.c = c; p.a = a;
        stt = eng::launch_tc<eng::kDraft>(map, p, nM * P, s, /*cooperative=*/true);
        if (g_timing.on) {
            cudaEventRecord(g_timing.ev[1], s);
            g_timing.recorded = 1;
        }
        return stt;
    } else {
        for (int k = 1; k <= gamma; ++k) {
            if (hd) {
                if (bf)
                    head_step<true><<<B, kStepThreads, 0, s>>>(hd->kind, B, gamma, V, H, r, k, hd_vec, W1, hd->Wg,
                                                               hd->Wc, x0, x, hd->hg, hd->hc, hd->state, hd->E,
                                                               ws.status);
                else
                    head_step<false><<<B, kStepThreads, 0, s>>>(hd->kind, B, gamma, V, H, r, k, hd_vec, W1, hd->Wg,
                                                                hd->Wc, x0, x, hd->hg, hd->hc, hd->state, hd->E,
                                                                ws.status);
                if ((stt = launch_status()) != DSPARK_OK) return stt;
            }
            if (g_timing.on) cudaEventRecord(g_timing.ev[2 * (k - 1)], s);
            if (tcp) {
                p.k = p.k_last = k;
                stt = eng::launch_tc<eng::kDraft>(map, p, nM * P, s, false);
            } else {
                dim3 grid(nchunk, B);
                if (bf)
                    draft_phase_simt<true><<<grid, kSimtThreads, 0, s>>>(B, gamma, V, r, k, U, W1, E, W2, x0, x,
                                                                         cscale, greedy, seed, nchunk, ws);
                else
                    draft_phase_simt<false><<<grid, kSimtThreads, 0, s>>>(B, gamma, V, r, k, U, W1, E, W2, x0, x,
                                                                          cscale, greedy, seed, nchunk, ws);
                stt = launch_status();
            }
            if (g_timing.on) {
                cudaEventRecord(g_timing.ev[2 * (k - 1) + 1], s);
                g_timing.recorded = k;
            }
            if (stt != DSPARK_OK) return stt;
            stt = launch_winner(B, gamma, V, k, x, ws, s);
            if (stt != DSPARK_OK) return stt;
        }
    }
    const int fthreads = 32 * gamma;
    // the chunks of the phase launches: P ranges of 128-token tiles (tensor cores) or
    // nchunk ranges of 64-token blocks (CUDA cores)
    const int unit = tcp ? eng::kBN : 64;
    const int nunits = (V + unit - 1) / unit;
    if (bf)
        draft_finalize<true><<<B, fthreads, 0, s>>>(B, gamma, V, H, r, h, W1, w, bias, x0, x, greedy, nchunk, unit,
                                                     nunits, lse_d, logp_d, c, a, ws);
    else
        draft_finalize<false><<<B, fthreads, 0, s>>>(B, gamma, V, H, r, h, W1, w, bias, x0, x, greedy, nchunk, unit,
                                                      nunits, lse_d, logp_d, c, a, ws);
    return launch_status();
}

// Debug: z = (U_k + W2 . W1[prev]) for one phase through the tcgen05 path,
// written as float [B][V].  `prev` plays the role of x0 (k = 1).
dspark_status_t debug_tc_logits(int B, int V, int r, const void* U, const void* W1, const void* W2,
                                const int32_t* prev, float* z, void* workspace, cudaStream_t s) {
    if (!eng::use_tc_path(DSPARK_BF16, r)) return DSPARK_ERR_UNSUPPORTED;
    CUtensorMap map;
    if (!eng::encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
    int nM, P;
    eng::tc_grid(B, V, &nM, &P);
    size_t clear = 0;
    const DraftWs ws = draft_ws(workspace, B, 1, &clear);
    if (cudaMemsetAsync(workspace, 0, clear, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    eng::TcParams p{};
    p.B = B; p.gamma = 1; p.V = V; p.r = r; p.k = 1; p.k_last = 1;
    p.U = static_cast<const uint16_t*>(U); p.W1 = static_cast<const uint16_t*>(W1);
    p.W2 = static_cast<const uint16_t*>(W2);
    p.x0 = prev; p.x = nullptr; p.cscale = 1.f; p.greedy = 1; p.seed = 0; p.keys = philox_keys(0);
    p.P = P; p.ws = ws; p.debug_z = z;
    return eng::launch_tc<eng::kDraft>(map, p, nM * P, s, false);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_draft_block_workspace_size(int B, int gamma, int V, int r) {
    (void)r;
    (void)V;
    if (B <= 0 || gamma <= 0 || V <= 0) return kStatusBytes;
    size_t ob, ow, op, oy;
    return draft_ws_layout(B, gamma, &ob, &ow, &op, &oy);
}

dspark_status_t dspark::draft_block_entry(int B, int gamma, int V, int H, int r, dspark_dtype_t dt, const void* U,
                                          const void* h, const void* W1, const void* W2, const void* w, float bias,
                                          const int32_t* x0, float temperature, uint64_t seed, int32_t* x,
                                          float* lse_d, float* logp_d, float* c, float* a, void* workspace,
                                          size_t workspace_bytes, dspark_stream_t stream, bool stage) {
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
    clear_stale_error();
    // the per-call inputs U, h and x0 may be in registered host memory.  U and h are
    // copied to the device first, each in one copy-engine transfer (the host link's
    // full rate); where that is not possible (stream capture) and for x0, the kernels
    // read them through the mapping's device address, each byte once, over the link
    const void* U_in = U;
    const void* h_in = h;
    if (!device_view(U, &U) || (H > 0 && !device_view(h, &h))) return DSPARK_ERR_INVALID_ARGUMENT;
    {
        const void* v = x0;
        if (!device_view(v, &v)) return DSPARK_ERR_INVALID_ARGUMENT;
        x0 = static_cast<const int32_t*>(v);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t esz = dt == DSPARK_BF16 ? 2 : 4;
    void* sU = stage && in_host_memory(U_in)
                   ? stage_to_device(U_in, static_cast<size_t>(B) * gamma * V * esz, s) : nullptr;
    void* sh = stage && H > 0 && in_host_memory(h_in)
                   ? stage_to_device(h_in, static_cast<size_t>(B) * gamma * H * esz, s) : nullptr;
    const dspark_status_t st = draft_block_impl(B, gamma, V, H, r, dt, sU ? sU : U, sh ? sh : h, W1, W2, w, bias,
                                                x0, temperature, seed, x, lse_d, logp_d, c, a, workspace, s, nullptr);
    stage_release(sU, s);
    stage_release(sh, s);
    return st;
}

extern "C" dspark_status_t dspark_draft_block(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                              const void* U, const void* h, const void* W1, const void* W2,
                                              const void* w, float bias, const int32_t* x0, float temperature,
                                              uint64_t seed, int32_t* x, float* lse_d, float* logp_d, float* c,
                                              float* a, void* workspace, size_t workspace_bytes,
                                              dspark_stream_t stream) {
    return draft_block_entry(B, gamma, V, H, r, dt, U, h, W1, W2, w, bias, x0, temperature, seed, x, lse_d, logp_d,
                             c, a, workspace, workspace_bytes, stream, /*stage=*/true);
}

// Workspace of dspark_draft_block_ex: dspark_draft_block's, then (gated, RNN) the
// split-K partials of the h_k products of Wg [splits][B gamma][r] float, and (RNN)
// those of Wc and the state [B][r].
static size_t draft_ex_layout(int B, int gamma, int V, int r, int kind, size_t* o_hg, size_t* o_hc, size_t* o_st) {
    size_t o = round_up(dspark_draft_block_workspace_size(B, gamma, V, r), 256);
    const size_t rows = static_cast<size_t>(kHpSplits) * B * gamma * r * 4;
    *o_hg = *o_hc = *o_st = 0;
    if (kind == DSPARK_HEAD_GATED || kind == DSPARK_HEAD_RNN) {
        *o_hg = o;
        o += round_up(rows, 256);
    }
    if (kind == DSPARK_HEAD_RNN) {
        *o_hc = o;
        o += round_up(rows, 256);
        *o_st = o;
        o += round_up(static_cast<size_t>(B) * r * 4, 256);
    }
    return o;
}

extern "C" size_t dspark_draft_block_ex_workspace_size(int B, int gamma, int V, int r, int kind) {
    if (B <= 0 || gamma <= 0 || V <= 0 || r <= 0) return kStatusBytes;
    size_t a, b, c;
    return draft_ex_layout(B, gamma, V, r, kind, &a, &b, &c);
}

extern "C" dspark_status_t dspark_draft_block_ex(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                                 const void* U, const void* h, const void* W1, const void* W2,
                                                 const void* w, float bias, const int32_t* x0, float temperature,
                                                 uint64_t seed, const dspark_head_t* head, int32_t* x, float* lse_d,
                                                 float* logp_d, float* c, float* a, void* workspace,
                                                 size_t workspace_bytes, dspark_stream_t stream) {
    const int kind = head ? head->kind : DSPARK_HEAD_MARKOV;
    if (kind == DSPARK_HEAD_MARKOV)
        return dspark_draft_block(B, gamma, V, H, r, dt, U, h, W1, W2, w, bias, x0, temperature, seed, x, lse_d,
                                  logp_d, c, a, workspace, workspace_bytes, stream);
    if (kind != DSPARK_HEAD_GATED && kind != DSPARK_HEAD_RNN) return DSPARK_ERR_INVALID_ARGUMENT;
    if (B <= 0 || B > 65535 || gamma <= 0 || gamma > DSPARK_MAX_GAMMA || V <= 0 || H <= 0 || r <= 0 || r > 256)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (dt != DSPARK_F32 && dt != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!(temperature >= 0.f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0 || r % 8 != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!U || !h || !W1 || !W2 || !w || !x0 || !x || !lse_d || !logp_d || !c || !a) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!head->Wg || !head->E || (kind == DSPARK_HEAD_RNN && !head->Wc)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!aligned16(U) || !aligned16(W1) || !aligned16(W2) || !aligned16(head->E)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    size_t ohg, ohc, ost;
    if (workspace_bytes < draft_ex_layout(B, gamma, V, r, kind, &ohg, &ohc, &ost))
        return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    clear_stale_error();
    uint8_t* base = static_cast<uint8_t*>(workspace);
    HeadCtx hd{};
    hd.kind = kind;
    hd.Wg = head->Wg;
    hd.Wc = head->Wc;
    hd.E = head->E;
    hd.hg = reinterpret_cast<float*>(base + ohg);
    hd.hc = kind == DSPARK_HEAD_RNN ? reinterpret_cast<float*>(base + ohc) : nullptr;
    hd.state = kind == DSPARK_HEAD_RNN ? reinterpret_cast<float*>(base + ost) : nullptr;
    return draft_block_impl(B, gamma, V, H, r, dt, U, h, W1, W2, w, bias, x0, temperature, seed, x, lse_d, logp_d,
                            c, a, workspace, reinterpret_cast<cudaStream_t>(stream), &hd);
}

extern "C" dspark_status_t dspark_debug_draft_logits(int B, int V, int r, const void* U_k, const void* W1,
                                                     const void* W2, const int32_t* prev, float* z,
                                                     void* workspace, size_t workspace_bytes,
                                                     dspark_stream_t stream) {
    if (B <= 0 || V <= 0 || V % 8 != 0 || r <= 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!U_k || !W1 || !W2 || !prev || !z || !workspace || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_draft_block_workspace_size(B, 1, V, r)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    clear_stale_error();
    return debug_tc_logits(B, V, r, U_k, W1, W2, prev, z, workspace, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" dspark_status_t dspark_debug_enable_phase_timing(int enable) {
    if (enable && g_timing.ev[0] == nullptr) {
        for (auto& e : g_timing.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return DSPARK_ERR_CUDA;
    }
    g_timing.on = enable != 0;
    g_timing.recorded = 0;
    return DSPARK_OK;
}

extern "C" dspark_status_t dspark_debug_set_draft_path(int mode) {
    if (mode < 0 || mode > 2) return DSPARK_ERR_INVALID_ARGUMENT;
    g_draft_path = mode;
    return DSPARK_OK;
}

extern "C" dspark_status_t dspark_debug_force_phase_launches(int enable) {
    g_force_phase_launches = enable != 0;
    return DSPARK_OK;
}

extern "C" int dspark_debug_phase_times(float* ms, int n) {
    if (!g_timing.on || g_timing.recorded == 0 || ms == nullptr) return 0;
    const int m = g_timing.recorded < n ? g_timing.recorded : n;
    if (cudaEventSynchronize(g_timing.ev[2 * (g_timing.recorded - 1) + 1]) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    for (int i = 0; i < m; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_timing.ev[2 * i], g_timing.ev[2 * i + 1]) != cudaSuccess) {
            cudaGetLastError();                           // not timeable: report nothing
            return 0;
        }
        ms[i] = t;
    }
    return m;
}

// ---------------------------------------------------------------- debug ---
namespace dspark {
namespace {
// One thread waits at the grid barrier of the draft workspace for an epoch
// that no CTA arrives at; the bounded wait must give up and report.
__global__ void debug_bounded_wait(const unsigned int* ctr, uint64_t limit_ns, StatusBlock* st) {
    if (threadIdx.x == 0 && !eng::grid_wait(ctr, 1u, limit_ns)) set_status(st, DSPARK_ERR_TIMEOUT, 99);
}
}  // namespace
}  // namespace dspark

extern "C" dspark_status_t dspark_debug_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                                     dspark_stream_t stream) {
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_draft_block_workspace_size(1, 1, 1, 8)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    if (limit_ns == 0 || limit_ns > 100000000ull) return DSPARK_ERR_INVALID_ARGUMENT;   // at most 100 ms
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    size_t clear = 0;
    const DraftWs ws = draft_ws(workspace, 1, 1, &clear);
    if (cudaMemsetAsync(workspace, 0, clear, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    debug_bounded_wait<<<1, 32, 0, s>>>(ws.gbar, limit_ns, ws.status);
    return launch_status();
}
