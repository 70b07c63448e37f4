// dspark_verify: target verification by rejection sampling (DeepSpec
// walkthrough, section 8.2 `verify_draft_tokens`; section 2.1: one bonus token
// when every proposed token is accepted), over the prefix l*_b that the
// scheduler kept (section 3.3, Algorithm 1).
//
//   plan    clears the per-call words and lists the scheduled rows;
//   rows    one pass over every scheduled target row (b, k), k <= l*_b + 1:
//           per 64-token block the logsumexp of t / T and a Gumbel key for a
//           draw from p_t (streams 6 / 5); greedy: the argmax of t;
//   chain   one warp per request: p_t(x_k) / p_d(x_k) against u (stream 1),
//           stop at the first rejection;
//   residual for the rejected rows only: the bias engine in its residual mode
//           (z rebuilt exactly as the draft built it), per block the mass of
//           max(0, p_t - p_d) and a Gumbel key (stream 4);
//   finish  two warps per request: the token inside the winning block --
//           residual (stream 2), or a draw from p_t (stream 5) for the bonus
//           row or a residual without mass.
#include <algorithm>

#include "engine.cuh"

namespace dspark {
namespace {

using eng::ld_elem;
using eng::lse_merge;
using eng::pack_key;
using eng::prev_token;
using eng::unpack_idx;

constexpr int kNchMax = 64;   // row chunks of the target pass

struct VerifyWs {
    StatusBlock* status;
    int32_t* rows;                 // [B][gamma+1] scheduled rows b*(gamma+1)+k-1, compacted in b order
    int32_t* first;                // [B] index of request b's first row in `rows`
    int32_t* plan;                 // [0] N scheduled rows, [1] blocks per rows-pass CTA
    unsigned long long* wt;        // [B][gamma+1] target-row word: draw key (T > 0) or argmax (T = 0)
    float2* part;                  // [B][gamma+1][kNchMax] (max, sum) of t log2e / T
    unsigned long long* res_word;  // [B] residual draw key
    int32_t* krow;                 // [B] rejected position (0: none)
    float* lt2;                    // [B] log2-sum-exp2 of t / T at the rejected row
    float* ld2;                    // [B] lse_d at the rejected row, log2 units
    int32_t* stop;                 // [B] row of the final draw
};

size_t verify_ws_layout(int B, int gamma, size_t* off) {
    size_t o = kStatusBytes;
    const size_t rows = static_cast<size_t>(B) * (gamma + 1);
    off[0] = o; o += round_up(rows * 8, 256);                 // wt
    off[1] = o; o += round_up(static_cast<size_t>(B) * 8, 256);   // res_word
    off[2] = o; o += round_up(rows * kNchMax * 8, 256);       // part
    off[3] = o; o += round_up(static_cast<size_t>(B) * 4, 256);   // krow
    off[4] = o; o += round_up(static_cast<size_t>(B) * 4, 256);   // lt2
    off[5] = o; o += round_up(static_cast<size_t>(B) * 4, 256);   // ld2
    off[6] = o; o += round_up(static_cast<size_t>(B) * 4, 256);   // stop
    off[7] = o; o += round_up(rows * 4, 256);                 // compacted rows
    off[8] = o; o += 256;                                     // plan
    off[9] = o; o += round_up(static_cast<size_t>(B) * 4, 256);   // first
    return o;
}

__device__ __forceinline__ int clamp_ell(const int32_t* ell, int b, int gamma, StatusBlock* st) {
    int e = ell[b];
    if (e < 0 || e > gamma) {
        set_status(st, DSPARK_ERR_DEVICE_CHECK, 4);
        e = e < 0 ? 0 : gamma;
    }
    return e;
}

// The rows pass splits the scheduled rows, each padded to a multiple of 4
// blocks (one Philox counter covers a quad of blocks), into equal contiguous
// ranges of `per` blocks, one range per CTA.  Slot c - first CTA of the row
// of part[row][.] holds the (max, sum) partial of CTA c's piece of the row.
__host__ __device__ __forceinline__ int padded_blocks(int V) { return ((V + 63) / 64 + 3) / 4 * 4; }

// ------------------------------------------------------------- plan pass ---
// One CTA: clears the status block and the per-row and residual words, clamps
// l*_b, writes the scheduled rows (k = 1 .. l*_b + 1 of every request) as a
// compact list with each request's first index, the row count N and the
// blocks per rows-pass CTA, so that no work is launched for rows that were not
// scheduled.
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads)
verify_plan(int B, int gamma, int V, int rows_ctas, const int32_t* __restrict__ ell, VerifyWs ws) {
    __shared__ int wsum[kPlanThreads / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t nrows = static_cast<size_t>(B) * (gamma + 1);
    for (size_t i = tid; i < nrows; i += kPlanThreads) ws.wt[i] = 0ull;
    for (int i = tid; i < B; i += kPlanThreads) ws.res_word[i] = 0ull;
    if (tid < static_cast<int>(kStatusBytes / 4)) reinterpret_cast<uint32_t*>(ws.status)[tid] = 0u;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += kPlanThreads) {
        const int b = base + tid;
        const int e = (b < B) ? clamp_ell(ell, b, gamma, ws.status) : -1;
        const int cnt = e + 1;
        int inc = cnt;                                    // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += v;
            }
            wsum[lane] = w;                               // inclusive over warps
        }
        __syncthreads();
        const int off = carry + (warp > 0 ? wsum[warp - 1] : 0) + inc - cnt;
        if (b < B) ws.first[b] = off;
        for (int j = 0; j < cnt; ++j) ws.rows[off + j] = b * (gamma + 1) + j;
        __syncthreads();
        if (tid == 0) carry += wsum[kPlanThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) {
        const long long total = static_cast<long long>(carry) * padded_blocks(V);
        // equal ranges over the CTAs, a multiple of 4 blocks, and a row split
        // over at most kNchMax CTAs
        long long per = (total + rows_ctas - 1) / rows_ctas;
        per = max(per, static_cast<long long>((padded_blocks(V) + kNchMax - 3) / (kNchMax - 2)));
        per = (per + 3) / 4 * 4;
        ws.plan[0] = carry;
        ws.plan[1] = static_cast<int>(per);
    }
}

// ------------------------------------------------------------- rows pass ---
// CTA c takes blocks [c per, (c+1) per) of the padded scheduled rows laid end
// to end, one piece per row it touches; per piece a warp covers 4 quads of 4
// consecutive blocks per step, 8 lanes per block, 8 logits per lane.  Per
// 64-token block: the logsumexp of t / T and a Gumbel key for a draw from p_t
// (greedy: the argmax of t); per piece the CTA's best and its (max, sum).
// Sixteen lanes finish the 16 blocks of a step, one block each.
constexpr int kRowsCtasPerSm = 4;

template <bool kBF16>
__global__ void __launch_bounds__(256, kRowsCtasPerSm)
verify_rows(int gamma, int V, const void* __restrict__ t, float cscale, int greedy, uint64_t seed, VerifyWs ws) {
    __shared__ float rk[8], rm[8], rs[8];
    __shared__ int ri[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane >> 3, part = lane & 7;
    const int nblk = (V + 63) / 64, npad = padded_blocks(V);
    const int N = ws.plan[0], per = ws.plan[1];
    const long long total = static_cast<long long>(N) * npad;
    const uint64_t pol = policy_evict_first();
    for (long long c = blockIdx.x; c * per < total; c += gridDim.x) {
        long long g = c * per;
        const long long gend = min(total, g + per);
        while (g < gend) {
            const int n = static_cast<int>(g / npad);
            const int lo = static_cast<int>(g - static_cast<long long>(n) * npad);
            const int hi_pad = static_cast<int>(min(static_cast<long long>(npad), lo + (gend - g)));
            const int hi = min(hi_pad, nblk);
            const int slot = static_cast<int>(c - static_cast<long long>(n) * npad / per);
            const int row = ws.rows[n];
            const int b = row / (gamma + 1), k = row % (gamma + 1) + 1;
            const size_t rowoff = static_cast<size_t>(row) * V;
            float best = -INFINITY, M = -INFINITY, S = 0.f;
            int best_i = 0x7FFFFFFF;
            // each warp takes 4 consecutive quads per step; all loads of a step are issued first
            constexpr int kU = 4;
            for (int q0 = lo / 4 + warp * kU; q0 * 4 < hi; q0 += 8 * kU) {
                float y[kU][8];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int blk = (q0 + u) * 4 + sub;
                    const int v = blk * 64 + part * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[u][i] = -INFINITY;
                    if (blk < hi) {
                        if constexpr (kBF16) {
                            if (v < V) {
                                uint32_t w[4];
                                eng::ld_u32x4(static_cast<const uint16_t*>(t) + rowoff + v, w, pol);
#pragma unroll
                                for (int i = 0; i < 4; ++i) { y[u][2 * i] = bf16lo(w[i]); y[u][2 * i + 1] = bf16hi(w[i]); }
                            }
                        } else {
#pragma unroll
                            for (int hq = 0; hq < 2; ++hq) {
                                if (v + 4 * hq < V) {
                                    uint32_t w[4];
                                    eng::ld_u32x4(static_cast<const float*>(t) + rowoff + v + 4 * hq, w, pol);
#pragma unroll
                                    for (int i = 0; i < 4; ++i) y[u][4 * hq + i] = __uint_as_float(w[i]);
                                }
                            }
                        }
                    }
                }
                if (greedy) {
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int v = ((q0 + u) * 4 + sub) * 64 + part * 8;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (y[u][i] > best) { best = y[u][i]; best_i = v + i; }
                    }
                    continue;
                }
                // per block (quad u, sub): max and sum of 2^(y c - m c) over its 8 lanes
                float mq[kU], sq[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    float m = y[u][0];
#pragma unroll
                    for (int i = 1; i < 8; ++i) m = fmaxf(m, y[u][i]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    const float mc = m * cscale;
                    float sum = 0.f;
                    if (m > -INFINITY) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) sum += fast_exp2(fmaf(y[u][i], cscale, -mc));
                    }
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                    mq[u] = mc;
                    sq[u] = sum;
                }
                // lane (sub, part < 4) finishes block (quad q0 + part, sub): its Philox
                // counter is that quad's, its word the block's
                const int pu = part & 3;
                const U4 pw = philox4x32_10(U4{static_cast<uint32_t>(q0 + pu), static_cast<uint32_t>(k),
                                               static_cast<uint32_t>(b), kStreamTargetBlock},
                                            static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
                const uint32_t word = sub == 0 ? pw.x : sub == 1 ? pw.y : sub == 2 ? pw.z : pw.w;
                const float m = pu == 0 ? mq[0] : pu == 1 ? mq[1] : pu == 2 ? mq[2] : mq[3];
                const float sum = pu == 0 ? sq[0] : pu == 1 ? sq[1] : pu == 2 ? sq[2] : sq[3];
                const int blk = (q0 + pu) * 4 + sub;
                if (part < 4 && blk < hi && sum > 0.f) {
                    const float key = (m + log2f(sum)) * kLn2 + gumbel_of(uniform_open(word));
                    if (key > best || (key == best && blk < best_i)) { best = key; best_i = blk; }
                    lse_merge(M, S, m, sum);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
                const float om = __shfl_xor_sync(0xffffffffu, M, o);
                const float os = __shfl_xor_sync(0xffffffffu, S, o);
                if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
                lse_merge(M, S, om, os);
            }
            if (lane == 0) { rk[warp] = best; ri[warp] = best_i; rm[warp] = M; rs[warp] = S; }
            __syncthreads();
            if (threadIdx.x == 0) {
                float bk = -INFINITY, m = -INFINITY, s = 0.f;
                int bi = 0x7FFFFFFF;
                for (int w = 0; w < 8; ++w) {
                    if (rk[w] > bk || (rk[w] == bk && ri[w] < bi)) { bk = rk[w]; bi = ri[w]; }
                    lse_merge(m, s, rm[w], rs[w]);
                }
                if (!greedy) ws.part[static_cast<size_t>(row) * kNchMax + slot] = make_float2(m, s);
                if (bk > -INFINITY) atomicMax(&ws.wt[row], pack_key(bk, static_cast<uint32_t>(bi)));
            }
            __syncthreads();                              // rk..ri are rewritten by the next piece
            g += hi_pad - lo;
        }
    }
}

// ------------------------------------------------------------ chain pass ---
template <bool kBF16>
__global__ void __launch_bounds__(256)
verify_chain(int B, int gamma, int V, const void* __restrict__ t, const int32_t* __restrict__ x,
             const float* __restrict__ lse_d, const float* __restrict__ logp_d, const int32_t* __restrict__ ell,
             float cscale, int greedy, uint64_t seed, int32_t* __restrict__ n_accept,
             int32_t* __restrict__ next_token, VerifyWs ws) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 8 + warp;
    if (b >= B) return;
    const int e = clamp_ell(ell, b, gamma, ws.status);
    const int per = ws.plan[1], npad = padded_blocks(V), n0 = ws.first[b];
    int nacc = 0, rej = 0;
    float rej_lt2 = 0.f;
    for (int k = 1; k <= e; ++k) {
        const int row = b * (gamma + 1) + (k - 1);
        int xk = x[b * gamma + k - 1];
        if (xk < 0 || xk >= V) {
            if (lane == 0) set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 5);
            xk = 0;
        }
        bool ok;
        float Lt2 = 0.f;
        if (greedy) {
            const unsigned long long w = ws.wt[row];
            ok = (w != 0ull) && static_cast<int>(unpack_idx(w)) == xk;
        } else {
            // the rows-pass CTAs that covered this row wrote slots 0 .. c_last - c_first
            const long long g0 = static_cast<long long>(n0 + k - 1) * npad;
            const int nch = static_cast<int>((g0 + npad - 1) / per - g0 / per) + 1;
            float m = -INFINITY, s = 0.f;
            for (int c = lane; c < nch; c += 32) {
                const float2 pr = ws.part[static_cast<size_t>(row) * kNchMax + c];
                lse_merge(m, s, pr.x, pr.y);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float om = __shfl_xor_sync(0xffffffffu, m, o);
                const float os = __shfl_xor_sync(0xffffffffu, s, o);
                lse_merge(m, s, om, os);
            }
            Lt2 = m + log2f(s);
            const float yk = ld_elem<kBF16>(t, static_cast<size_t>(row) * V + xk) * cscale;
            const float ratio = expf((yk - Lt2) * kLn2 - logp_d[b * gamma + k - 1]);
            const float u = uniform_accept(draw_word(seed, b, k, kStreamAccept, 0));
            ok = u < ratio;
        }
        if (ok) {
            ++nacc;
        } else {
            rej = k;
            rej_lt2 = Lt2;
            break;
        }
    }
    if (lane == 0) {
        n_accept[b] = nacc;
        const int srow = nacc + 1;                        // row of the final draw
        ws.stop[b] = srow;
        if (greedy) {
            const unsigned long long w = ws.wt[b * (gamma + 1) + srow - 1];
            if (w == 0ull) set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 6);
            next_token[b] = (w == 0ull || unpack_idx(w) >= static_cast<uint32_t>(V)) ? 0 : static_cast<int>(unpack_idx(w));
            ws.krow[b] = 0;
        } else {
            ws.krow[b] = rej;
            ws.lt2[b] = rej_lt2;
            ws.ld2[b] = rej ? lse_d[b * gamma + rej - 1] * kLog2e : 0.f;
        }
    }
}

// ---------------------------------------------------- residual, CUDA cores ---
template <bool kBF16>
__global__ void __launch_bounds__(256)
residual_simt(int B, int gamma, int V, int r, const void* __restrict__ t, const void* __restrict__ U,
              const void* __restrict__ W1, const void* __restrict__ W2, const int32_t* __restrict__ x0,
              const int32_t* __restrict__ x, float cscale, uint64_t seed, int nchunk, VerifyWs ws) {
    __shared__ float e[256];
    __shared__ float rk[8];
    __shared__ int ri[8];
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int k = ws.krow[b];
    if (k <= 0) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
    for (int j = threadIdx.x; j < r; j += blockDim.x) e[j] = ld_elem<kBF16>(W1, static_cast<size_t>(prev) * r + j);
    __syncthreads();
    const float lt2 = ws.lt2[b], ld2 = ws.ld2[b];
    const int nblk = (V + 63) / 64;
    const int lo = static_cast<int>(static_cast<long long>(chunk) * nblk / nchunk);
    const int hi = static_cast<int>(static_cast<long long>(chunk + 1) * nblk / nchunk);
    const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
    const size_t trow = (static_cast<size_t>(b) * (gamma + 1) + (k - 1)) * V;
    float best = -INFINITY;
    int best_i = 0x7FFFFFFF;
    for (int blk = lo + warp; blk < hi; blk += 8) {
        float qs = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = blk * 64 + h * 32 + lane;
            if (v < V) {
                float acc = 0.f;
                for (int j = 0; j < r; ++j) acc = fmaf(ld_elem<kBF16>(W2, static_cast<size_t>(v) * r + j), e[j], acc);
                const float yd = (ld_elem<kBF16>(U, urow + v) + acc) * cscale;
                const float yt = ld_elem<kBF16>(t, trow + v) * cscale;
                qs += fmaxf(fast_exp2(yt - lt2) - fast_exp2(yd - ld2), 0.f);
            }
        }
        const float Q = warp_sum(qs);
        if (Q > 0.f) {
            const float u = uniform_open(draw_word(seed, b, k, kStreamResidualBlock, static_cast<uint32_t>(blk)));
            const float key = log2f(Q) * kLn2 + gumbel_of(u);
            if (key > best) { best = key; best_i = blk; }   // blocks ascend per warp
        }
    }
    if (lane == 0) { rk[warp] = best; ri[warp] = best_i; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float bk = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int w = 0; w < 8; ++w)
            if (rk[w] > bk || (rk[w] == bk && ri[w] < bi)) { bk = rk[w]; bi = ri[w]; }
        if (bk > -INFINITY) atomicMax(&ws.res_word[b], pack_key(bk, static_cast<uint32_t>(bi)));
    }
}

// ----------------------------------------------------------- finish pass ---
// Two warps per request (T > 0): the token inside the winning block of the
// residual, or of the draw from p_t at the stop row.
template <bool kBF16, int kCPL>
__global__ void __launch_bounds__(64)
verify_finish(int B, int gamma, int V, int r, const void* __restrict__ t, const void* __restrict__ U,
              const void* __restrict__ W1, const void* __restrict__ W2, const int32_t* __restrict__ x0,
              const int32_t* __restrict__ x, float cscale, uint64_t seed, int32_t* __restrict__ next_token,
              VerifyWs ws) {
    __shared__ float sbest[2];
    __shared__ int sidx[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    const int kr = ws.krow[b];
    const unsigned long long rw = (kr > 0) ? ws.res_word[b] : 0ull;
    const uint32_t nblk = static_cast<uint32_t>((V + 63) / 64);
    bool residual = rw != 0ull && unpack_idx(rw) < nblk;
    float score = -INFINITY;
    int v = 0x7FFFFFFF;
    if (residual) {
        const int blk = static_cast<int>(unpack_idx(rw));
        const float z = eng::block_logit<kBF16, kCPL>(b, gamma, kr, V, r, blk, U, W1, W2, x0, x, ws.status);
        v = blk * 64 + warp * 32 + lane;
        if (z > -INFINITY) {
            const float yd = z * cscale;
            const float yt = ld_elem<kBF16>(t, (static_cast<size_t>(b) * (gamma + 1) + (kr - 1)) * V + v) * cscale;
            const float qv = fast_exp2(yt - ws.lt2[b]) - fast_exp2(yd - ws.ld2[b]);
            if (qv > 0.f) {
                const float g = gumbel_of(uniform_open(draw_word(seed, b, kr, kStreamResidualToken, static_cast<uint32_t>(v))));
                score = log2f(qv) * kLn2 + g;
            }
        }
        if (!__syncthreads_or(score > -INFINITY)) residual = false;   // no mass left after rounding
    }
    if (!residual) {
        const int srow = (kr > 0) ? kr : ws.stop[b];
        const unsigned long long w = ws.wt[b * (gamma + 1) + srow - 1];
        if (w == 0ull) {
            if (threadIdx.x == 0) { set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 7); next_token[b] = 0; }
            return;
        }
        if (unpack_idx(w) >= nblk) {
            if (threadIdx.x == 0) { set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 9); next_token[b] = 0; }
            return;
        }
        const int blk = static_cast<int>(unpack_idx(w));
        v = blk * 64 + warp * 32 + lane;
        score = -INFINITY;
        if (v < V) {
            const float yt = ld_elem<kBF16>(t, (static_cast<size_t>(b) * (gamma + 1) + (srow - 1)) * V + v) * cscale;
            const float g = gumbel_of(uniform_open(draw_word(seed, b, srow, kStreamTargetToken, static_cast<uint32_t>(v))));
            score = yt + g * kLog2e;
        }
    }
    int bi = (score > -INFINITY) ? v : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, score, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (os > score || (os == score && oi < bi)) { score = os; bi = oi; }
    }
    if (lane == 0) { sbest[warp] = score; sidx[warp] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        int w = 0;
        if (sbest[1] > sbest[0] || (sbest[1] == sbest[0] && sidx[1] < sidx[0])) w = 1;
        next_token[b] = (sidx[w] == 0x7FFFFFFF) ? 0 : sidx[w];
    }
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_verify_workspace_size(int B, int gamma, int V, int r) {
    (void)V;
    (void)r;
    if (B <= 0 || gamma <= 0) return kStatusBytes;
    size_t off[10];
    return verify_ws_layout(B, gamma, off);
}

extern "C" dspark_status_t dspark_verify(int B, int gamma, int V, int r, dspark_dtype_t dt, const void* t_logits,
                                         const void* U, const void* W1, const void* W2, const int32_t* x0,
                                         const int32_t* x, const float* lse_d, const float* logp_d,
                                         const int32_t* ell, float temperature, uint64_t seed, int32_t* n_accept,
                                         int32_t* next_token, void* workspace, size_t workspace_bytes,
                                         dspark_stream_t stream) {
    if (B <= 0 || gamma <= 0 || gamma > DSPARK_MAX_GAMMA || V <= 0 || r <= 0 || r > 256 || r % 8 != 0)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (static_cast<long long>(B) * (gamma + 1) > 65535) return DSPARK_ERR_UNSUPPORTED;
    if (dt != DSPARK_F32 && dt != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!(temperature >= 0.f) || temperature == INFINITY) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!t_logits || !U || !W1 || !W2 || !x0 || !x || !lse_d || !logp_d || !ell || !n_accept || !next_token)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (!aligned16(t_logits) || !aligned16(U) || !aligned16(W1) || !aligned16(W2)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_verify_workspace_size(B, gamma, V, r)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    size_t off[10];
    verify_ws_layout(B, gamma, off);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    VerifyWs ws{reinterpret_cast<StatusBlock*>(wsb), reinterpret_cast<int32_t*>(wsb + off[7]),
                reinterpret_cast<int32_t*>(wsb + off[9]), reinterpret_cast<int32_t*>(wsb + off[8]), reinterpret_cast<unsigned long long*>(wsb + off[0]),
                reinterpret_cast<float2*>(wsb + off[2]), reinterpret_cast<unsigned long long*>(wsb + off[1]),
                reinterpret_cast<int32_t*>(wsb + off[3]), reinterpret_cast<float*>(wsb + off[4]),
                reinterpret_cast<float*>(wsb + off[5]), reinterpret_cast<int32_t*>(wsb + off[6])};
    const int greedy = (temperature == 0.f);
    const float cscale = greedy ? 1.f : kLog2e / temperature;
    const bool bf = (dt == DSPARK_BF16);
    const int nblk = (V + 63) / 64;
    // persistent rows pass: all resident CTAs
    const int rgrid = kRowsCtasPerSm * sm_count(current_device());
    verify_plan<<<1, kPlanThreads, 0, s>>>(B, gamma, V, rgrid, ell, ws);
    dspark_status_t stt = launch_status();
    if (stt != DSPARK_OK) return stt;
    if (bf) verify_rows<true><<<rgrid, 256, 0, s>>>(gamma, V, t_logits, cscale, greedy, seed, ws);
    else verify_rows<false><<<rgrid, 256, 0, s>>>(gamma, V, t_logits, cscale, greedy, seed, ws);
    if ((stt = launch_status()) != DSPARK_OK) return stt;
    const int cgrid = (B + 7) / 8;
    if (bf)
        verify_chain<true><<<cgrid, 256, 0, s>>>(B, gamma, V, t_logits, x, lse_d, logp_d, ell, cscale, greedy, seed,
                                                 n_accept, next_token, ws);
    else
        verify_chain<false><<<cgrid, 256, 0, s>>>(B, gamma, V, t_logits, x, lse_d, logp_d, ell, cscale, greedy,
                                                  seed, n_accept, next_token, ws);
    if ((stt = launch_status()) != DSPARK_OK || greedy) return stt;

    if (eng::use_tc_path(dt, r)) {
        CUtensorMap map;
        if (!eng::encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
        int nM, P;
        eng::tc_grid(B, V, &nM, &P);
        eng::TcParams p{};
        p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.k = 1;
        p.U = static_cast<const uint16_t*>(U); p.W1 = static_cast<const uint16_t*>(W1);
        p.W2 = static_cast<const uint16_t*>(W2); p.k_last = 1;
        p.x0 = x0; p.x = const_cast<int32_t*>(x); p.cscale = cscale; p.greedy = 0;   // read only here
        p.seed = seed; p.P = P;
        p.ws = eng::Ws{ws.status, ws.res_word, nullptr, nullptr, nullptr, nullptr};
        p.krow = ws.krow; p.T = static_cast<const uint16_t*>(t_logits); p.lt2 = ws.lt2; p.ld2 = ws.ld2;
        if ((stt = eng::launch_tc<eng::kResidual>(map, p, nM * P, s, false)) != DSPARK_OK) return stt;
    } else {
        int nchunk = (nblk + 7) / 8;
        if (nchunk > 256) nchunk = 256;
        const dim3 g(nchunk, B);
        if (bf) residual_simt<true><<<g, 256, 0, s>>>(B, gamma, V, r, t_logits, U, W1, W2, x0, x, cscale, seed, nchunk, ws);
        else residual_simt<false><<<g, 256, 0, s>>>(B, gamma, V, r, t_logits, U, W1, W2, x0, x, cscale, seed, nchunk, ws);
        if ((stt = launch_status()) != DSPARK_OK) return stt;
    }
    if (bf)
        verify_finish<true, 1><<<B, 64, 0, s>>>(B, gamma, V, r, t_logits, U, W1, W2, x0, x, cscale, seed, next_token, ws);
    else if (r <= 128)
        verify_finish<false, 1><<<B, 64, 0, s>>>(B, gamma, V, r, t_logits, U, W1, W2, x0, x, cscale, seed, next_token, ws);
    else
        verify_finish<false, 2><<<B, 64, 0, s>>>(B, gamma, V, r, t_logits, U, W1, W2, x0, x, cscale, seed, next_token, ws);
    return launch_status();
}
