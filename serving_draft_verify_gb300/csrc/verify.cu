// dspark_verify: target verification by rejection sampling (DeepSpec
// walkthrough, section 8.2 `verify_draft_tokens`; section 2.1: one bonus token
// when every proposed token is accepted), over the prefix l*_b that the
// scheduler kept (section 3.3, Algorithm 1).
//
//   plan    clears the per-call words and lists the scheduled rows;
//   rows    one pass over every scheduled target row (b, k), k <= l*_b + 1:
//           rows k <= l*_b: the logsumexp of t / T (for p_t(x_k) and the
//           residual); row l*_b + 1: the Gumbel-max draw from p_t over the
//           vocabulary (stream 2), the bonus token if nothing is rejected;
//           greedy: the argmax of t;
//   decide  by the CTA that completes a row: p_t(x_k) / p_d(x_k) against u
//           (stream 1); by the CTA that completes a request: n_accept, and
//           the bonus token, or the rejected position for the residual;
//   residual for the rejected rows only (listed by the rows pass as it decides
//           them, so the launch's grid covers just those rows): the bias
//           engine in its residual mode (z rebuilt exactly as the draft built
//           it), the Gumbel-max draw from max(0, p_t - p_d) over the
//           vocabulary (stream 2);
//   finish  a rejected request takes the residual's winner, or, if the
//           residual has no mass, a draw from p_t at that row (stream 2).
#include <algorithm>

#include "engine.cuh"

namespace dspark {
namespace {

using eng::Best;
using eng::best_take;
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
    unsigned long long* wt;        // [B][gamma+1] row l*_b + 1: Gumbel-max winner (T > 0); every row: argmax (T = 0)
    float2* part;                  // [B][gamma+1][kNchMax] (max, sum) of t log2e / T
    unsigned long long* res_word;  // [B] residual winner (key, ~token)
    int32_t* krow;                 // [B] rejected position (0: none)
    float* lt2;                    // [B] log2-sum-exp2 of t / T at the rejected row
    float* ld2;                    // [B] lse_d at the rejected row, log2 units
    int32_t* row_cnt;              // [N] rows-pass CTAs done with compacted row n
    int32_t* req_cnt;              // [B] rows of request b whose decision is made
    int32_t* dec;                  // [B][gamma+1] acceptance of x_k at row k (k <= l*_b)
    float* lt2row;                 // [B][gamma+1] log2-sum-exp2 of t / T per decided row
    float* tx;                     // [B][gamma+1] t[b][k][x_k] for k <= l*_b, picked up by the rows pass
    unsigned int* gbar;            // grid barrier of the residual launch
    int32_t* rej_count;            // [1] rejected requests so far
    int32_t* rej_list;             // [B] the rejected requests, in the order their outcomes were decided
};

// Workspace: status | plan | gbar | rej_count | wt | res_word | row_cnt | req_cnt
// (cleared by the plan kernel) | part | krow | lt2 | ld2 | rows | first | dec |
// lt2row | tx | rej_list.
struct VerifyLayout {
    size_t plan, gbar, rej_count, wt, res_word, row_cnt, req_cnt, part, krow, lt2, ld2, rows, first, dec, lt2row, tx,
        rej_list, total;
};

VerifyLayout verify_ws_layout(int B, int gamma) {
    VerifyLayout L{};
    const size_t rows = static_cast<size_t>(B) * (gamma + 1), nb = static_cast<size_t>(B);
    size_t o = kStatusBytes;
    auto take = [&](size_t& off, size_t bytes) { off = o; o += round_up(bytes, 256); };
    take(L.plan, 16);
    take(L.gbar, 16);
    take(L.rej_count, 16);
    take(L.wt, rows * 8);
    take(L.res_word, nb * 8);
    take(L.row_cnt, rows * 4);
    take(L.req_cnt, nb * 4);
    take(L.part, rows * kNchMax * 8);
    take(L.krow, nb * 4);
    take(L.lt2, nb * 4);
    take(L.ld2, nb * 4);
    take(L.rows, rows * 4);
    take(L.first, nb * 4);
    take(L.dec, rows * 4);
    take(L.lt2row, rows * 4);
    take(L.tx, rows * 4);
    take(L.rej_list, nb * 4);
    L.total = o;
    return L;
}

VerifyWs verify_ws(void* workspace, int B, int gamma) {
    const VerifyLayout L = verify_ws_layout(B, gamma);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    VerifyWs ws;
    ws.status = reinterpret_cast<StatusBlock*>(w);
    ws.rows = reinterpret_cast<int32_t*>(w + L.rows);
    ws.first = reinterpret_cast<int32_t*>(w + L.first);
    ws.plan = reinterpret_cast<int32_t*>(w + L.plan);
    ws.wt = reinterpret_cast<unsigned long long*>(w + L.wt);
    ws.part = reinterpret_cast<float2*>(w + L.part);
    ws.res_word = reinterpret_cast<unsigned long long*>(w + L.res_word);
    ws.krow = reinterpret_cast<int32_t*>(w + L.krow);
    ws.lt2 = reinterpret_cast<float*>(w + L.lt2);
    ws.ld2 = reinterpret_cast<float*>(w + L.ld2);
    ws.row_cnt = reinterpret_cast<int32_t*>(w + L.row_cnt);
    ws.req_cnt = reinterpret_cast<int32_t*>(w + L.req_cnt);
    ws.dec = reinterpret_cast<int32_t*>(w + L.dec);
    ws.lt2row = reinterpret_cast<float*>(w + L.lt2row);
    ws.tx = reinterpret_cast<float*>(w + L.tx);
    ws.gbar = reinterpret_cast<unsigned int*>(w + L.gbar);
    ws.rej_count = reinterpret_cast<int32_t*>(w + L.rej_count);
    ws.rej_list = reinterpret_cast<int32_t*>(w + L.rej_list);
    return ws;
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
    for (size_t i = tid; i < nrows; i += kPlanThreads) {
        ws.wt[i] = 0ull;
        ws.row_cnt[i] = 0;
    }
    for (int i = tid; i < B; i += kPlanThreads) {
        ws.res_word[i] = 0ull;
        ws.req_cnt[i] = 0;
    }
    if (tid < static_cast<int>(kStatusBytes / 4)) reinterpret_cast<uint32_t*>(ws.status)[tid] = 0u;
    if (tid == 0) { *ws.gbar = 0u; *ws.rej_count = 0; }
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

// --------------------------------------------------------- row decisions ---
// One warp, run by the rows-pass CTA that finished row (b, k) last: for
// k <= l*_b the acceptance test of x_k (u < p_t(x_k) / p_d(x_k), u from
// stream 1; greedy: x_k == argmax t_k), and, if this was the last of request
// b's l*_b + 1 rows, the request's outcome: n_accept, and either the final
// token (greedy: argmax t at the stop row; T > 0 with nothing rejected: the
// bonus row's Gumbel-max winner) or the rejected position for the residual.
template <bool kBF16>
__device__ __noinline__ void decide_row(int n, int row, int b, int k, int gamma, int V, int per, int npad,
                                        const void* __restrict__ t, const int32_t* __restrict__ x,
                                        const float* __restrict__ lse_d, const float* __restrict__ logp_d,
                                        const int32_t* __restrict__ ell, float cscale, int greedy, uint64_t seed,
                                        int32_t* __restrict__ n_accept, int32_t* __restrict__ next_token,
                                        const VerifyWs& ws) {
    const int lane = threadIdx.x & 31;
    const int e = clamp_ell(ell, b, gamma, ws.status);
    if (k <= e) {
        int xk = x[b * gamma + k - 1];
        if (xk < 0 || xk >= V) {
            if (lane == 0) set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 5);
            xk = 0;
        }
        bool ok;
        float Lt2 = 0.f;
        if (greedy) {
            const unsigned long long w = __ldcg(ws.wt + row);
            ok = (w != 0ull) && static_cast<int>(unpack_idx(w)) == xk;
        } else {
            // the rows-pass CTAs that covered this row wrote slots 0 .. c_last - c_first
            const long long g0 = static_cast<long long>(n) * npad;
            const int nch = static_cast<int>((g0 + npad - 1) / per - g0 / per) + 1;
            float m = -INFINITY, s = 0.f;
            for (int c = lane; c < nch; c += 32) {
                const float2 pr = __ldcg(ws.part + static_cast<size_t>(row) * kNchMax + c);
                lse_merge(m, s, pr.x, pr.y);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float om = __shfl_xor_sync(0xffffffffu, m, o);
                const float os = __shfl_xor_sync(0xffffffffu, s, o);
                lse_merge(m, s, om, os);
            }
            Lt2 = m + log2f(s);
            const float yk = __ldcg(ws.tx + row) * cscale;
            const float ratio = expf((yk - Lt2) * kLn2 - logp_d[b * gamma + k - 1]);
            const float u = uniform_accept(draw_word(seed, b, k, kStreamAccept, 0));
            ok = u < ratio;
        }
        if (lane == 0) {
            ws.dec[row] = ok ? 1 : 0;
            ws.lt2row[row] = Lt2;
        }
    }
    int last = 0;
    if (lane == 0) {
        __threadfence();                                  // this row's decision before the count
        last = atomicAdd(ws.req_cnt + b, 1) == e;         // rows k = 1 .. e + 1
        __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    // the request's first rejection (gamma <= 32: one lane per position)
    const int kk = lane + 1;
    const bool rejected = kk <= e && __ldcg(ws.dec + b * (gamma + 1) + kk - 1) == 0;
    const unsigned mask = __ballot_sync(0xffffffffu, rejected);
    const int rej = mask ? __ffs(mask) : 0;
    if (lane == 0) {
        const int nacc = rej ? rej - 1 : e;
        n_accept[b] = nacc;
        ws.krow[b] = greedy ? 0 : rej;
        if (greedy || rej == 0) {
            // greedy: argmax t at the stop row nacc + 1; otherwise the bonus row e + 1's draw
            const unsigned long long w = __ldcg(ws.wt + static_cast<size_t>(b) * (gamma + 1) + nacc);
            if (w == 0ull || unpack_idx(w) >= static_cast<uint32_t>(V)) set_status(ws.status, DSPARK_ERR_DEVICE_CHECK, 6);
            next_token[b] = (w == 0ull || unpack_idx(w) >= static_cast<uint32_t>(V)) ? 0 : static_cast<int>(unpack_idx(w));
        } else {
            ws.lt2[b] = __ldcg(ws.lt2row + b * (gamma + 1) + rej - 1);
            ws.ld2[b] = lse_d[b * gamma + rej - 1] * kLog2e;
            ws.rej_list[atomicAdd(ws.rej_count, 1)] = b;   // a row of the residual launch
        }
    }
}

// ------------------------------------------------------------- rows pass ---
// CTA c takes blocks [c per, (c+1) per) of the padded scheduled rows laid end
// to end, one piece per row it touches; per piece a warp covers 4 quads of 4
// consecutive 64-token blocks per step, 8 lanes per block, 8 logits per lane
// (all loads of a step issued first).  What a piece reduces depends on its row:
//   T = 0            the argmax of t;
//   rows k <= l*_b   the (max, sum) of 2^(t log2e / T), online per lane;
//   row  l*_b + 1    the Gumbel-max winner over the row: the token maximising
//                    t_v log2e / T - log2 E_v, E_v = -ln u_v (stream 2).
// Per piece the CTA publishes its (max, sum) or its winner (atomicMax).
#ifndef DSPARK_ROWS_CTAS_PER_SM
#define DSPARK_ROWS_CTAS_PER_SM 3
#endif
constexpr int kRowsCtasPerSm = DSPARK_ROWS_CTAS_PER_SM;   // resident rows-pass CTAs per SM

template <bool kBF16>
__global__ void __launch_bounds__(256, kRowsCtasPerSm)
verify_rows(int gamma, int V, const void* __restrict__ t, const int32_t* __restrict__ x,
            const float* __restrict__ lse_d, const float* __restrict__ logp_d, const int32_t* __restrict__ ell,
            float cscale, int greedy, uint64_t seed, int32_t* __restrict__ n_accept, int32_t* __restrict__ next_token,
            VerifyWs ws, const PhiloxKeys keys) {
    __shared__ float rk[8], rm[8], rs[8];
    __shared__ int ri[8];
    __shared__ int s_last;
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
            // x_k of a decided row: the lane that loads it keeps t[x_k] for the decision
            int e = ell[b];
            e = e < 0 ? 0 : (e > gamma ? gamma : e);
            const int xk = (k <= e) ? x[b * gamma + k - 1] : -1;
            const bool draw = !greedy && k == e + 1;      // the bonus row's Gumbel-max draw
            float txk = 0.f;
            bool have_tx = false;
            float best = -INFINITY, M = -INFINITY, S = 0.f;
            int best_i = 0x7FFFFFFF;
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
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int d = xk - (((q0 + u) * 4 + sub) * 64 + part * 8);
                    if (static_cast<unsigned>(d) < 8u && (q0 + u) * 4 + sub < hi) {   // rare: one lane, one step
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (i == d) txk = y[u][i];
                        have_tx = true;
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
                } else if (draw) {
                    // the row's Philox constants, formed per step (cheaper than holding them in registers)
                    const PhiloxRow pr = philox_row_setup(seed, static_cast<uint32_t>(k), static_cast<uint32_t>(b),
                                                          kStreamVerifyToken);
                    // token v beats the lane's best iff y_v c - log2 E_v > best; E_v >= s_v = 1 - u_v,
                    // so only tokens with s_v < 2^(y_v c - best) (raised by 2^-10 for rounding) can,
                    // and only those take E_v (a warp enters when any lane has one).  -inf past V
                    // gives 2^-inf = 0: never a candidate.
                    constexpr float kSlack = 1.0009765625f;
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int v = ((q0 + u) * 4 + sub) * 64 + part * 8;
                        uint32_t wv[8];
                        uint32_t cmask = 0u;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const U4 pw = philox_row(pr, (static_cast<uint32_t>(v) >> 2) + h, keys);
                            wv[4 * h] = pw.x; wv[4 * h + 1] = pw.y; wv[4 * h + 2] = pw.z; wv[4 * h + 3] = pw.w;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (eng::one_plus_m(wv[i]) > fmaf(fast_exp2(y[u][i] * cscale - best), -kSlack, eng::kTopU))
                                cmask |= 1u << i;
                        if (__any_sync(0xffffffffu, cmask != 0u)) {
                            // each lane walks its own candidates of each group of four, lowest first
#pragma unroll
                            for (int q4 = 0; q4 < 2; ++q4) {
                                uint32_t bits = (cmask >> (4 * q4)) & 0xFu;
                                while (bits != 0u) {
                                    const int j = __ffs(bits) - 1;
                                    bits &= bits - 1u;
                                    const int i = 4 * q4 + j;
                                    const float yi = j == 0 ? y[u][4 * q4] : j == 1 ? y[u][4 * q4 + 1]
                                                   : j == 2 ? y[u][4 * q4 + 2] : y[u][4 * q4 + 3];
                                    const uint32_t wi = j == 0 ? wv[4 * q4] : j == 1 ? wv[4 * q4 + 1]
                                                      : j == 2 ? wv[4 * q4 + 2] : wv[4 * q4 + 3];
                                    const float key = yi * cscale - fast_log2(exp_draw(wi));
                                    if (key > best) { best = key; best_i = v + i; }
                                }
                            }
                        }
                    }
                } else {
                    // online (max, sum) of 2^(y c) per lane: a new maximum rescales the sum
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const float m = eng::fmax3(eng::fmax3(y[u][0], y[u][1], y[u][2]),
                                                   eng::fmax3(y[u][3], y[u][4], y[u][5]), fmaxf(y[u][6], y[u][7]));
                        if (!(m > -INFINITY)) continue;
                        const float mc = m * cscale;
                        if (mc > M) {
                            S = (S > 0.f) ? S * fast_exp2(M - mc) : 0.f;
                            M = mc;
                        }
                        float s = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) s += fast_exp2(fmaf(y[u][i], cscale, -M));
                        S += s;
                    }
                }
            }
            if (greedy || draw) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
                    if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
                }
            } else {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float om = __shfl_xor_sync(0xffffffffu, M, o);
                    const float os = __shfl_xor_sync(0xffffffffu, S, o);
                    lse_merge(M, S, om, os);
                }
            }
            if (have_tx) ws.tx[row] = txk;
            if (lane == 0) { rk[warp] = best; ri[warp] = best_i; rm[warp] = M; rs[warp] = S; }
            __syncthreads();
            if (threadIdx.x == 0) {
                float bk = -INFINITY, m = -INFINITY, s = 0.f;
                int bi = 0x7FFFFFFF;
                for (int w = 0; w < 8; ++w) {
                    if (rk[w] > bk || (rk[w] == bk && ri[w] < bi)) { bk = rk[w]; bi = ri[w]; }
                    lse_merge(m, s, rm[w], rs[w]);
                }
                if (!greedy && !draw) ws.part[static_cast<size_t>(row) * kNchMax + slot] = make_float2(m, s);
                if (bk > -INFINITY) atomicMax(&ws.wt[row], pack_key(bk, static_cast<uint32_t>(bi)));
                // the CTA that completes the row makes its decision
                const long long g0 = static_cast<long long>(n) * npad;
                const int ncta = static_cast<int>((g0 + npad - 1) / per - g0 / per) + 1;
                __threadfence();
                s_last = atomicAdd(ws.row_cnt + n, 1) == ncta - 1;
                __threadfence();
            }
            __syncthreads();                              // rk..ri are rewritten by the next piece
            if (s_last && warp == 0)
                decide_row<kBF16>(n, row, b, k, gamma, V, per, npad, t, x, lse_d, logp_d, ell, cscale, greedy, seed,
                                  n_accept, next_token, ws);
            g += hi_pad - lo;
        }
    }
}

// ---------------------------------------------------- residual, CUDA cores ---
// Request b (blockIdx.y) rejected at k, chunk blockIdx.x of the 64-token
// blocks: per token q = max(0, p_t - p_d) with p_d rebuilt from U_k + W2 . e,
// and the Gumbel-max winner of ln q (stream 2): the token maximising q_v / E_v
// (cross-multiplied), published with key log2 q - log2 E.
template <bool kBF16>
__global__ void __launch_bounds__(256)
residual_simt(int B, int gamma, int V, int r, const void* __restrict__ t, const void* __restrict__ U,
              const void* __restrict__ W1, const void* __restrict__ E, const void* __restrict__ W2,
              const int32_t* __restrict__ x0,
              const int32_t* __restrict__ x, float cscale, uint64_t seed, int nchunk, VerifyWs ws) {
    __shared__ float e[256];
    __shared__ float rk[8];
    __shared__ int ri[8];
    const int b = blockIdx.y, chunk = blockIdx.x;
    const int k = ws.krow[b];
    if (k <= 0) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int prev = prev_token(x0, x, b, gamma, k, V, ws.status);
    const void* erow = eng::bias_row<kBF16>(E, W1, b, gamma, k, r, prev);
    for (int j = threadIdx.x; j < r; j += blockDim.x) e[j] = ld_elem<kBF16>(erow, j);
    __syncthreads();
    const float lt2 = ws.lt2[b], ld2 = ws.ld2[b];
    const int nblk = (V + 63) / 64;
    const int lo = static_cast<int>(static_cast<long long>(chunk) * nblk / nchunk);
    const int hi = static_cast<int>(static_cast<long long>(chunk + 1) * nblk / nchunk);
    const size_t urow = (static_cast<size_t>(b) * gamma + (k - 1)) * V;
    const size_t trow = (static_cast<size_t>(b) * (gamma + 1) + (k - 1)) * V;
    const PhiloxRow pr = philox_row_setup(seed, static_cast<uint32_t>(k), static_cast<uint32_t>(b), kStreamVerifyToken);
    float qb = 0.f, Eb = 1.f;
    int ib = 0x7FFFFFFF;
    for (int blk = lo + warp; blk < hi; blk += 8) {
        const int v = blk * 64 + 2 * lane;
        const U4 pw = philox_row(pr, static_cast<uint32_t>(v) >> 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (v + h < V) {
                float acc = 0.f;
                for (int j = 0; j < r; ++j)
                    acc = fmaf(ld_elem<kBF16>(W2, static_cast<size_t>(v + h) * r + j), e[j], acc);
                const float yd = (ld_elem<kBF16>(U, urow + v + h) + acc) * cscale;
                const float yt = ld_elem<kBF16>(t, trow + v + h) * cscale;
                const float q = fmaxf(fast_exp2(yt - lt2) - fast_exp2(yd - ld2), 0.f);
                const float Ev = exp_draw(u4_word(pw, (v + h) & 3));
                if (q * Eb > qb * Ev) { qb = q; Eb = Ev; ib = v + h; }   // tokens ascend per thread
            }
        }
    }
    float best = (qb > 0.f) ? fast_log2(qb) - fast_log2(Eb) : -INFINITY;
    int best_i = ib;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (ob > best || (ob == best && oi < best_i)) { best = ob; best_i = oi; }
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
// Two warps per request (T > 0): eng::finish_pair, for the paths whose
// residual launch does not write the final token itself.
template <bool kBF16>
__global__ void __launch_bounds__(64)
verify_finish(int gamma, int V, eng::FinishArgs f, float cscale, uint64_t seed, StatusBlock* st) {
    __shared__ float xch[2];
    __shared__ int xchi[2];
    eng::finish_pair<kBF16>(f, blockIdx.x, gamma, V, cscale, seed, st, 1, xch, xchi);
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_verify_workspace_size(int B, int gamma, int V, int r) {
    (void)V;
    (void)r;
    if (B <= 0 || gamma <= 0) return kStatusBytes;
    return verify_ws_layout(B, gamma).total;
}

// E: the bias rows [B][gamma][r] of a gated or recurrent head, or null (Markov head).
static dspark_status_t verify_impl(int B, int gamma, int V, int r, dspark_dtype_t dt, const void* t_logits,
                                   const void* U, const void* W1, const void* E, const void* W2, const int32_t* x0,
                                   const int32_t* x, const float* lse_d, const float* logp_d, const int32_t* ell,
                                   float temperature, uint64_t seed, int32_t* n_accept, int32_t* next_token,
                                   void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
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
    clear_stale_error();
    // target rows (and U, x0, x) may be in registered host memory: the kernels read them
    // through the mapping's device address (only the rows verification needs cross the link)
    if (!device_view(t_logits, &t_logits) || !device_view(U, &U)) return DSPARK_ERR_INVALID_ARGUMENT;
    {
        const void* v = x0;
        if (!device_view(v, &v)) return DSPARK_ERR_INVALID_ARGUMENT;
        x0 = static_cast<const int32_t*>(v);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const VerifyWs ws = verify_ws(workspace, B, gamma);
    const int greedy = (temperature == 0.f);
    const float cscale = greedy ? 1.f : kLog2e / temperature;
    const bool bf = (dt == DSPARK_BF16);
    const int nblk = (V + 63) / 64;
    // plan, then the persistent rows pass (all resident CTAs) with the per-row
    // decisions and per-request outcomes made by the CTAs that finish them
    const int rgrid = kRowsCtasPerSm * sm_count(current_device());
    verify_plan<<<1, kPlanThreads, 0, s>>>(B, gamma, V, rgrid, ell, ws);
    dspark_status_t stt = launch_status();
    if (stt != DSPARK_OK) return stt;
    if (bf)
        verify_rows<true><<<rgrid, 256, 0, s>>>(gamma, V, t_logits, x, lse_d, logp_d, ell, cscale, greedy, seed,
                                                n_accept, next_token, ws, philox_keys(seed));
    else
        verify_rows<false><<<rgrid, 256, 0, s>>>(gamma, V, t_logits, x, lse_d, logp_d, ell, cscale, greedy, seed,
                                                 n_accept, next_token, ws, philox_keys(seed));
    if ((stt = launch_status()) != DSPARK_OK || greedy) return stt;

    eng::FinishArgs f{};
    f.T = bf ? static_cast<const uint16_t*>(t_logits) : nullptr;
    f.Tf = bf ? nullptr : static_cast<const float*>(t_logits);
    f.krow = ws.krow;
    f.res_word = ws.res_word;
    f.next_token = next_token;
    bool drawn = false;                                   // final tokens written by the residual launch
    if (eng::use_tc_path(dt, r)) {
        CUtensorMap map;
        if (!eng::encode_w2_map(&map, W2, V, r)) return DSPARK_ERR_CUDA;
        int nM, P;
        eng::tc_grid(B, V, &nM, &P);
        eng::TcParams p{};
        p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.k = 1;
        p.U = static_cast<const uint16_t*>(U); p.W1 = static_cast<const uint16_t*>(W1);
        p.E = static_cast<const uint16_t*>(E);
        p.W2 = static_cast<const uint16_t*>(W2); p.k_last = 1;
        p.x0 = x0; p.x = const_cast<int32_t*>(x); p.cscale = cscale; p.greedy = 0;   // read only here
        p.seed = seed; p.keys = philox_keys(seed); p.P = P;
        p.ws = eng::Ws{ws.status, ws.res_word, nullptr, nullptr, ws.gbar};
        p.krow = ws.krow; p.T = static_cast<const uint16_t*>(t_logits); p.lt2 = ws.lt2; p.ld2 = ws.ld2;
        p.rej_list = ws.rej_list; p.rej_count = ws.rej_count;
        // with a co-resident grid the same launch writes the final tokens
        drawn = nM * P <= sm_count(current_device());
        p.fuse_tail = drawn ? 1 : 0;
        p.fin = f;
        if ((stt = eng::launch_tc<eng::kResidual>(map, p, nM * P, s, drawn)) != DSPARK_OK) return stt;
    } else {
        int nchunk = (nblk + 7) / 8;
        if (nchunk > 256) nchunk = 256;
        const dim3 g(nchunk, B);
        if (bf) residual_simt<true><<<g, 256, 0, s>>>(B, gamma, V, r, t_logits, U, W1, E, W2, x0, x, cscale, seed, nchunk, ws);
        else residual_simt<false><<<g, 256, 0, s>>>(B, gamma, V, r, t_logits, U, W1, E, W2, x0, x, cscale, seed, nchunk, ws);
        if ((stt = launch_status()) != DSPARK_OK) return stt;
    }
    if (drawn) return DSPARK_OK;
    if (bf)
        verify_finish<true><<<B, 64, 0, s>>>(gamma, V, f, cscale, seed, ws.status);
    else
        verify_finish<false><<<B, 64, 0, s>>>(gamma, V, f, cscale, seed, ws.status);
    return launch_status();
}

extern "C" dspark_status_t dspark_verify(int B, int gamma, int V, int r, dspark_dtype_t dt, const void* t_logits,
                                         const void* U, const void* W1, const void* W2, const int32_t* x0,
                                         const int32_t* x, const float* lse_d, const float* logp_d,
                                         const int32_t* ell, float temperature, uint64_t seed, int32_t* n_accept,
                                         int32_t* next_token, void* workspace, size_t workspace_bytes,
                                         dspark_stream_t stream) {
    return verify_impl(B, gamma, V, r, dt, t_logits, U, W1, nullptr, W2, x0, x, lse_d, logp_d, ell, temperature,
                       seed, n_accept, next_token, workspace, workspace_bytes, stream);
}

extern "C" dspark_status_t dspark_verify_ex(int B, int gamma, int V, int r, dspark_dtype_t dt, const void* t_logits,
                                            const void* U, const void* W1, const void* W2, const int32_t* x0,
                                            const int32_t* x, const float* lse_d, const float* logp_d,
                                            const int32_t* ell, float temperature, uint64_t seed,
                                            const dspark_head_t* head, int32_t* n_accept, int32_t* next_token,
                                            void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
    const void* E = nullptr;
    if (head != nullptr && head->kind != DSPARK_HEAD_MARKOV) {
        if (head->kind != DSPARK_HEAD_GATED && head->kind != DSPARK_HEAD_RNN) return DSPARK_ERR_INVALID_ARGUMENT;
        if (head->E == nullptr || !aligned16(head->E)) return DSPARK_ERR_INVALID_ARGUMENT;
        E = head->E;
    }
    return verify_impl(B, gamma, V, r, dt, t_logits, U, W1, E, W2, x0, x, lse_d, logp_d, ell, temperature, seed,
                       n_accept, next_token, workspace, workspace_bytes, stream);
}
