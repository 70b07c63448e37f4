// dspark_schedule_prefix: the hardware-aware prefix scheduler, Algorithm 1
// (DeepSpec walkthrough, section 3.3 flowchart): sort all (b, j) pairs by the
// survival a_{b,j} descending, scan them greedily while
// Theta = (E / N) * SPS(N) rises, stop at the first pair that does not raise it.
//
// schedule_sort, one CTA of 1024 threads, everything in shared memory
// (B * gamma <= 16384):
//   1. keys k = ~bits(a) (ascending k = descending a), values = pair index
//      b * gamma + j - 1, padded with k = ~0 to a multiple of 1024;
//   2. stable LSD radix sort, four 8-bit passes; within a warp, equal digits
//      are ranked by a ballot per digit bit, so ties keep (b, j) order (up to 1024
//      pairs: a stable rank by counting instead);
//   3. exact prefix sums of a * 2^149 (each float32 a in [0, 1] is an integer
//      below 2^150 at that scale) in 192-bit integers, plus B * 2^149;
//   4. E_m = the prefix of the first m sorted pairs rounded once to double
//      (round-to-nearest-even, assembled from its bits: no floating-point
//      arithmetic), and the request of every sorted pair, to the workspace.
// schedule_theta, a grid over the pairs:
//   5. Theta_m = (E_m / (B + m)) * sps[B + m] with IEEE double ops, every m in
//      parallel, and the first m with !(Theta_m > Theta_{m-1}) (atomicMin);
//   6. the CTA that finishes last: n* (the pairs before that first drop),
//      Theta_best = Theta_{n*}, N = B + n*, and l*_b = the number of pairs of
//      request b among the first n* sorted pairs.
#include "common.cuh"
#include "host_common.h"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPairs = 16384;

struct U192 {
    unsigned long long w0, w1, w2;   // little-endian limbs
};
__device__ __forceinline__ U192 add192(U192 a, U192 b) {
    U192 r;
    r.w0 = a.w0 + b.w0;
    unsigned long long c = r.w0 < a.w0;
    const unsigned long long t1 = a.w1 + b.w1;
    const unsigned long long c1 = t1 < a.w1;
    r.w1 = t1 + c;
    c = c1 | (r.w1 < t1);
    r.w2 = a.w2 + b.w2 + c;
    return r;
}
__device__ __forceinline__ U192 shfl_up192(U192 v, int d) {
    return U192{__shfl_up_sync(0xffffffffu, v.w0, d), __shfl_up_sync(0xffffffffu, v.w1, d),
                __shfl_up_sync(0xffffffffu, v.w2, d)};
}
// a * 2^149 for a float32 a in [0, 1] (bits already validated).
__device__ __forceinline__ U192 scaled_survival(uint32_t bits) {
    const uint32_t e = (bits >> 23) & 0xFFu, m = bits & 0x7FFFFFu;
    const unsigned long long mant = (e == 0) ? m : (m | 0x800000u);
    const int sh = (e == 0) ? 0 : static_cast<int>(e) - 1;     // 0..126
    U192 r{0, 0, 0};
    if (sh < 64) {
        r.w0 = mant << sh;
        r.w1 = sh ? (mant >> (64 - sh)) : 0;
    } else if (sh < 128) {
        r.w1 = mant << (sh - 64);
        r.w2 = (sh > 64) ? (mant >> (128 - sh)) : 0;
    } else {
        r.w2 = mant << (sh - 128);
    }
    return r;
}
// round(v) to double (nearest, ties to even), times 2^-149, assembled from its
// bits (an exponent field and a 52-bit fraction).  Here v >= B 2^149 >= 2^149,
// so the result is a normal double >= 1.
__device__ __forceinline__ double u192_to_double_scaled(U192 v) {
    int hb;   // index of the highest set bit
    if (v.w2) hb = 191 - __clzll(v.w2);
    else if (v.w1) hb = 127 - __clzll(v.w1);
    else if (v.w0) hb = 63 - __clzll(v.w0);
    else return 0.0;
    // left-justify so that bit hb lands on bit 191
    const int sh = 191 - hb, q = sh >> 6, r = sh & 63;
    unsigned long long a0 = v.w0, a1 = v.w1, a2 = v.w2;
    if (q == 1) { a2 = a1; a1 = a0; a0 = 0; }
    else if (q == 2) { a2 = a0; a1 = 0; a0 = 0; }
    if (r) {
        a2 = (a2 << r) | (a1 >> (64 - r));
        a1 = (a1 << r) | (a0 >> (64 - r));
        a0 <<= r;
    }
    unsigned long long mant = a2 >> 11;                 // 53 bits, top bit set
    const bool round = (a2 >> 10) & 1ull;
    const bool sticky = (a2 & 0x3FFull) != 0 || a1 != 0 || a0 != 0;
    if (round && (sticky || (mant & 1ull))) mant += 1;
    int e = hb - 149;                                   // value = mant 2^(e - 52)
    if (mant >> 53) { mant >>= 1; e += 1; }             // the rounding carried into bit 53
    const unsigned long long bits =
        (static_cast<unsigned long long>(e + 1023) << 52) | (mant & 0xFFFFFFFFFFFFFull);
    return __longlong_as_double(static_cast<long long>(bits));
}

// The scheduler's scratch: the first-drop word and the done counter of
// schedule_theta, E_m for m = 0..n (double) and the request of each sorted pair.
struct SchedWs {
    int32_t* first_fail;
    uint32_t* done;
    double* Ed;                  // [n + 1]
    int32_t* req;                // [n]
};
inline size_t sched_ws_layout(int n, size_t* o_ctl, size_t* o_ed, size_t* o_req) {
    size_t o = kStatusBytes;
    *o_ctl = o;
    o += 256;
    *o_ed = o;
    o += round_up(static_cast<size_t>(n + 1) * 8, 256);
    *o_req = o;
    o += round_up(static_cast<size_t>(n) * 4, 256);
    return o;
}

// The lanes of this warp whose 8-bit digit equals this lane's: one ballot per
// bit, each lane keeping the lanes that agree with it on that bit.
__device__ __forceinline__ uint32_t match_digit8(uint32_t dg) {
    uint32_t peers = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const bool bit = (dg >> b) & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? bal : ~bal;
    }
    return peers;
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_sort(const float* __restrict__ a, int B, int gamma, int32_t* __restrict__ ell, StatusBlock* status,
              SchedWs ws) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = B * gamma;
    const int R = (n + kThreads - 1) / kThreads;      // rounds per warp chunk
    const int npad = R * kThreads;
    // shared memory (sized by the launch to npad): keys [2][npad] | values [2][npad] | hist
    uint32_t* key[2] = {reinterpret_cast<uint32_t*>(smem), reinterpret_cast<uint32_t*>(smem) + npad};
    uint16_t* val[2] = {reinterpret_cast<uint16_t*>(smem + 2 * npad * 4),
                        reinterpret_cast<uint16_t*>(smem + 2 * npad * 4) + npad};
    uint16_t* hist = reinterpret_cast<uint16_t*>(smem + 2 * npad * 6);   // [256][kWarps] (radix path)
    __shared__ unsigned long long wsum[3 * kWarps];
    __shared__ int red_min[kWarps];
    __shared__ uint32_t bad_seen;
    if (tid == 0) {
        bad_seen = 0;
        status->code = 0u;                            // this call's status starts clear
        status->detail = 0u;
    }
    __syncthreads();

    // 1. keys in pair order; validate a in [0, 1]
    for (int i = tid; i < npad; i += kThreads) {
        uint32_t k = 0xFFFFFFFFu;
        if (i < n) {
            const float v = a[i];
            uint32_t bits = __float_as_uint(v);
            if (!(v >= 0.f && v <= 1.f)) {
                bits = 0;
                atomicOr(&bad_seen, 1u);
            }
            if (bits == 0x80000000u) bits = 0;      // -0 counts as +0
            k = ~bits;
        }
        key[0][i] = k;
        val[0][i] = static_cast<uint16_t>(i < n ? i : 0xFFFF);
    }
    __syncthreads();
    if (tid == 0 && bad_seen) set_status(status, DSPARK_ERR_DEVICE_CHECK, 1);

    int src = 0;
    if (n <= kThreads) {
        // 2a. up to 1024 pairs: rank by counting.  rank(i) = #{j : k_j < k_i} +
        //     #{j < i : k_j == k_i}, a stable order.  Each pair gets `per` threads
        //     (as many as fit in the block, at most 8), each counting over its share
        //     of the keys in groups of four; the partial counts meet in shared memory.
        int* rk = reinterpret_cast<int*>(hist);          // [n] ranks (the radix histogram is unused here)
        const int per = min(8, kThreads / n);
        const int i = tid % n, part = tid / n;
        for (int e = tid; e < n; e += kThreads) rk[e] = 0;
        __syncthreads();
        if (part < per) {
            const uint32_t ki = key[0][i];
            const int n4 = (n + 3) / 4;                   // keys past n are ~0: never counted
            const int j0 = part * n4 / per, j1 = (part + 1) * n4 / per;
            const uint4* k4 = reinterpret_cast<const uint4*>(key[0]);
            // groups wholly before the 32 keys around i (j < i: count k_j <= k_i), those
            // wholly after them (j > i: count k_j < k_i), and the eight groups in between
            const int ib = i & ~31;
            int rank = 0;
            for (int j4 = j0; j4 < min(j1, ib / 4); ++j4) {
                const uint4 q = k4[j4];
                rank += (q.x <= ki) + (q.y <= ki) + (q.z <= ki) + (q.w <= ki);
            }
            for (int j = 4 * max(j0, ib / 4); j < 4 * min(j1, (ib + 32) / 4) && j < n; ++j) {
                const uint32_t kj = key[0][j];
                rank += (kj < ki) || (kj == ki && j < i);
            }
            for (int j4 = max(j0, (ib + 32) / 4); j4 < j1; ++j4) {
                const uint4 q = k4[j4];
                rank += (q.x < ki) + (q.y < ki) + (q.z < ki) + (q.w < ki);
            }
            atomicAdd(&rk[i], rank);
        }
        __syncthreads();
        if (tid < n) {
            key[1][rk[tid]] = key[0][tid];
            val[1][rk[tid]] = static_cast<uint16_t>(tid);
        }
        src = 1;
        __syncthreads();
    }
    // 2b. stable LSD radix sort: warp w owns elements [w R 32, (w+1) R 32) in order
    for (int shift = 0; shift < 32 && n > kThreads; shift += 8) {
        for (int i = tid; i < 256 * kWarps; i += kThreads) hist[i] = 0;
        __syncthreads();
        const int base = warp * R * 32;
        for (int rd = 0; rd < R; ++rd) {
            const int e = base + rd * 32 + lane;
            const uint32_t dg = (key[src][e] >> shift) & 0xFFu;
            const uint32_t peers = match_digit8(dg);
            if (lane == __ffs(peers) - 1) hist[dg * kWarps + warp] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // exclusive scan of hist in digit-major order (8192 entries, 8 per thread)
        {
            unsigned s = 0;
            uint16_t loc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) { loc[q] = hist[tid * 8 + q]; s += loc[q]; }
            unsigned inc = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            if (lane == 31) red_min[warp] = static_cast<int>(inc);
            __syncthreads();
            unsigned wpre = 0;
            for (int q = 0; q < warp; ++q) wpre += static_cast<unsigned>(red_min[q]);
            unsigned run = wpre + inc - s;
            __syncthreads();
#pragma unroll
            for (int q = 0; q < 8; ++q) { hist[tid * 8 + q] = static_cast<uint16_t>(run); run += loc[q]; }
        }
        __syncthreads();
        for (int rd = 0; rd < R; ++rd) {
            const int e = base + rd * 32 + lane;
            const uint32_t k = key[src][e];
            const uint16_t v = val[src][e];
            const uint32_t dg = (k >> shift) & 0xFFu;
            const uint32_t peers = match_digit8(dg);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int pos = hist[dg * kWarps + warp] + rank;
            key[src ^ 1][pos] = k;
            val[src ^ 1][pos] = v;
            __syncwarp();
            if (lane == __ffs(peers) - 1) hist[dg * kWarps + warp] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        src ^= 1;
    }
    const uint32_t* skey = key[src];
    const uint16_t* sval = val[src];

    // 3. exact prefix sums: thread t owns sorted positions [PT t, PT t + PT)
    const int PT = R;                                 // ceil(n / 1024), at most 16
    const int p0 = tid * PT;
    U192 tot{0, 0, 0};
    for (int q = 0; q < PT && p0 + q < n; ++q) tot = add192(tot, scaled_survival(~skey[p0 + q]));
    U192 inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const U192 y = shfl_up192(inc, o);
        if (lane >= o) inc = add192(inc, y);
    }
    if (lane == 31) { wsum[3 * warp] = inc.w0; wsum[3 * warp + 1] = inc.w1; wsum[3 * warp + 2] = inc.w2; }
    __syncthreads();
    if (warp == 0) {                                  // exclusive scan of the warp totals, plus B * 2^149
        const U192 wt{wsum[3 * lane], wsum[3 * lane + 1], wsum[3 * lane + 2]};
        U192 wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const U192 y = shfl_up192(wi, o);
            if (lane >= o) wi = add192(wi, y);
        }
        U192 we = add192(wi, U192{~wt.w0, ~wt.w1, ~wt.w2});
        we = add192(we, U192{1, 0, 0});               // wi - wt (two's complement)
        we = add192(we, U192{0, 0, static_cast<unsigned long long>(B) << 21});
        __syncwarp();
        wsum[3 * lane] = we.w0;
        wsum[3 * lane + 1] = we.w1;
        wsum[3 * lane + 2] = we.w2;
    }
    __syncthreads();
    U192 excl{wsum[3 * warp], wsum[3 * warp + 1], wsum[3 * warp + 2]};
    {
        const U192 y = shfl_up192(inc, 1);
        if (lane >= 1) excl = add192(excl, y);
    }

    // 4. E_m for the thread's positions (m = p0 + q + 1 pairs taken), E_0 = B, the
    //    request of each sorted pair; ell cleared for schedule_theta's counts
    if (p0 < n) {
        U192 run = excl;
        for (int q = 0; q < PT && p0 + q < n; ++q) {
            const int m = p0 + q + 1;
            run = add192(run, scaled_survival(~skey[m - 1]));
            ws.Ed[m] = u192_to_double_scaled(run);
            ws.req[m - 1] = sval[m - 1] / gamma;
        }
    }
    if (tid == 0) {
        ws.Ed[0] = static_cast<double>(B);
        *ws.first_fail = 0x7FFFFFFF;
        *ws.done = 0u;
    }
    for (int b = tid; b < B; b += kThreads) ell[b] = 0;
}

// 5-6.  Thread m (1..n) forms Theta_m and compares it with Theta_{m-1} (from the
// lane before it; lane 0 forms that one itself); the first failing m goes to an
// atomicMin.  The CTA that finishes last reads n*, writes N and Theta_best and
// counts the pairs of each request among the first n*.
constexpr int kThetaThreads = 256;

__device__ __forceinline__ double theta_of(const SchedWs& ws, const double* sps, int B, int m) {
    return __dmul_rn(__ddiv_rn(__ldcg(ws.Ed + m), static_cast<double>(B + m)), sps[B + m]);
}

__global__ void __launch_bounds__(kThetaThreads)
schedule_theta(const double* __restrict__ sps, int B, int gamma, int32_t* __restrict__ ell,
               int32_t* __restrict__ n_sched, double* __restrict__ theta, SchedWs ws) {
    __shared__ int red[kThetaThreads / 32];
    __shared__ bool last;
    const int n = B * gamma;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m = blockIdx.x * kThetaThreads + threadIdx.x + 1;
    int fail = 0x7FFFFFFF;
    double th = 0.0;
    if (m <= n) th = theta_of(ws, sps, B, m);
    double before = __shfl_up_sync(0xffffffffu, th, 1);
    if (lane == 0 && m <= n) before = theta_of(ws, sps, B, m - 1);
    if (m <= n && !(th > before)) fail = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fail = min(fail, __shfl_xor_sync(0xffffffffu, fail, o));
    if (lane == 0) red[warp] = fail;
    __syncthreads();
    if (threadIdx.x == 0) {
        int f = 0x7FFFFFFF;
        for (int w = 0; w < kThetaThreads / 32; ++w) f = min(f, red[w]);
        if (f != 0x7FFFFFFF) atomicMin(ws.first_fail, f);
        __threadfence();
        last = atomicAdd(ws.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int ff = atomicAdd(ws.first_fail, 0);
    const int nstar = (ff == 0x7FFFFFFF) ? n : ff - 1;
    if (threadIdx.x == 0) {
        *n_sched = B + nstar;
        *theta = theta_of(ws, sps, B, nstar);
    }
    for (int q = threadIdx.x; q < nstar; q += kThetaThreads) atomicAdd(&ell[__ldcg(ws.req + q)], 1);
}

// Shared memory for npad padded pairs: keys and values double-buffered, the radix
// histogram (or the ranks of the counting path).
constexpr size_t smem_bytes(int npad) {
    return 2 * static_cast<size_t>(npad) * 4 + 2 * static_cast<size_t>(npad) * 2 + 256 * kWarps * 2;
}
constexpr size_t kSmem = smem_bytes(kMaxPairs);

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_schedule_prefix_workspace_size(int B, int gamma) {
    if (B <= 0 || gamma <= 0 || static_cast<long long>(B) * gamma > kMaxPairs) return kStatusBytes;
    size_t oc, oe, orq;
    return sched_ws_layout(B * gamma, &oc, &oe, &orq);
}

extern "C" dspark_status_t dspark_schedule_prefix(int B, int gamma, const float* a, const double* sps,
                                                  int32_t* ell, int32_t* n_sched, double* theta,
                                                  void* workspace, size_t workspace_bytes,
                                                  dspark_stream_t stream) {
    if (B <= 0 || gamma <= 0 || gamma > DSPARK_MAX_GAMMA) return DSPARK_ERR_INVALID_ARGUMENT;
    if (static_cast<long long>(B) * gamma > kMaxPairs) return DSPARK_ERR_UNSUPPORTED;
    if (!a || !sps || !ell || !n_sched || !theta) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_schedule_prefix_workspace_size(B, gamma)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    clear_stale_error();
    {   // the SPS table may be in registered host memory (read through its mapping)
        const void* v = sps;
        if (!device_view(v, &v)) return DSPARK_ERR_INVALID_ARGUMENT;
        sps = static_cast<const double*>(v);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    static OncePerDevice once;
    if (once.run(current_device(), [] {
            return cudaFuncSetAttribute(schedule_sort, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int n = B * gamma;
    const int npad = (n + kThreads - 1) / kThreads * kThreads;
    size_t oc, oe, orq;
    sched_ws_layout(n, &oc, &oe, &orq);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const SchedWs ws{reinterpret_cast<int32_t*>(w + oc), reinterpret_cast<uint32_t*>(w + oc + 16),
                     reinterpret_cast<double*>(w + oe), reinterpret_cast<int32_t*>(w + orq)};
    schedule_sort<<<1, kThreads, smem_bytes(npad), s>>>(a, B, gamma, ell, static_cast<StatusBlock*>(workspace), ws);
    dspark_status_t st = launch_status();
    if (st != DSPARK_OK) return st;
    schedule_theta<<<(n + kThetaThreads - 1) / kThetaThreads, kThetaThreads, 0, s>>>(sps, B, gamma, ell, n_sched,
                                                                                    theta, ws);
    return launch_status();
}
