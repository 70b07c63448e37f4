// dspark_schedule_prefix: the hardware-aware prefix scheduler, Algorithm 1
// (DeepSpec walkthrough, section 3.3 flowchart): sort all (b, j) pairs by the
// survival a_{b,j} descending, scan them greedily while
// Theta = (E / N) * SPS(N) rises, stop at the first pair that does not raise it.
//
// Three launches over chunks of 128 pairs in pair order (B * gamma <= 16384, so
// at most 128 CTAs: one wave):
// schedule_chunks, one CTA per chunk:
//   1. keys k = ~bits(a) (ascending k = descending a), each chunk sorted by a
//      stable rank by counting (rank = #{k_j < k_i} + #{j < i : k_j == k_i});
//      a outside [0, 1] is flagged per chunk; ell and the control words cleared.
// schedule_rank, one CTA per chunk, every chunk's keys in shared memory:
//   2. the sorted position of each pair = its rank in its chunk + the keys of
//      every earlier chunk that are <= its key + those of every later chunk that
//      are < it (binary searches in the sorted chunks): a stable order, ties kept
//      in (b, j) order.  Scatters the key and the request of each pair there and
//      adds a * 2^149 to the sum of its 128 sorted positions (48-bit limbs,
//      64-bit atomics: exact, whatever the order).
// schedule_scan, one CTA per 128 sorted positions:
//   3. exact prefix sums of a * 2^149 (each float32 a in [0, 1] is an integer
//      below 2^150 at that scale) in 192-bit integers, plus B * 2^149 (the sums
//      of the sorted chunks before the CTA's range, then a scan of its own);
//   4. E_m = the prefix of the first m sorted pairs rounded once to double
//      (round-to-nearest-even, assembled from its bits: no floating-point
//      arithmetic);
//   5. Theta_m = (E_m / (B + m)) * sps[B + m] with IEEE double ops, and the first
//      m with !(Theta_m > Theta_{m-1}) (atomicMin);
//   6. the CTA that finishes last: the status, n* (the pairs before that first
//      drop), Theta_best = Theta_{n*}, N = B + n*, and l*_b = the number of pairs
//      of request b among the first n* sorted pairs.
#include "common.cuh"
#include "host_common.h"

namespace dspark {
namespace {

constexpr int kChunk = 128;                        // pairs per chunk: threads of schedule_chunks / _scan
constexpr int kRankThreads = 1024;                 // schedule_rank: kRankParts threads per pair
constexpr int kRankParts = kRankThreads / kChunk;
constexpr int kMaxPairs = 16384;
constexpr int kMaxChunks = kMaxPairs / kChunk;

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
// v < 2^150 as four 48-bit limbs (v = l0 + l1 2^48 + l2 2^96 + l3 2^144): sums of up
// to 2^14 such limbs stay below 2^62, so limb-wise 64-bit adds (atomics included)
// never carry.
constexpr unsigned long long kLimb = (1ull << 48) - 1;
__device__ __forceinline__ void limbs48(U192 v, unsigned long long l[4]) {
    l[0] = v.w0 & kLimb;
    l[1] = ((v.w0 >> 48) | (v.w1 << 16)) & kLimb;
    l[2] = ((v.w1 >> 32) | (v.w2 << 32)) & kLimb;
    l[3] = v.w2 >> 16;
}
__device__ __forceinline__ U192 from_limbs48(const unsigned long long l[4]) {
    U192 r{l[0], 0, 0};
    r = add192(r, U192{l[1] << 48, l[1] >> 16, 0});
    r = add192(r, U192{0, l[2] << 32, l[2] >> 32});
    r = add192(r, U192{0, 0, l[3] << 16});
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
// schedule_scan, a flag per chunk, the chunk-sorted keys and pair indices, the
// keys and requests in sorted order, and E_m for m = 0..n (double).
struct SchedWs {
    int32_t* first_fail;
    uint32_t* done;
    uint32_t* bad;               // [chunks] nonzero where the chunk held an a outside [0, 1]
    unsigned long long* acc;     // [chunks][4] sum of a 2^149 over each 128 sorted positions, in 48-bit limbs
    uint32_t* ckey;              // [n] keys, sorted within each chunk
    int32_t* cval;               // [n] the pair index of each, in the same order
    uint32_t* skey;              // [n] keys in sorted order
    int32_t* req;                // [n] the request of each sorted pair
    double* Ed;                  // [n + 1]
};
inline size_t sched_ws_layout(int n, SchedWs* ws, uint8_t* w) {
    size_t o = kStatusBytes;
    const size_t ctl = o;
    o += 256;
    const size_t bad = o;
    o += round_up(static_cast<size_t>(kMaxChunks) * 4, 256);
    const size_t acc = o;
    o += round_up(static_cast<size_t>(kMaxChunks) * 32, 256);
    const size_t ckey = o;
    o += round_up(static_cast<size_t>(n) * 4, 256);
    const size_t cval = o;
    o += round_up(static_cast<size_t>(n) * 4, 256);
    const size_t skey = o;
    o += round_up(static_cast<size_t>(n) * 4, 256);
    const size_t req = o;
    o += round_up(static_cast<size_t>(n) * 4, 256);
    const size_t ed = o;
    o += round_up(static_cast<size_t>(n + 1) * 8, 256);
    if (ws != nullptr) {
        *ws = SchedWs{reinterpret_cast<int32_t*>(w + ctl), reinterpret_cast<uint32_t*>(w + ctl + 16),
                      reinterpret_cast<uint32_t*>(w + bad), reinterpret_cast<unsigned long long*>(w + acc),
                      reinterpret_cast<uint32_t*>(w + ckey),
                      reinterpret_cast<int32_t*>(w + cval), reinterpret_cast<uint32_t*>(w + skey),
                      reinterpret_cast<int32_t*>(w + req), reinterpret_cast<double*>(w + ed)};
    }
    return o;
}

// 1.  One chunk of 128 pairs: validate, key, stable rank by counting, write the
//     chunk in key order.  CTA 0 also clears the status and the control words;
//     every CTA clears its share of ell.
__global__ void __launch_bounds__(kChunk)
schedule_chunks(const float* __restrict__ a, int B, int gamma, int32_t* __restrict__ ell, StatusBlock* status,
                SchedWs ws) {
    __shared__ uint32_t ks[kChunk];
    __shared__ uint32_t bad;
    const int n = B * gamma, c = blockIdx.x, tid = threadIdx.x;
    const int base = c * kChunk, len = min(kChunk, n - base);
    if (tid == 0) bad = 0u;
    __syncthreads();
    uint32_t k = 0xFFFFFFFFu;
    if (tid < len) {
        const float v = a[base + tid];
        uint32_t bits = __float_as_uint(v);
        if (!(v >= 0.f && v <= 1.f)) {
            bits = 0;
            bad = 1u;
        }
        if (bits == 0x80000000u) bits = 0;          // -0 counts as +0
        k = ~bits;
    }
    ks[tid] = k;
    __syncthreads();
    if (tid < len) {
        int r = 0;
        for (int j = 0; j < len; ++j) {
            const uint32_t kj = ks[j];
            r += (kj < k) || (kj == k && j < tid);
        }
        ws.ckey[base + r] = k;
        ws.cval[base + r] = base + tid;
    }
    if (tid == 0) ws.bad[c] = bad;
    if (tid < 4) ws.acc[4 * c + tid] = 0ull;
    for (int b = base + tid; b < B; b += gridDim.x * kChunk) ell[b] = 0;
    if (c == 0 && tid == 0) {
        status->code = 0u;                            // this call's status starts clear
        status->detail = 0u;
        *ws.first_fail = 0x7FFFFFFF;
        *ws.done = 0u;
    }
}

// 2.  Thread (part, q) of CTA c counts, for pair q of chunk c, the keys ordered
//     before it in the chunks c2 = part + i kRankParts (i < kPer); the partial
//     counts meet in shared memory and the pair is scattered to its sorted
//     position.  kPer kRankParts >= the number of chunks; chunks past the last
//     are all padding.
template <int kPer>
__global__ void __launch_bounds__(kRankThreads)
schedule_rank(int n, int gamma, SchedWs ws) {
    extern __shared__ __align__(16) uint32_t keys[];   // kPer kRankParts chunks, each in key order
    __shared__ int cnt[kRankParts][kChunk];
    const int c = blockIdx.x, tid = threadIdx.x;
    constexpr int npad = kPer * kRankParts * kChunk;
    // padding keys ~0 are never below a key, and every padded chunk is later than
    // any real one, so it is only ever searched with "<"
    if ((n & 3) == 0) {
        const uint4* src = reinterpret_cast<const uint4*>(ws.ckey);
        uint4* dst = reinterpret_cast<uint4*>(keys);
        constexpr int kU = npad / 4 / kRankThreads > 0 ? npad / 4 / kRankThreads : 1;
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = tid + u * kRankThreads;
            v[u] = (i < n / 4) ? __ldcg(src + i) : make_uint4(~0u, ~0u, ~0u, ~0u);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = tid + u * kRankThreads;
            if (i < npad / 4) dst[i] = v[u];
        }
    } else {
        for (int i = tid; i < npad; i += kRankThreads) keys[i] = (i < n) ? __ldcg(ws.ckey + i) : 0xFFFFFFFFu;
    }
    __syncthreads();
    const int base = c * kChunk, len = min(kChunk, n - base);
    const int q = tid % kChunk, part = tid / kChunk;
    // #{keys <= x} of each earlier chunk (its pairs win ties) and #{keys < x} =
    // #{keys <= x - 1} of each later one (x >= ~bits(1.0) > 0), by binary searches
    // over the bits of the count from the highest down; the chunks' searches run
    // interleaved, step by step
    int before = 0;
    if (q < len) {
        const uint32_t x = keys[base + q];
        int pos[kPer];                                // index into keys, within chunk c2
        uint32_t th[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int c2 = part + i * kRankParts;
            pos[i] = c2 * kChunk;
            th[i] = (c2 < c) ? x : x - 1u;
        }
#pragma unroll
        for (int step = kChunk / 2; step > 0; step >>= 1) {
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (keys[pos[i] + (step - 1)] <= th[i]) pos[i] += step;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int c2 = part + i * kRankParts;
            const int k = pos[i] - c2 * kChunk + (keys[pos[i]] <= th[i]);
            before += (c2 != c) ? k : 0;
        }
    }
    cnt[part][q] = before;
    __syncthreads();
    if (tid < len) {
        int r = tid;                                  // sorted position: rank in the chunk + the counts
#pragma unroll
        for (int p = 0; p < kRankParts; ++p) r += cnt[p][tid];
        const uint32_t k = keys[base + tid];
        ws.skey[r] = k;
        ws.req[r] = __ldcg(ws.cval + base + tid) / gamma;
        unsigned long long l[4];
        limbs48(scaled_survival(~k), l);
        unsigned long long* dst = ws.acc + 4 * (r / kChunk);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (l[i]) atomicAdd(dst + i, l[i]);
    }
}

// Theta_m = (E_m / (B + m)) * SPS(B + m), one IEEE division and one multiplication.
__device__ __forceinline__ double theta_of(double E, const double* sps, int B, int m) {
    return __dmul_rn(__ddiv_rn(E, static_cast<double>(B + m)), sps[B + m]);
}

// Up to 1024 pairs: every step in one CTA and its shared memory (one launch).
// Thread p keys pair p; the pairs are ranked as in the chunked path (within
// chunks of 128 by counting, then binary searches in the other chunks),
// scattered, scanned (192-bit), and thread p forms Theta_{p+1}; the first drop
// is a block minimum and l* is counted with shared-memory atomics.
constexpr int kSmallPairs = 1024;

__global__ void __launch_bounds__(kSmallPairs, 1)
schedule_small(const float* __restrict__ a, const double* __restrict__ sps, int B, int gamma,
               int32_t* __restrict__ ell, int32_t* __restrict__ n_sched, double* __restrict__ theta,
               StatusBlock* status) {
    constexpr int kW = kSmallPairs / 32;
    __shared__ __align__(16) uint32_t ks[kSmallPairs];
    __shared__ uint32_t rk[kSmallPairs];
    __shared__ uint32_t sk[kSmallPairs];
    __shared__ int sq[kSmallPairs];
    __shared__ int el[kSmallPairs];
    __shared__ unsigned long long tot[3 * kW];
    __shared__ int red[kW];
    __shared__ uint32_t bad;
    const int n = B * gamma, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = 0u;
    el[tid] = 0;
    uint32_t k = 0xFFFFFFFFu;
    __syncthreads();
    if (tid < n) {
        const float v = a[tid];
        uint32_t bits = __float_as_uint(v);
        if (!(v >= 0.f && v <= 1.f)) {
            bits = 0;
            bad = 1u;
        }
        if (bits == 0x80000000u) bits = 0;          // -0 counts as +0
        k = ~bits;
    }
    ks[tid] = k;
    __syncthreads();
    // rank(i) = #{j : k_j < k_i} + #{j < i : k_j == k_i}, in two steps: the rank
    // within i's chunk of 128 pairs (counting), then binary searches in the other
    // chunks, sorted meanwhile (their keys <= k_i for earlier chunks, < k_i later)
    const int cc = tid / kChunk, cb = cc * kChunk, il = tid - cb;
    const int nchunks = (n + kChunk - 1) / kChunk;
    rk[tid] = 0xFFFFFFFF;                             // the chunk-sorted keys; ~0 pads the last chunk
    int r = 0;
    if (tid < n) {
        const int cl = min(kChunk, n - cb);
        const uint4* k4 = reinterpret_cast<const uint4*>(ks + cb);
        const int own = il / 4;
        for (int g = 0; g < own; ++g) {               // wholly before i: ties count
            const uint4 q = k4[g];
            r += (q.x <= k) + (q.y <= k) + (q.z <= k) + (q.w <= k);
        }
        for (int j = 4 * own; j < min(4 * own + 4, cl); ++j) {
            const uint32_t kj = ks[cb + j];
            r += (kj < k) || (kj == k && j < il);
        }
        const int ng = cl / 4;                        // whole groups (keys past n in a group are ~0)
        for (int g = own + 1; g < ng; ++g) {          // wholly after i
            const uint4 q = k4[g];
            r += (q.x < k) + (q.y < k) + (q.z < k) + (q.w < k);
        }
        for (int j = max(4 * ng, 4 * own + 4); j < cl; ++j) r += ks[cb + j] < k;
    }
    __syncthreads();
    if (tid < n) rk[cb + r] = k;
    __syncthreads();
    if (tid < n) {
        const uint32_t* csk = rk;
        for (int c2 = 0; c2 < nchunks; ++c2) {
            if (c2 == cc) continue;
            const uint32_t th = (c2 < cc) ? k : k - 1u;   // k >= ~bits(1.0) > 0
            const uint32_t* y = csk + c2 * kChunk;
#pragma unroll
            for (int step = kChunk / 2; step > 0; step >>= 1)
                if (y[step - 1] <= th) y += step;
            r += static_cast<int>(y - (csk + c2 * kChunk)) + (y[0] <= th);
        }
        sk[r] = k;
        sq[r] = tid / gamma;
    }
    __syncthreads();
    // E_m 2^149 = B 2^149 + the survivals of the first m sorted pairs (m = p + 1)
    const int p = tid;
    const U192 v = (p < n) ? scaled_survival(~sk[p]) : U192{0, 0, 0};
    U192 inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const U192 y = shfl_up192(inc, o);
        if (lane >= o) inc = add192(inc, y);
    }
    if (lane == 31) { tot[3 * warp] = inc.w0; tot[3 * warp + 1] = inc.w1; tot[3 * warp + 2] = inc.w2; }
    __syncthreads();
    if (warp == 0) {                                  // exclusive scan of the warp totals, plus B 2^149
        const U192 wt{tot[3 * lane], tot[3 * lane + 1], tot[3 * lane + 2]};
        U192 wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const U192 y = shfl_up192(wi, o);
            if (lane >= o) wi = add192(wi, y);
        }
        U192 we = shfl_up192(wi, 1);
        if (lane == 0) we = U192{0, 0, 0};
        we = add192(we, U192{0, 0, static_cast<unsigned long long>(B) << 21});
        __syncwarp();
        tot[3 * lane] = we.w0;
        tot[3 * lane + 1] = we.w1;
        tot[3 * lane + 2] = we.w2;
    }
    __syncthreads();
    U192 ex = shfl_up192(inc, 1);
    if (lane == 0) ex = U192{0, 0, 0};
    const U192 excl = add192(U192{tot[3 * warp], tot[3 * warp + 1], tot[3 * warp + 2]}, ex);
    const U192 incl = add192(excl, v);
    // Theta_m in blocks of 128 m (four warps), stopping after the block with the
    // first drop: double division is slow on this part, and n* is often small
    const double Em = u192_to_double_scaled(incl);
    double th = 0.0, before = 0.0;
    int f = 0x7FFFFFFF;
    for (int blk = 0; blk * 128 < n; ++blk) {
        if (warp / 4 == blk) {
            int fail = 0x7FFFFFFF;
            if (p < n) th = theta_of(Em, sps, B, p + 1);
            before = __shfl_up_sync(0xffffffffu, th, 1);   // Theta_{m-1} from the lane before
            if (lane == 0 && p < n) before = theta_of(u192_to_double_scaled(excl), sps, B, p);
            if (p < n && !(th > before)) fail = p + 1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) fail = min(fail, __shfl_xor_sync(0xffffffffu, fail, o));
            if (lane == 0) red[warp] = fail;
        }
        __syncthreads();
#pragma unroll
        for (int w = 0; w < 4; ++w) f = min(f, red[4 * blk + w]);
        if (f != 0x7FFFFFFF) break;                   // uniform: every thread read the same red[]
    }
    const int nstar = (f == 0x7FFFFFFF) ? n : f - 1;
    if (p < nstar) atomicAdd(&el[sq[p]], 1);
    if (nstar > 0 ? p == nstar - 1 : p == 0) *theta = nstar > 0 ? th : before;   // Theta_{n*}
    __syncthreads();
    if (tid < B) ell[tid] = el[tid];
    if (tid == 0) {
        *n_sched = B + nstar;
        status->code = bad ? static_cast<uint32_t>(DSPARK_ERR_DEVICE_CHECK) : 0u;
        status->detail = bad ? 1u : 0u;
    }
}

template <int kPer>
dspark_status_t launch_rank(int chunks, int n, int gamma, const SchedWs& ws, cudaStream_t s) {
    constexpr size_t smem = static_cast<size_t>(kPer) * kRankParts * kChunk * sizeof(uint32_t);
    static OncePerDevice once;
    if (smem > 48 * 1024 && once.run(current_device(), [] {
            return cudaFuncSetAttribute(schedule_rank<kPer>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    schedule_rank<kPer><<<chunks, kRankThreads, smem, s>>>(n, gamma, ws);
    return launch_status();
}

// 3-6.  CTA c owns sorted positions p = 128 c + t (m = p + 1 pairs taken).
__global__ void __launch_bounds__(kChunk)
schedule_scan(const double* __restrict__ sps, int B, int gamma, int32_t* __restrict__ ell,
              int32_t* __restrict__ n_sched, double* __restrict__ theta, StatusBlock* status, SchedWs ws) {
    constexpr int kW = kChunk / 32;
    __shared__ unsigned long long tot[3 * kW], prs[3 * kW];
    __shared__ int red[kW];
    __shared__ bool last;
    const int n = B * gamma, c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int base = c * kChunk, p = base + tid;
    // every global read this CTA needs before its Theta, issued together
    unsigned long long lp[4] = {0ull, 0ull, 0ull, 0ull};
    uint32_t key = 0xFFFFFFFFu;
    double s_m = 0.0, s_b = 0.0;                      // SPS(B + m), SPS(B + m - 1)
    if (tid < c) {
        const ulonglong2* q = reinterpret_cast<const ulonglong2*>(ws.acc + 4 * tid);
        const ulonglong2 x = __ldcg(q), y = __ldcg(q + 1);
        lp[0] = x.x; lp[1] = x.y; lp[2] = y.x; lp[3] = y.y;
    }
    if (p < n) {
        key = __ldcg(ws.skey + p);
        s_m = sps[B + p + 1];
        if (lane == 0) s_b = sps[B + p];
    }
    // the pairs before this range: the 48-bit limb sums of the sorted chunks before c
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp[i] += __shfl_xor_sync(0xffffffffu, lp[i], o);
    const U192 pre = from_limbs48(lp);                // this warp's share
    // this range: inclusive scan of a * 2^149 within each warp
    const U192 v = (p < n) ? scaled_survival(~key) : U192{0, 0, 0};
    U192 inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const U192 y = shfl_up192(inc, o);
        if (lane >= o) inc = add192(inc, y);
    }
    U192 ex = shfl_up192(inc, 1);                     // exclusive within the warp
    if (lane == 0) ex = U192{0, 0, 0};
    // the warps' totals of this range and their shares of the pairs before it
    if (lane == 31) { tot[3 * warp] = inc.w0; tot[3 * warp + 1] = inc.w1; tot[3 * warp + 2] = inc.w2; }
    if (lane == 0) { prs[3 * warp] = pre.w0; prs[3 * warp + 1] = pre.w1; prs[3 * warp + 2] = pre.w2; }
    __syncthreads();
    U192 run{0, 0, static_cast<unsigned long long>(B) << 21};   // B 2^149
#pragma unroll
    for (int w = 0; w < kW; ++w) {
        run = add192(run, U192{prs[3 * w], prs[3 * w + 1], prs[3 * w + 2]});
        if (w < warp) run = add192(run, U192{tot[3 * w], tot[3 * w + 1], tot[3 * w + 2]});
    }
    const U192 excl = add192(run, ex);                // E_{m-1} 2^149 (m = p + 1)
    const U192 incl = add192(excl, v);                // E_m 2^149
    int fail = 0x7FFFFFFF;
    double th = 0.0;
    if (p < n) {
        const double Em = u192_to_double_scaled(incl);
        ws.Ed[p + 1] = Em;
        th = __dmul_rn(__ddiv_rn(Em, static_cast<double>(B + p + 1)), s_m);   // theta_of(Em, m = p + 1)
    }
    double before = __shfl_up_sync(0xffffffffu, th, 1);   // Theta_{m-1} from the lane before
    if (lane == 0 && p < n) {
        const double Eb = u192_to_double_scaled(excl);
        if (p == 0) ws.Ed[0] = Eb;                    // = B exactly
        before = __dmul_rn(__ddiv_rn(Eb, static_cast<double>(B + p)), s_b);
    }
    if (p < n && !(th > before)) fail = p + 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fail = min(fail, __shfl_xor_sync(0xffffffffu, fail, o));
    if (lane == 0) red[warp] = fail;
    __syncthreads();
    if (tid == 0) {
        int f = 0x7FFFFFFF;
        for (int w = 0; w < kW; ++w) f = min(f, red[w]);
        if (f != 0x7FFFFFFF) atomicMin(ws.first_fail, f);
        __threadfence();
        last = atomicAdd(ws.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int ff = atomicAdd(ws.first_fail, 0);
    const int nstar = (ff == 0x7FFFFFFF) ? n : ff - 1;
    const int any_bad = __syncthreads_or(tid < gridDim.x && __ldcg(ws.bad + tid) != 0u);
    if (tid == 0) {
        if (any_bad) set_status(status, DSPARK_ERR_DEVICE_CHECK, 1);
        *n_sched = B + nstar;
        *theta = theta_of(__ldcg(ws.Ed + nstar), sps, B, nstar);
    }
    // l*_b: the requests of the first n* sorted pairs, eight loads in flight per thread
    for (int q0 = tid; q0 < nstar; q0 += 8 * kChunk) {
        int rq[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rq[u] = (q0 + u * kChunk < nstar) ? __ldcg(ws.req + q0 + u * kChunk) : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (rq[u] >= 0) atomicAdd(&ell[rq[u]], 1);
    }
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_schedule_prefix_workspace_size(int B, int gamma) {
    if (B <= 0 || gamma <= 0 || static_cast<long long>(B) * gamma > kMaxPairs) return kStatusBytes;
    return sched_ws_layout(B * gamma, nullptr, nullptr);
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
    const int n = B * gamma;
    StatusBlock* status = static_cast<StatusBlock*>(workspace);
    if (n <= kSmallPairs) {
        schedule_small<<<1, kSmallPairs, 0, s>>>(a, sps, B, gamma, ell, n_sched, theta, status);
        return launch_status();
    }
    const int chunks = (n + kChunk - 1) / kChunk;
    SchedWs ws;
    sched_ws_layout(n, &ws, static_cast<uint8_t*>(workspace));
    schedule_chunks<<<chunks, kChunk, 0, s>>>(a, B, gamma, ell, status, ws);
    dspark_status_t st = launch_status();
    if (st != DSPARK_OK) return st;
    const int per = (chunks + kRankParts - 1) / kRankParts;   // chunks per part: 2 .. 16 (n > 1024)
    st = per <= 2 ? launch_rank<2>(chunks, n, gamma, ws, s)
         : per <= 4 ? launch_rank<4>(chunks, n, gamma, ws, s)
         : per <= 8 ? launch_rank<8>(chunks, n, gamma, ws, s)
                    : launch_rank<16>(chunks, n, gamma, ws, s);
    if (st != DSPARK_OK) return st;
    schedule_scan<<<chunks, kChunk, 0, s>>>(sps, B, gamma, ell, n_sched, theta, status, ws);
    return launch_status();
}
