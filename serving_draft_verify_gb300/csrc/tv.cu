// dspark_accept_rate_tv: c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 per row
// (DeepSpec walkthrough, section 3.3, paper eq. 8 / `_compute_accept_rate_3d`),
// computed as sum_v exp(min(d_v - L_d, t_v - L_t)) with L = logsumexp of the row;
// and dspark_training_loss (section 7.2, `compute_dspark_loss`), the same pass
// extended to the joint loss and its gradient.
//
// One HBM pass per row.  A thread-block cluster of cs CTAs of 640 threads (cs the
// smallest of 1, 2, 4, 8, 16 whose slices fit; 4 for bf16 rows of the Qwen3
// vocabulary) owns one row at a time; each CTA bulk-copies its 1/cs slice of d
// and t into shared memory.  Slices stream through three slots in the order d_0,
// t_0, d_1, t_1, ..., so row i+1's d lands while row i is reduced:
//   AB. per tensor: each thread's max (packed bf16 max) and sum of
//       2^((x - m) log2e) over its elements (two reads of shared memory); merged
//       per warp (max, then rescaled sum), per CTA;
//   -- cluster barrier: the CTAs' (m, s) through distributed shared memory (and
//      the previous row's partials, which rank 0 sums into c*) --
//   C.  sum of 2^(min(d - L_d, t - L_t) log2e) from shared memory;
//   loss mode: C also sums p_d over d - t < L_d - L_t and over ties, a second
//   cluster barrier exchanges them with the target logit, and pass D writes
//   dL/dd from shared memory.
// Three exponentials per logit pair (four with the gradient); every byte of d
// and t is read once from HBM.
#include <cooperative_groups.h>

#include "common.cuh"
#include "host_common.h"

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kMaxCS = 16;      // CTAs per cluster at most (one row per cluster)
constexpr int kThreads = 640;
constexpr int kWarps = kThreads / 32;
constexpr int kSlots = 3;       // slice slots: d_i, t_i and d_{i+1} resident at once
constexpr int kGMax = 8;        // 16-byte groups per thread and slice (a slot holds at most 8 x 640 x 16 B)
constexpr size_t kSmemCap = 227 * 1024;

template <bool kBF16>
struct TVTraits {
    static constexpr int kEPG = kBF16 ? 8 : 4;   // elements per 16-byte group
    static constexpr int kESZ = kBF16 ? 2 : 4;
};

template <bool kBF16>
__device__ __forceinline__ void unpack(const uint4 v, float* out) {
    if constexpr (kBF16) {
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z); out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
    } else {
        out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
    }
}

// Packed pairs of float32 (Blackwell f32x2 arithmetic): two lanes of work per
// instruction for the element-wise part of the sums.
__device__ __forceinline__ unsigned long long pk(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 upk(unsigned long long v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Two floats -> a bf16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// One CTA's exchange slot, double-buffered by row parity: a CTA writes row it+2's
// values only after a cluster barrier that every CTA reaches after its reads of
// row it's values.
struct Slot {
    float4 ms[2];           // slice (max, sum of 2^((x - max) log2e)) of d and t: (md, sd, mt, st)
    float4 q[2];            // loss mode: (sum of 2^(min) terms, sum p_d over d - t < L_d - L_t, over ties, d[target] or -inf)
    float p[2];             // CTA partial of sum min(p_d, p_t)
    float pad[2];
};

// The training loss (loss mode of the kernel): per row, with p = softmax,
//   ce = logsumexp(d) - d[target], c* = sum min(p_d, p_t), l1 = 1 - c*,
//   bce = softplus(s) - c* s, row = omega (a_ce ce + a_l1 l1 + a_conf bce),
//   dL/dd_v = omega (a_ce (p_d(v) - [v = target]) + a_l1 / 2 p_d(v) (sgn_v - sum_u p_d(u) sgn_u)),
//   dL/ds = omega a_conf (sigmoid(s) - c*), sgn_v = sign(p_d(v) - p_t(v)).
// sum_u p_d(u) sgn_u = 1 - 2 P_lt - P_eq, with P_lt (P_eq) the p_d mass where
// p_d < p_t (p_d = p_t): pass C's terms there are p_d itself.
struct LossArgs {
    const int32_t* target;  // [rows]
    const float* s;         // [rows] confidence head logits
    const float* omega;     // [rows] row weights
    float a_ce, a_l1, a_conf;
    float* row_out;         // [rows][4] (ce, c*, bce, row)
    void* grad;             // [rows][V] dL/dd (input dtype), or null
    float* grad_s;          // [rows] dL/ds, or null
    float* cl_part;         // [clusters] each cluster's sum of row totals
    unsigned int* cl_done;  // clusters finished (starts at 0)
    float* loss;            // [1] sum of row totals
};

// (m, s) with s a sum of 2^((x - m) log2e): merge across a warp (the warp's max of
// the m that carry mass, then the rescaled sum).
__device__ __forceinline__ void warp_lse(float& m, float& s) {
    const float M = warp_max(s > 0.f ? m : -INFINITY);
    const float r = s > 0.f ? s * fast_exp2((m - M) * kLog2e) : 0.f;
    s = warp_sum(r);
    m = M > -INFINITY ? M : 0.f;
}

// log2 on the special-function unit (lg2.approx.ftz: absolute error about 2^-22).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// This thread's (max, sum of 2^((x - max) log2e)) over its groups of a slice.
// e = 2^((x - m) log2e): the difference is formed first, so it is exactly 0 at the
// max and <= 0 elsewhere, whatever the magnitude of x; a thread without a finite
// logit keeps reference 0 so that its terms are 0.
template <bool kBF16>
__device__ __forceinline__ void thread_lse(const uint4* __restrict__ g, int ngroups, int tid, float& m_out,
                                           float& s_out) {
    constexpr int EPG = TVTraits<kBF16>::kEPG;
    float mx = -INFINITY;
    if constexpr (kBF16) {
        uint32_t am = 0xFF80FF80u;                        // (-inf, -inf)
#pragma unroll
        for (int j = 0; j < kGMax; ++j) {
            const int gi = tid + j * kThreads;
            if (gi < ngroups) {
                const uint4 v = g[gi];
                am = bmax2(am, bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)));
            }
        }
        mx = fmaxf(bf16lo(am), bf16hi(am));
    } else {
#pragma unroll
        for (int j = 0; j < kGMax; ++j) {
            const int gi = tid + j * kThreads;
            if (gi < ngroups) {
                const uint4 v = g[gi];
                mx = fmaxf(mx, fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w))));
            }
        }
    }
    const float m = (mx > -INFINITY) ? mx : 0.f;
    const unsigned long long L2E = pk(kLog2e, kLog2e), nm = pk(-m, -m);
    unsigned long long acc = pk(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kGMax; ++j) {
        const int gi = tid + j * kThreads;
        if (gi < ngroups) {
            float a[EPG];
            unpack<kBF16>(g[gi], a);                      // second read of the slice from shared memory
#pragma unroll
            for (int e = 0; e < EPG; e += 2) {
                const float2 y = upk(mul2(add2(pk(a[e], a[e + 1]), nm), L2E));
                acc = add2(acc, pk(fast_exp2(y.x), fast_exp2(y.y)));
            }
        }
    }
    m_out = m;
    s_out = upk(acc).x + upk(acc).y;
}

template <bool kBF16, bool kLoss>
__global__ void __launch_bounds__(kThreads, 1)
tv_kernel(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star,
          int64_t rows, int V, int slice, StatusBlock* status, LossArgs la) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ;
    extern __shared__ __align__(128) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cs = static_cast<int>(cluster.num_blocks());
    const uint32_t rank = cluster.block_rank();
    const int64_t cid = blockIdx.x / cs;
    const int64_t ncl = gridDim.x / cs;
    const int lo = static_cast<int>(rank) * slice;
    const int len = max(0, min(V, lo + slice) - lo);
    const uint32_t bytes = static_cast<uint32_t>(len) * ESZ;
    const int ngroups = len / EPG;
    const size_t slot_bytes = static_cast<size_t>(slice) * ESZ;
    const int64_t my_rows = (cid < rows) ? (rows - 1 - cid) / ncl + 1 : 0;
    const int64_t Q = 2 * my_rows;                        // slices this CTA streams: d_0, t_0, d_1, ...

    // shared memory: slots (each a multiple of 16 bytes) | mbarriers (32 B) |
    // red_ab, red_c (16-byte aligned float4 per warp) | exchange slot
    uint8_t* buf = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSlots * slot_bytes);
    float4* red_ab = reinterpret_cast<float4*>(smem + kSlots * slot_bytes + 32);   // (md, sd, mt, st) per warp
    float4* red_c = red_ab + kWarps;                                               // pass C partials per warp
    Slot* slot = reinterpret_cast<Slot*>(red_c + kWarps);

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    // slice q: tensor q & 1 (d, t) of this cluster's row q >> 1, in slot q % kSlots
    auto issue = [&](int64_t q) {
        const int s = static_cast<int>(q % kSlots);
        const int64_t row = cid + (q >> 1) * ncl;
        mbar_arrive_expect_tx(&bars[s], bytes);
        if (bytes) {
            const uint8_t* src = (q & 1) ? t : d;
            bulk_g2s(buf + s * slot_bytes, src + (static_cast<size_t>(row) * V + lo) * ESZ, bytes, &bars[s], pol);
        }
    };
    int64_t q_issued = Q < kSlots ? Q : kSlots;           // slices issued so far (same value in every thread)
    int64_t q_landed = 0;                                 // slices waited for
    if (tid == 0)
        for (int64_t q = 0; q < q_issued; ++q) issue(q);

    bool failed = false;
    auto wait_slice = [&](int64_t q) {
        bool bad = false;
        if (!failed) {
            bad = !mbar_wait(&bars[q % kSlots], static_cast<uint32_t>(q / kSlots) & 1u);
            if (!bad) q_landed = q + 1;
        }
        if (__syncthreads_or(bad)) {
            if (!failed && tid == 0) set_status(status, DSPARK_ERR_TIMEOUT, 1);
            failed = true;
        }
    };

    float cl_sum = 0.f;                                   // loss mode: this cluster's row totals, in row order
    int64_t prev_row = -1;                                // row whose partials wait in the slots
    int it = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++it) {
        const int64_t qd = 2 * static_cast<int64_t>(it), qt = qd + 1;
        const uint4* dg = reinterpret_cast<const uint4*>(buf + (qd % kSlots) * slot_bytes);
        const uint4* tg = reinterpret_cast<const uint4*>(buf + (qt % kSlots) * slot_bytes);

        // AB: the slices' (max, sum) of d, then of t
        wait_slice(qd);
        float md = 0.f, sd = 0.f, mt = 0.f, st = 0.f;
        if (!failed) thread_lse<kBF16>(dg, ngroups, tid, md, sd);
        // loss mode: the target's logit, from the CTA whose slice holds it
        int tgt = -1;
        float dtgt = -INFINITY;
        if constexpr (kLoss) {
            tgt = la.target[row];
            if (tgt < 0 || tgt >= V) {
                if (tid == 0 && rank == 0) set_status(status, DSPARK_ERR_DEVICE_CHECK, 30);
                tgt = -1;
            }
            if (tid == 0 && !failed && tgt >= lo && tgt < lo + len) {
                const uint8_t* src = reinterpret_cast<const uint8_t*>(dg) + static_cast<size_t>(tgt - lo) * ESZ;
                dtgt = kBF16 ? bf16lo(*reinterpret_cast<const uint16_t*>(src)) : *reinterpret_cast<const float*>(src);
            }
        }
        warp_lse(md, sd);
        wait_slice(qt);
        if (!failed) thread_lse<kBF16>(tg, ngroups, tid, mt, st);
        warp_lse(mt, st);
        if (lane == 0) red_ab[warp] = make_float4(md, sd, mt, st);
        __syncthreads();
        if (warp == 0) {
            const float4 r = lane < kWarps ? red_ab[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            float a = r.x, b = r.y, c = r.z, e = r.w;
            warp_lse(a, b);
            warp_lse(c, e);
            if (lane == 0) slot->ms[it & 1] = make_float4(a, b, c, e);
        }
        cluster.sync();                                   // slices' (m, s) and the previous row's partials

        // the previous row's c*: rank 0 sums its CTAs' partials in rank order
        if (!kLoss && rank == 0 && warp == 1 && prev_row >= 0) {
            const float pr = (lane < cs) ? cluster.map_shared_rank(slot, lane)->p[(it - 1) & 1] : 0.f;
            const float c = warp_sum(pr);
            if (lane == 0 && !failed) c_star[prev_row] = c;
        }
        // every warp combines the cs slots itself: lane r reads CTA r's slot
        float rmd = -INFINITY, rsd = 0.f, rmt = -INFINITY, rst = 0.f;
        if (lane < cs) {
            const float4 rs = cluster.map_shared_rank(slot, lane)->ms[it & 1];
            rsd = rs.y; rst = rs.w;
            rmd = rsd > 0.f ? rs.x : -INFINITY;            // empty slices do not set the reference
            rmt = rst > 0.f ? rs.z : -INFINITY;
        }
        const float Md = warp_max(rmd), Mt = warp_max(rmt);
        const float Sd = warp_sum(rsd > 0.f ? rsd * fast_exp2((rmd - Md) * kLog2e) : 0.f);
        const float St = warp_sum(rst > 0.f ? rst * fast_exp2((rmt - Mt) * kLog2e) : 0.f);
        const float lsd = fast_log2(Sd) * kLn2, lst = fast_log2(St) * kLn2;
        const float Ld = Md + lsd, Lt = Mt + lst;         // natural-log logsumexp
        // p_d < p_t  <=>  d - t < L_d - L_t: the difference of the two logsumexps formed
        // from their parts, so that it keeps the precision of a small number
        const float dL = (Md - Mt) + (lsd - lst);

        // C: sum of 2^(min(d - L_d, t - L_t) log2e); loss mode also the p_d mass where
        // d - L_d < t - L_t and where they tie
        const unsigned long long L2E = pk(kLog2e, kLog2e), nLd = pk(-Ld, -Ld), nLt = pk(-Lt, -Lt);
        unsigned long long pc = pk(0.f, 0.f);
        float plt = 0.f, peq = 0.f;
        if (!failed) {
#pragma unroll
            for (int j = 0; j < kGMax; ++j) {
                const int gi = tid + j * kThreads;
                if (gi < ngroups) {
                    float a[EPG], b[EPG];
                    unpack<kBF16>(dg[gi], a);
                    unpack<kBF16>(tg[gi], b);
#pragma unroll
                    for (int e = 0; e < EPG; e += 2) {
                        const float2 x = upk(add2(pk(a[e], a[e + 1]), nLd));
                        const float2 y = upk(add2(pk(b[e], b[e + 1]), nLt));
                        const float2 z = upk(mul2(pk(fminf(x.x, y.x), fminf(x.y, y.y)), L2E));
                        const float e0 = fast_exp2(z.x), e1 = fast_exp2(z.y);
                        pc = add2(pc, pk(e0, e1));
                        if constexpr (kLoss) {
                            const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                            plt += (r0 < dL ? e0 : 0.f) + (r1 < dL ? e1 : 0.f);
                            peq += (r0 == dL ? e0 : 0.f) + (r1 == dL ? e1 : 0.f);
                        }
                    }
                }
            }
        }
        const float p = warp_sum(upk(pc).x + upk(pc).y);
        if constexpr (kLoss) {
            plt = warp_sum(plt);
            peq = warp_sum(peq);
        }
        if (lane == 0) red_c[warp] = make_float4(p, plt, peq, 0.f);
        __syncthreads();                                  // every thread is past pass C
        if constexpr (!kLoss) {
            // both slots of this row are free: refill them two slices ahead
            if (!failed) {
                const int64_t q_next = qd + kSlots + 2 < Q ? qd + kSlots + 2 : Q;
                if (tid == 0 && q_issued < q_next) {
                    fence_proxy_async_smem();
                    for (int64_t q = q_issued; q < q_next; ++q) issue(q);
                }
                if (q_issued < q_next) q_issued = q_next;
            }
            if (warp == 0) {
                const float q = warp_sum(lane < kWarps ? red_c[lane].x : 0.f);
                if (lane == 0) slot->p[it & 1] = q;
            }
        } else {
            if (warp == 0) {
                const float4 r = lane < kWarps ? red_c[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float q0 = warp_sum(r.x), q1 = warp_sum(r.y), q2 = warp_sum(r.z);
                if (lane == 0) slot->q[it & 1] = make_float4(q0, q1, q2, dtgt);
            }
            cluster.sync();                               // this row's partials, every CTA
            float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = -INFINITY;
            if (lane < cs) {
                const float4 rq = cluster.map_shared_rank(slot, lane)->q[it & 1];
                c0 = rq.x; c1 = rq.y; c2 = rq.z; c3 = rq.w;
            }
            // the same sums, in rank order, in every warp
            const float cstar = warp_sum(c0), p_lt = warp_sum(c1), p_eq = warp_sum(c2), dt_t = warp_max(c3);
            const float sbar = 1.f - 2.f * p_lt - p_eq;   // sum_u p_d(u) sign(p_d(u) - p_t(u))
            const float om = la.omega[row];
            // D: dL/dd from shared memory
            if (la.grad != nullptr && !failed) {
                const float ka = om * la.a_ce, kl = 0.5f * om * la.a_l1;
#pragma unroll
                for (int j = 0; j < kGMax; ++j) {
                    const int gi = tid + j * kThreads;
                    if (gi < ngroups) {
                        float a[EPG], b[EPG], gv[EPG];
                        unpack<kBF16>(dg[gi], a);
                        unpack<kBF16>(tg[gi], b);
#pragma unroll
                        for (int e = 0; e < EPG; e += 2) {
                            const float2 z = upk(mul2(add2(pk(a[e], a[e + 1]), nLd), L2E));
                            const float p0 = fast_exp2(z.x), p1 = fast_exp2(z.y);
                            const float r0 = a[e] - b[e], r1 = a[e + 1] - b[e + 1];
                            const float sg0 = r0 > dL ? 1.f : (r0 < dL ? -1.f : 0.f);
                            const float sg1 = r1 > dL ? 1.f : (r1 < dL ? -1.f : 0.f);
                            const int v = lo + gi * EPG + e;
                            gv[e] = ka * (p0 - (v == tgt ? 1.f : 0.f)) + kl * p0 * (sg0 - sbar);
                            gv[e + 1] = ka * (p1 - (v + 1 == tgt ? 1.f : 0.f)) + kl * p1 * (sg1 - sbar);
                        }
                        uint8_t* dst = static_cast<uint8_t*>(la.grad) + (static_cast<size_t>(row) * V + lo + gi * EPG) * ESZ;
                        if constexpr (kBF16) {
                            uint4 o;
                            o.x = pack_bf16(gv[0], gv[1]); o.y = pack_bf16(gv[2], gv[3]);
                            o.z = pack_bf16(gv[4], gv[5]); o.w = pack_bf16(gv[6], gv[7]);
                            *reinterpret_cast<uint4*>(dst) = o;
                        } else {
                            *reinterpret_cast<float4*>(dst) = make_float4(gv[0], gv[1], gv[2], gv[3]);
                        }
                    }
                }
            }
            if (rank == 0 && tid == 0 && !failed) {
                const float sv = la.s[row];
                const float ce = Ld - dt_t;
                const float sp = fmaxf(sv, 0.f) + log1pf(expf(-fabsf(sv)));   // softplus
                const float bce = sp - cstar * sv;
                const float tot = om * (la.a_ce * ce + la.a_l1 * (1.f - cstar) + la.a_conf * bce);
                reinterpret_cast<float4*>(la.row_out)[row] = make_float4(ce, cstar, bce, tot);
                if (la.grad_s != nullptr) la.grad_s[row] = om * la.a_conf * (1.f / (1.f + expf(-sv)) - cstar);
                cl_sum += tot;
            }
            __syncthreads();                              // every thread is past pass D
            if (!failed) {
                const int64_t q_next = qd + kSlots + 2 < Q ? qd + kSlots + 2 : Q;
                if (tid == 0 && q_issued < q_next) {
                    fence_proxy_async_smem();
                    for (int64_t q = q_issued; q < q_next; ++q) issue(q);
                }
                if (q_issued < q_next) q_issued = q_next;
            }
        }
        prev_row = row;
    }
    // the last row's c*, and no CTA leaves while a peer may still read its shared memory
    cluster.sync();
    if (!kLoss && rank == 0 && warp == 1 && prev_row >= 0) {
        const float pr = (lane < cs) ? cluster.map_shared_rank(slot, lane)->p[(it - 1) & 1] : 0.f;
        const float c = warp_sum(pr);
        if (lane == 0 && !failed) c_star[prev_row] = c;
    }
    if constexpr (kLoss) {
        // the loss: each cluster's sum of its rows, then the last cluster to finish adds
        // the clusters' sums in cluster order
        if (rank == 0 && tid == 0) {
            la.cl_part[cid] = cl_sum;
            __threadfence();
            const bool last = atomicAdd(la.cl_done, 1u) == static_cast<unsigned>(ncl) - 1u;
            if (last) {
                __threadfence();
                float tot = 0.f;
                for (int64_t c = 0; c < ncl; ++c) tot += __ldcg(la.cl_part + c);
                *la.loss = tot;
            }
        }
    }
    cluster.sync();
    // after a timeout, give every copy still in flight a bounded chance to land
    if (failed && tid == 0)
        for (int64_t q = q_landed; q < q_issued; ++q)
            mbar_wait(&bars[q % kSlots], static_cast<uint32_t>(q / kSlots) & 1u);
}

// Shared memory beyond the slots: mbarriers, two float4 per warp, the exchange slot, slack.
constexpr size_t kTvExtraSmem = 32 + 2 * kWarps * sizeof(float4) + sizeof(Slot) + 128;

// The cluster size: the smallest of 1, 2, 4, 8, 16 whose slices fit three slots in
// shared memory.  Returns 0 if none does.
template <bool kBF16>
int tv_cluster_size(int V, int* slice_out) {
    using Tr = TVTraits<kBF16>;
    for (int cs = 1; cs <= kMaxCS; cs *= 2) {
        const int per = (V + cs - 1) / cs;
        const int slice = (per + Tr::kEPG - 1) / Tr::kEPG * Tr::kEPG;
        if (kSlots * static_cast<size_t>(slice) * Tr::kESZ + kTvExtraSmem <= kSmemCap) {
            *slice_out = slice;
            return cs;
        }
    }
    return 0;
}

// Clusters of a loss launch are at most this many (their partial sums live in
// the workspace).
constexpr int kMaxLossClusters = 1024;

template <bool kBF16, bool kLoss>
dspark_status_t launch_tv(int64_t rows, int V, const void* d, const void* t, float* c_star,
                          StatusBlock* status, const LossArgs& la, cudaStream_t stream) {
    using Tr = TVTraits<kBF16>;
    int slice = 0;
    const int cs = tv_cluster_size<kBF16>(V, &slice);
    if (cs == 0) return DSPARK_ERR_UNSUPPORTED;
    if (slice / Tr::kEPG > kGMax * kThreads) return DSPARK_ERR_UNSUPPORTED;
    const size_t smem = kSlots * static_cast<size_t>(slice) * Tr::kESZ + kTvExtraSmem;
    const int dev = current_device();
    auto* kern = tv_kernel<kBF16, kLoss>;
    static OncePerDevice once;
    if (once.run(dev, [kern] {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(kSmemCap));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            return e;
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(cs * 256);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters < 1) {
        cudaGetLastError();
        max_clusters = sm_count(dev) / cs;
        if (max_clusters < 1) max_clusters = 1;
    }
    if (max_clusters > kMaxLossClusters) max_clusters = kMaxLossClusters;
    const int64_t ncl = rows < max_clusters ? rows : max_clusters;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs));
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(d),
                                             static_cast<const uint8_t*>(t), c_star, rows, V, slice,
                                             status, la);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// ------------------------------------------------------- accept rate, two passes
// dspark_accept_rate_tv's kernel: one CTA of 1024 threads per SM takes rows in
// turn.  Pass 1 streams the row's d and t from HBM (L2 evict-last) and forms each
// thread's online (max, sum of 2^((x - max) log2e)) of both; a block reduction
// gives L_d and L_t; pass 2 streams the same row again -- from L2, where pass 1
// left it (a CTA's row is 607,744 B for bf16 and V = 151936, so one row per SM,
// 92 MB in all, stays within the L2) -- with the evict-first policy, summing
// 2^(min(d - L_d, t - L_t) log2e).  No clusters, and each logit pair costs about
// half the instructions of the single-pass kernel's three readings of shared
// memory.
//
// Loads: every thread copies its own 16-byte groups into its own slots of a ring
// in shared memory with cp.async (no block barrier guards a slot: only the thread
// that copied it reads it), kTv2Stages - 1 groups of d and of t ahead of the one
// it is summing: 96 KB in flight per SM.
constexpr int kTv2Threads = 1024;
constexpr int kTv2Stages = 4;
constexpr size_t kTv2Smem = static_cast<size_t>(kTv2Stages) * 2 * kTv2Threads * 16;

// The group's max (raw units), -inf if it has no finite element.
template <bool kBF16>
__device__ __forceinline__ float group_max(const uint4 v) {
    if constexpr (kBF16) {
        const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
        return fmaxf(bf16lo(m), bf16hi(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}

// (m, s) += the group's elements, s a sum of 2^((x - m) log2e): a larger group
// max first rescales s (rare once m has settled).  For bf16 the exponent is one
// fused x log2e - (m log2e): every term carries the rounding error r of m log2e
// (|r| <= ulp(m log2e) / 2, a relative 1e-5 at |m| = 100, inside the bf16 bound).
// For float32, whose bound is tighter, x - m is formed first, so the maximum's
// term is exactly 1.
template <bool kBF16>
__device__ __forceinline__ void group_lse(const uint4 v, float& m, float& s) {
    constexpr int EPG = TVTraits<kBF16>::kEPG;
    const float gm = group_max<kBF16>(v);
    if (!(gm > -INFINITY)) return;                        // no mass in this group
    if (gm > m) {
        s = (s > 0.f) ? s * fast_exp2((m - gm) * kLog2e) : 0.f;
        m = gm;
    }
    float a[EPG];
    unpack<kBF16>(v, a);
    const unsigned long long L2E = pk(kLog2e, kLog2e);
    const unsigned long long nm = kBF16 ? pk(-m * kLog2e, -m * kLog2e) : pk(-m, -m);
    unsigned long long acc = pk(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < EPG; e += 2) {
        const float2 y = kBF16 ? upk(fma2(pk(a[e], a[e + 1]), L2E, nm)) : upk(mul2(add2(pk(a[e], a[e + 1]), nm), L2E));
        acc = add2(acc, pk(fast_exp2(y.x), fast_exp2(y.y)));
    }
    s += upk(acc).x + upk(acc).y;
}

// Block-wide merge of every thread's (m, s) pair for d and t: all threads get (L_d, L_t)
// in natural units.
__device__ __forceinline__ float2 block_lse2(float md, float sd, float mt, float st, float4* red, float2* fin) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_lse(md, sd);
    warp_lse(mt, st);
    if (lane == 0) red[warp] = make_float4(md, sd, mt, st);
    __syncthreads();
    if (warp == 0) {
        float4 r = (lane < kTv2Threads / 32) ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        warp_lse(r.x, r.y);
        warp_lse(r.z, r.w);
        if (lane == 0) {
            const float Ld = (r.y > 0.f) ? r.x + fast_log2(r.y) * kLn2 : -INFINITY;
            const float Lt = (r.w > 0.f) ? r.z + fast_log2(r.w) * kLn2 : -INFINITY;
            *fin = make_float2(Ld, Lt);
        }
    }
    __syncthreads();
    return *fin;
}

// One 16-byte asynchronous copy global -> shared with an L2 policy (cp.async.cg).
__device__ __forceinline__ void cp16_hint(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One pass over a row: a thread's groups i = 0 .. nmine - 1 (group tid + i T) of d
// and t go through its ring, copied kTv2Stages - 1 groups ahead of the one that
// body(vd, vt) sums.  Each issue commits one cp.async group, empty past the last,
// so that "group i has landed" is always wait_group(S - 2) after i + S - 1 commits.
template <class F>
__device__ __forceinline__ void tv2_pass(const uint4* gd, const uint4* gt, int nmine, uint4* ring, uint64_t pol,
                                         F&& body) {
    const int tid = threadIdx.x;
    auto issue = [&](int i) {
        if (i < nmine) {
            const int g = tid + i * kTv2Threads;
            uint4* slot = ring + static_cast<size_t>(i % kTv2Stages) * 2 * kTv2Threads + tid;
            cp16_hint(slot, gd + g, pol);
            cp16_hint(slot + kTv2Threads, gt + g, pol);
        }
        cp_commit();
    };
#pragma unroll
    for (int i = 0; i < kTv2Stages - 1; ++i) issue(i);
    for (int i = 0; i < nmine; ++i) {
        cp_wait<kTv2Stages - 2>();                        // group i has landed
        const uint4* slot = ring + static_cast<size_t>(i % kTv2Stages) * 2 * kTv2Threads + tid;
        const uint4 vd = slot[0], vt = slot[kTv2Threads];
        issue(i + kTv2Stages - 1);                        // refills the slot read one group ago
        body(vd, vt);
    }
    cp_wait<0>();
}

template <bool kBF16>
__global__ void __launch_bounds__(kTv2Threads, 1)
tv_two_pass(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star, int64_t rows,
            int V) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ;
    extern __shared__ __align__(16) uint8_t tv2_smem[];
    uint4* ring = reinterpret_cast<uint4*>(tv2_smem);
    __shared__ float4 red[kTv2Threads / 32];
    __shared__ float2 fin;
    __shared__ float red2[kTv2Threads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ngroups = V / EPG;
    const int nmine = (ngroups > tid) ? (ngroups - tid + kTv2Threads - 1) / kTv2Threads : 0;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint4* gd = reinterpret_cast<const uint4*>(d + static_cast<size_t>(row) * V * ESZ);
        const uint4* gt = reinterpret_cast<const uint4*>(t + static_cast<size_t>(row) * V * ESZ);
        // pass 1: (max, sum) of d and t, from HBM
        float md = -INFINITY, sd = 0.f, mt = -INFINITY, st = 0.f;
        tv2_pass(gd, gt, nmine, ring, keep, [&](const uint4 vd, const uint4 vt) {
            group_lse<kBF16>(vd, md, sd);
            group_lse<kBF16>(vt, mt, st);
        });
        if (!(md > -INFINITY)) { md = 0.f; sd = 0.f; }
        if (!(mt > -INFINITY)) { mt = 0.f; st = 0.f; }
        const float2 L = block_lse2(md, sd, mt, st, red, &fin);
        // pass 2: sum of 2^(min(d - L_d, t - L_t) log2e), from L2 (for bf16 the
        // exponents are the fused d log2e - L_d log2e and t log2e - L_t log2e)
        unsigned long long acc = pk(0.f, 0.f);
        if (L.x > -INFINITY && L.y > -INFINITY) {
            const unsigned long long L2E = pk(kLog2e, kLog2e);
            const float sc = kBF16 ? kLog2e : 1.f;
            const unsigned long long nLd = pk(-L.x * sc, -L.x * sc), nLt = pk(-L.y * sc, -L.y * sc);
            tv2_pass(gd, gt, nmine, ring, drop, [&](const uint4 vd, const uint4 vt) {
                float a[EPG], b[EPG];
                unpack<kBF16>(vd, a);
                unpack<kBF16>(vt, b);
#pragma unroll
                for (int e = 0; e < EPG; e += 2) {
                    if constexpr (kBF16) {
                        const float2 x = upk(fma2(pk(a[e], a[e + 1]), L2E, nLd));
                        const float2 y = upk(fma2(pk(b[e], b[e + 1]), L2E, nLt));
                        acc = add2(acc, pk(fast_exp2(fminf(x.x, y.x)), fast_exp2(fminf(x.y, y.y))));
                    } else {
                        const float2 x = upk(add2(pk(a[e], a[e + 1]), nLd));
                        const float2 y = upk(add2(pk(b[e], b[e + 1]), nLt));
                        const float2 z = upk(mul2(pk(fminf(x.x, y.x), fminf(x.y, y.y)), L2E));
                        acc = add2(acc, pk(fast_exp2(z.x), fast_exp2(z.y)));
                    }
                }
            });
        }
        float part = upk(acc).x + upk(acc).y;
        part = warp_sum(part);
        if (lane == 0) red2[warp] = part;
        __syncthreads();
        if (warp == 0) {
            float v = (lane < kTv2Threads / 32) ? red2[lane] : 0.f;
            v = warp_sum(v);
            if (lane == 0) c_star[row] = v;
        }
        // red, fin and red2 are rewritten by the next row after a barrier in block_lse2
    }
}

template <bool kBF16>
dspark_status_t launch_tv_two_pass(int64_t rows, int V, const void* d, const void* t, float* c_star,
                                   cudaStream_t stream) {
    const int dev = current_device();
    static OncePerDevice once;
    if (once.run(dev, [] {
            return cudaFuncSetAttribute(tv_two_pass<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kTv2Smem));
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    const int sms = sm_count(dev);
    const int64_t grid = rows < sms ? rows : sms;
    tv_two_pass<kBF16><<<static_cast<unsigned>(grid), kTv2Threads, kTv2Smem, stream>>>(
        static_cast<const uint8_t*>(d), static_cast<const uint8_t*>(t), c_star, rows, V);
    return launch_status();
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_accept_rate_tv_workspace_size(int64_t rows, int V) {
    (void)rows;
    (void)V;
    return kStatusBytes;
}

extern "C" dspark_status_t dspark_accept_rate_tv(int64_t rows, int V, dspark_dtype_t dt, const void* d,
                                                 const void* t, float* c_star, void* workspace,
                                                 size_t workspace_bytes, dspark_stream_t stream) {
    if (rows < 0 || V <= 0 || (dt != DSPARK_F32 && dt != DSPARK_BF16)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_accept_rate_tv_workspace_size(rows, V)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    if (rows == 0) return DSPARK_OK;
    if (d == nullptr || t == nullptr || c_star == nullptr) return DSPARK_ERR_INVALID_ARGUMENT;
    if (!aligned16(d) || !aligned16(t)) return DSPARK_ERR_INVALID_ARGUMENT;
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_status(workspace, s) != DSPARK_OK) return DSPARK_ERR_CUDA;
    return dt == DSPARK_BF16 ? launch_tv_two_pass<true>(rows, V, d, t, c_star, s)
                             : launch_tv_two_pass<false>(rows, V, d, t, c_star, s);
}

// Workspace of the loss: status block | cluster counter (own 256 bytes) | one
// float per cluster.
extern "C" size_t dspark_training_loss_workspace_size(int64_t rows, int V) {
    (void)rows;
    (void)V;
    return kStatusBytes + 256 + static_cast<size_t>(kMaxLossClusters) * sizeof(float);
}

extern "C" dspark_status_t dspark_training_loss(int64_t rows, int V, dspark_dtype_t dt, const void* d,
                                                const void* t, const int32_t* target, const float* conf_logit,
                                                const float* omega, float alpha_ce, float alpha_l1,
                                                float alpha_conf, float* row_out, float* loss, void* grad_d,
                                                float* grad_conf, void* workspace, size_t workspace_bytes,
                                                dspark_stream_t stream) {
    if (rows < 0 || V <= 0 || (dt != DSPARK_F32 && dt != DSPARK_BF16)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V % (dt == DSPARK_BF16 ? 8 : 4) != 0) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < dspark_training_loss_workspace_size(rows, V)) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    if (loss == nullptr) return DSPARK_ERR_INVALID_ARGUMENT;
    if (V > 163840) return DSPARK_ERR_UNSUPPORTED;
    if (rows > 0) {
        if (d == nullptr || t == nullptr || target == nullptr || conf_logit == nullptr || omega == nullptr ||
            row_out == nullptr)
            return DSPARK_ERR_INVALID_ARGUMENT;
        if (!aligned16(d) || !aligned16(t) || !aligned16(row_out)) return DSPARK_ERR_INVALID_ARGUMENT;
        if (grad_d != nullptr && !aligned16(grad_d)) return DSPARK_ERR_INVALID_ARGUMENT;
    }
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // status and the cluster counter
    if (cudaMemsetAsync(workspace, 0, kStatusBytes + 256, s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (rows == 0) return cudaMemsetAsync(loss, 0, sizeof(float), s) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
    StatusBlock* st = static_cast<StatusBlock*>(workspace);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    LossArgs la{};
    la.target = target;
    la.s = conf_logit;
    la.omega = omega;
    la.a_ce = alpha_ce;
    la.a_l1 = alpha_l1;
    la.a_conf = alpha_conf;
    la.row_out = row_out;
    la.grad = grad_d;
    la.grad_s = grad_conf;
    la.cl_done = reinterpret_cast<unsigned int*>(base + kStatusBytes);
    la.cl_part = reinterpret_cast<float*>(base + kStatusBytes + 256);
    la.loss = loss;
    return dt == DSPARK_BF16 ? launch_tv<true, true>(rows, V, d, t, nullptr, st, la, s)
                             : launch_tv<false, true>(rows, V, d, t, nullptr, st, la, s);
}
