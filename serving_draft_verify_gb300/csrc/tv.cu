// dspark_accept_rate_tv: c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 per row
// (DeepSpec walkthrough, section 3.3, paper eq. 8 / `_compute_accept_rate_3d`),
// computed as sum_v min(p_d(v), p_t(v)).
//
// One HBM pass per row.  A thread-block cluster of kCS CTAs owns one row at a
// time; each CTA bulk-copies its 1/kCS slice of d and t into shared memory
// (double-buffered, so the next row streams in while this one is reduced):
//   A. each thread's max of its d and t elements (packed bf16 max);
//   B. e_d = 2^(d log2e - m_d), e_t likewise, kept in registers as packed
//      float pairs; the thread's sums, merged per warp and per CTA;
//   -- one cluster barrier per row: the CTAs' (m, s) through distributed shared
//      memory (and the previous row's partials, which rank 0 sums into c*) --
//   C. sum min(e_d 2^(m_d - L_d), e_t 2^(m_t - L_t)) from registers (no exp).
// Two exponentials per logit pair; every byte of d and t is read once from HBM.
#include <cooperative_groups.h>

#include "common.cuh"
#include "host_common.h"

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kCS = 8;          // CTAs per cluster (one row per cluster)
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

template <bool kBF16>
struct TVTraits {
    static constexpr int kEPG = kBF16 ? 8 : 4;   // elements per 16-byte group
    static constexpr int kESZ = kBF16 ? 2 : 4;
    static constexpr int kStages = kBF16 ? 2 : 1;     // at most 2: their mbarriers fit in 16 bytes
    static constexpr int kGMax = kBF16 ? 5 : 10;  // groups per thread held in registers
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

// One CTA's exchange slot, double-buffered by row parity: a CTA writes row it+1's
// values only after the cluster barrier of row it+1, which every CTA reaches
// only after its reads of row it-1's values, so parity it+1 is free.
struct Slot {
    float4 ms[2];           // slice max and sum of 2^((x - m) log2e) of d and t: (md, sd, mt, st)
    float4 q[2];            // loss mode: partials (sum min(p_d, p_t), sum p_d sign(p_d - p_t), d[target] or -inf)
    float p[2];             // CTA partial of sum min(p_d, p_t)
    float pad[2];
};

// The training loss (loss mode of the kernel): per row, with p = softmax,
//   ce = logsumexp(d) - d[target], c* = sum min(p_d, p_t), l1 = 1 - c*,
//   bce = softplus(s) - c* s, row = omega (a_ce ce + a_l1 l1 + a_conf bce),
//   dL/dd_v = omega (a_ce (p_d(v) - [v = target]) + a_l1 / 2 p_d(v) (sgn_v - sum_u p_d(u) sgn_u)),
//   dL/ds = omega a_conf (sigmoid(s) - c*), sgn_v = sign(p_d(v) - p_t(v)).
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

// (m, s) with s a sum of 2^((x - m) log2e): merge across a warp.
__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        if (os > 0.f) {
            if (s <= 0.f) { m = om; s = os; }
            else {
                const float M = fmaxf(m, om);
                s = s * fast_exp2((m - M) * kLog2e) + os * fast_exp2((om - M) * kLog2e);
                m = M;
            }
        }
    }
}

template <bool kBF16, bool kLoss>
__global__ void __launch_bounds__(kThreads, 1)
tv_kernel(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star,
          int64_t rows, int V, int slice, StatusBlock* status, LossArgs la) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ, STAGES = Tr::kStages, GMAX = Tr::kGMax;
    extern __shared__ __align__(128) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster.block_rank();
    const int64_t cid = blockIdx.x / kCS;
    const int64_t ncl = gridDim.x / kCS;
    const int lo = static_cast<int>(rank) * slice;
    const int len = max(0, min(V, lo + slice) - lo);
    const uint32_t bytes = static_cast<uint32_t>(len) * ESZ;
    const int ngroups = len / EPG;
    const size_t stage_bytes = static_cast<size_t>(slice) * ESZ;

    // shared memory: data stages (each a multiple of 16 bytes) | mbarriers (16 B) | pad |
    // red (16-byte aligned float4 per warp) | slot
    uint8_t* buf = smem;
    const size_t data_bytes = static_cast<size_t>(STAGES) * 2 * stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + data_bytes);
    float4* red = reinterpret_cast<float4*>(smem + data_bytes + 32);   // (md, sd, mt, st) / partials
    Slot* slot = reinterpret_cast<Slot*>(red + kWarps);

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    int pend_it[STAGES];   // iteration whose copy is in flight on stage s, or -1
#pragma unroll
    for (int s = 0; s < STAGES; ++s) pend_it[s] = -1;
    auto issue = [&](int64_t row, int s) {
        mbar_arrive_expect_tx(&bars[s], 2 * bytes);
        if (bytes) {
            const size_t off = (static_cast<size_t>(row) * V + lo) * ESZ;
            bulk_g2s(buf + (2 * s) * stage_bytes, d + off, bytes, &bars[s], pol);
            bulk_g2s(buf + (2 * s + 1) * stage_bytes, t + off, bytes, &bars[s], pol);
        }
    };
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        const int64_t row = cid + s * ncl;
        if (row < rows) {
            if (tid == 0) issue(row, s);
            pend_it[s] = s;
        }
    }

    bool failed = false;
    int it = 0;
    int64_t prev_row = -1;                                // row whose partials wait in the slots
    float cl_sum = 0.f;                                   // loss mode: this cluster's row totals, in row order
    for (int64_t row = cid; row < rows; row += ncl, ++it) {
        const int s = it % STAGES;
        const uint32_t par = static_cast<uint32_t>(it / STAGES) & 1u;
        bool bad = false;
        if (!failed) {
            bad = !mbar_wait(&bars[s], par);
            if (!bad) pend_it[s] = -1;
        }
        if (__syncthreads_or(bad)) {
            if (!failed && tid == 0) set_status(status, DSPARK_ERR_TIMEOUT, 1);
            failed = true;
        }
        const uint4* dg = reinterpret_cast<const uint4*>(buf + (2 * s) * stage_bytes);
        const uint4* tg = reinterpret_cast<const uint4*>(buf + (2 * s + 1) * stage_bytes);

        // A: this thread's maxima (bf16: packed, exact)
        float mxd = -INFINITY, mxt = -INFINITY;
        if constexpr (kBF16) {
            uint32_t ad = 0xFF80FF80u, at = 0xFF80FF80u;  // (-inf, -inf)
#pragma unroll
            for (int gi = 0; gi < GMAX; ++gi) {
                const int g = tid + gi * kThreads;
                if (!failed && g < ngroups) {
                    const uint4 a = dg[g], b = tg[g];
                    ad = bmax2(bmax2(ad, a.x), bmax2(a.y, bmax2(a.z, a.w)));
                    at = bmax2(bmax2(at, b.x), bmax2(b.y, bmax2(b.z, b.w)));
                }
            }
            mxd = fmaxf(bf16lo(ad), bf16hi(ad));
            mxt = fmaxf(bf16lo(at), bf16hi(at));
        } else {
#pragma unroll
            for (int gi = 0; gi < GMAX; ++gi) {
                const int g = tid + gi * kThreads;
                if (!failed && g < ngroups) {
                    float a[EPG], b[EPG];
                    unpack<kBF16>(dg[g], a);
                    unpack<kBF16>(tg[g], b);
#pragma unroll
                    for (int e = 0; e < EPG; ++e) { mxd = fmaxf(mxd, a[e]); mxt = fmaxf(mxt, b[e]); }
                }
            }
        }
        // e = 2^((x - m) log2e): the difference is formed first, so it is exactly 0 at
        // the max and <= 0 elsewhere, whatever the magnitude of x (a multiply-add of
        // x log2e - m log2e would leave the product's rounding error in the exponent);
        // a thread without a finite logit keeps reference 0 so that its terms are 0
        const float md = (mxd > -INFINITY) ? mxd : 0.f;
        const float mt = (mxt > -INFINITY) ? mxt : 0.f;
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
                const uint8_t* src = buf + (2 * s) * stage_bytes + static_cast<size_t>(tgt - lo) * ESZ;
                dtgt = kBF16 ? bf16lo(*reinterpret_cast<const uint16_t*>(src)) : *reinterpret_cast<const float*>(src);
            }
        }

        // B: e in registers (packed pairs), the thread's sums
        unsigned long long ed[GMAX * EPG / 2], et[GMAX * EPG / 2];
        const unsigned long long L2E = pk(kLog2e, kLog2e);
        const unsigned long long nmd = pk(-md, -md), nmt = pk(-mt, -mt);
        unsigned long long sdp = pk(0.f, 0.f), stp = pk(0.f, 0.f);
#pragma unroll
        for (int gi = 0; gi < GMAX; ++gi) {
            const int g = tid + gi * kThreads;
            if (!failed && g < ngroups) {
                float a[EPG], b[EPG];
                unpack<kBF16>(dg[g], a);
                unpack<kBF16>(tg[g], b);
#pragma unroll
                for (int e = 0; e < EPG; e += 2) {
                    const float2 ya = upk(mul2(add2(pk(a[e], a[e + 1]), nmd), L2E));
                    const float2 yb = upk(mul2(add2(pk(b[e], b[e + 1]), nmt), L2E));
                    const unsigned long long va = pk(fast_exp2(ya.x), fast_exp2(ya.y));
                    const unsigned long long vb = pk(fast_exp2(yb.x), fast_exp2(yb.y));
                    ed[(gi * EPG + e) / 2] = va;
                    et[(gi * EPG + e) / 2] = vb;
                    sdp = add2(sdp, va);
                    stp = add2(stp, vb);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPG; e += 2) { ed[(gi * EPG + e) / 2] = 0ull; et[(gi * EPG + e) / 2] = 0ull; }
            }
        }
        float tmd = md, tsd = upk(sdp).x + upk(sdp).y;
        float tmt = mt, tst = upk(stp).x + upk(stp).y;
        float wmd = tmd, wsd = tsd, wmt = tmt, wst = tst;
        warp_lse(wmd, wsd);
        warp_lse(wmt, wst);
        if (lane == 0) red[warp] = make_float4(wmd, wsd, wmt, wst);
        __syncthreads();                                  // every thread is past its reads of this stage

        // refill this stage with the row STAGES iterations ahead
        {
            const int64_t nrow = row + STAGES * ncl;
            if (!failed && nrow < rows) {
                if (tid == 0) {
                    fence_proxy_async_smem();
                    issue(nrow, s);
                }
                pend_it[s] = it + STAGES;
            }
        }
        if (warp == 0) {
            float4 r = (lane < kWarps) ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            float a = r.x, b = r.y, c = r.z, e = r.w;
            warp_lse(a, b);
            warp_lse(c, e);
            if (lane == 0) slot->ms[it & 1] = make_float4(a, b, c, e);
        }
        cluster.sync();                                   // slices' (m, s) and the previous row's partials

        // the previous row's c*: rank 0 sums its CTAs' partials in rank order
        if (!kLoss && rank == 0 && warp == 1 && prev_row >= 0) {
            const float pr = (lane < kCS) ? cluster.map_shared_rank(slot, lane)->p[(it - 1) & 1] : 0.f;
            const float c = warp_sum(pr);
            if (lane == 0 && !failed) c_star[prev_row] = c;
        }
        // every warp combines the kCS slots itself: lane r reads CTA r's slot
        float rmd = -INFINITY, rsd = 0.f, rmt = -INFINITY, rst = 0.f;
        if (lane < kCS) {
            const float4 rs = cluster.map_shared_rank(slot, lane)->ms[it & 1];
            rsd = rs.y; rst = rs.w;
            rmd = rsd > 0.f ? rs.x : -INFINITY;            // empty slices do not set the reference
            rmt = rst > 0.f ? rs.z : -INFINITY;
        }
        const float Md = warp_max(rmd), Mt = warp_max(rmt);
        const float Sd = warp_sum(rsd > 0.f ? rsd * exp2f((rmd - Md) * kLog2e) : 0.f);
        const float St = warp_sum(rst > 0.f ? rst * exp2f((rmt - Mt) * kLog2e) : 0.f);
        // p = e 2^((m_thread - M) log2e) / S
        const float alpha = (tsd > 0.f) ? exp2f((tmd - Md) * kLog2e - log2f(Sd)) : 0.f;
        const float beta = (tst > 0.f) ? exp2f((tmt - Mt) * kLog2e - log2f(St)) : 0.f;

        // C: sum of min(p_d, p_t) over this thread's elements, from registers
        const unsigned long long al = pk(alpha, alpha), be = pk(beta, beta);
        unsigned long long pp = pk(0.f, 0.f), sp = pk(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < GMAX * EPG / 2; ++i) {
            const float2 x = upk(mul2(ed[i], al)), y = upk(mul2(et[i], be));
            pp = add2(pp, pk(fminf(x.x, y.x), fminf(x.y, y.y)));
            if constexpr (kLoss) {
                const float s0 = x.x > y.x ? x.x : (x.x < y.x ? -x.x : 0.f);   // p_d sign(p_d - p_t)
                const float s1 = x.y > y.y ? x.y : (x.y < y.y ? -x.y : 0.f);
                sp = add2(sp, pk(s0, s1));
            }
        }
        float p = warp_sum(upk(pp).x + upk(pp).y);
        float sgs = kLoss ? warp_sum(upk(sp).x + upk(sp).y) : 0.f;
        __syncthreads();                                  // red is free again
        if (lane == 0) { red[warp].x = p; red[warp].y = sgs; }
        __syncthreads();
        if (warp == 0) {
            float q = (lane < kWarps) ? red[lane].x : 0.f;
            q = warp_sum(q);
            if constexpr (kLoss) {
                float q2 = (lane < kWarps) ? red[lane].y : 0.f;
                q2 = warp_sum(q2);
                if (lane == 0) slot->q[it & 1] = make_float4(q, q2, dtgt, 0.f);
            } else {
                if (lane == 0) slot->p[it & 1] = q;
            }
        }
        if constexpr (kLoss) {
            cluster.sync();                               // this row's partials, every CTA
            float c0 = 0.f, c1 = 0.f, c2 = -INFINITY;
            if (lane < kCS) {
                const float4 rq = cluster.map_shared_rank(slot, lane)->q[it & 1];
                c0 = rq.x; c1 = rq.y; c2 = rq.z;
            }
            // rank order within each reduction: every warp gets the same sums
            const float cstar = warp_sum(c0), sbar = warp_sum(c1), dt_t = warp_max(c2);
            // D: dL/dd from registers
            const float om = la.omega[row];
            if (la.grad != nullptr && !failed) {
                const float ka = om * la.a_ce, kl = 0.5f * om * la.a_l1;
#pragma unroll
                for (int gi = 0; gi < GMAX; ++gi) {
                    const int g = tid + gi * kThreads;
                    if (g < ngroups) {
                        float gv[EPG];
#pragma unroll
                        for (int e = 0; e < EPG; e += 2) {
                            const float2 x = upk(mul2(ed[(gi * EPG + e) / 2], al));
                            const float2 y = upk(mul2(et[(gi * EPG + e) / 2], be));
                            const float sg0 = x.x > y.x ? 1.f : (x.x < y.x ? -1.f : 0.f);
                            const float sg1 = x.y > y.y ? 1.f : (x.y < y.y ? -1.f : 0.f);
                            const int v = lo + g * EPG + e;
                            gv[e] = ka * (x.x - (v == tgt ? 1.f : 0.f)) + kl * x.x * (sg0 - sbar);
                            gv[e + 1] = ka * (x.y - (v + 1 == tgt ? 1.f : 0.f)) + kl * x.y * (sg1 - sbar);
                        }
                        uint8_t* dst = static_cast<uint8_t*>(la.grad) + (static_cast<size_t>(row) * V + lo + g * EPG) * ESZ;
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
            if (rank == 0 && warp == 0 && lane == 0 && !failed) {
                const float sv = la.s[row];
                const float ce = (Md + log2f(Sd) * kLn2) - dt_t;   // natural-log logsumexp minus d[target]
                const float sp_ = fmaxf(sv, 0.f) + log1pf(expf(-fabsf(sv)));
                const float bce = sp_ - cstar * sv;
                const float tot = om * (la.a_ce * ce + la.a_l1 * (1.f - cstar) + la.a_conf * bce);
                reinterpret_cast<float4*>(la.row_out)[row] = make_float4(ce, cstar, bce, tot);
                if (la.grad_s != nullptr) la.grad_s[row] = om * la.a_conf * (1.f / (1.f + expf(-sv)) - cstar);
                cl_sum += tot;
                if (c_star != nullptr) c_star[row] = cstar;
            }
        }
        prev_row = row;
    }
    // the last row's c*, and no CTA leaves while a peer may still read its shared memory
    cluster.sync();
    if (!kLoss && rank == 0 && warp == 1 && prev_row >= 0) {
        const float pr = (lane < kCS) ? cluster.map_shared_rank(slot, lane)->p[(it - 1) & 1] : 0.f;
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
    // after a timeout, give any copy still in flight a bounded chance to land
    if (failed && tid == 0) {
        for (int s = 0; s < STAGES; ++s)
            if (pend_it[s] >= 0) mbar_wait(&bars[s], static_cast<uint32_t>(pend_it[s] / STAGES) & 1u);
    }
}

template <bool kBF16>
size_t tv_smem_bytes(int slice) {
    using Tr = TVTraits<kBF16>;
    return static_cast<size_t>(Tr::kStages) * 2 * slice * Tr::kESZ + 32 + kWarps * sizeof(float4) +
           sizeof(Slot) + 128;
}

// Clusters of the loss launch are at most this many (their partial sums live in
// the workspace).
constexpr int kMaxLossClusters = 1024;

template <bool kBF16, bool kLoss>
dspark_status_t launch_tv(int64_t rows, int V, const void* d, const void* t, float* c_star,
                          StatusBlock* status, const LossArgs& la, cudaStream_t stream) {
    using Tr = TVTraits<kBF16>;
    const int per = (V + kCS - 1) / kCS;
    const int slice = (per + Tr::kEPG - 1) / Tr::kEPG * Tr::kEPG;
    if (slice / Tr::kEPG > Tr::kGMax * kThreads) return DSPARK_ERR_UNSUPPORTED;
    const size_t smem = tv_smem_bytes<kBF16>(slice);
    if (smem > 227 * 1024) return DSPARK_ERR_UNSUPPORTED;
    const int dev = current_device();
    auto* kern = tv_kernel<kBF16, kLoss>;
    static OncePerDevice once;
    if (once.run(dev, [kern] {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        }) != cudaSuccess)
        return DSPARK_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(kCS * 256);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters < 1) {
        cudaGetLastError();
        max_clusters = sm_count(dev) / kCS;
        if (max_clusters < 1) max_clusters = 1;
    }
    if (max_clusters > kMaxLossClusters) max_clusters = kMaxLossClusters;
    const int64_t ncl = rows < max_clusters ? rows : max_clusters;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * kCS));
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(d),
                                             static_cast<const uint8_t*>(t), c_star, rows, V, slice,
                                             status, la);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
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
    if (V > 163840) return DSPARK_ERR_UNSUPPORTED;
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_status(workspace, s) != DSPARK_OK) return DSPARK_ERR_CUDA;
    StatusBlock* st = static_cast<StatusBlock*>(workspace);
    const LossArgs none{};
    return dt == DSPARK_BF16 ? launch_tv<true, false>(rows, V, d, t, c_star, st, none, s)
                             : launch_tv<false, false>(rows, V, d, t, c_star, st, none, s);
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
