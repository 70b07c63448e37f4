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
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// One CTA's exchange slot, double-buffered by row parity: a CTA writes row it+1's
// values only after the cluster barrier of row it+1, which every CTA reaches
// only after its reads of row it-1's values, so parity it+1 is free.
struct Slot {
    float4 ms[2];           // slice max (log2 units) and sum of 2^(y - m) of d and t: (md, sd, mt, st)
    float p[2];             // CTA partial of sum min(p_d, p_t)
    float pad[2];
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

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
tv_kernel(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star,
          int64_t rows, int V, int slice, StatusBlock* status) {
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
        if (rank == 0 && warp == 1 && prev_row >= 0) {
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
        unsigned long long pp = pk(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < GMAX * EPG / 2; ++i) {
            const float2 x = upk(mul2(ed[i], al)), y = upk(mul2(et[i], be));
            pp = add2(pp, pk(fminf(x.x, y.x), fminf(x.y, y.y)));
        }
        float p = warp_sum(upk(pp).x + upk(pp).y);
        __syncthreads();                                  // red is free again
        if (lane == 0) red[warp].x = p;
        __syncthreads();
        if (warp == 0) {
            float q = (lane < kWarps) ? red[lane].x : 0.f;
            q = warp_sum(q);
            if (lane == 0) slot->p[it & 1] = q;
        }
        prev_row = row;
    }
    // the last row's c*, and no CTA leaves while a peer may still read its shared memory
    cluster.sync();
    if (rank == 0 && warp == 1 && prev_row >= 0) {
        const float pr = (lane < kCS) ? cluster.map_shared_rank(slot, lane)->p[(it - 1) & 1] : 0.f;
        const float c = warp_sum(pr);
        if (lane == 0 && !failed) c_star[prev_row] = c;
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

template <bool kBF16>
dspark_status_t launch_tv(int64_t rows, int V, const void* d, const void* t, float* c_star,
                          StatusBlock* status, cudaStream_t stream) {
    using Tr = TVTraits<kBF16>;
    const int per = (V + kCS - 1) / kCS;
    const int slice = (per + Tr::kEPG - 1) / Tr::kEPG * Tr::kEPG;
    if (slice / Tr::kEPG > Tr::kGMax * kThreads) return DSPARK_ERR_UNSUPPORTED;
    const size_t smem = tv_smem_bytes<kBF16>(slice);
    if (smem > 227 * 1024) return DSPARK_ERR_UNSUPPORTED;
    const int dev = current_device();
    static OncePerDevice once;
    if (once.run(dev, [] {
            return cudaFuncSetAttribute(tv_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        227 * 1024);
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
    if (cudaOccupancyMaxActiveClusters(&max_clusters, tv_kernel<kBF16>, &cfg) != cudaSuccess ||
        max_clusters < 1) {
        cudaGetLastError();
        max_clusters = sm_count(dev) / kCS;
        if (max_clusters < 1) max_clusters = 1;
    }
    const int64_t ncl = rows < max_clusters ? rows : max_clusters;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * kCS));
    const cudaError_t e = cudaLaunchKernelEx(&cfg, tv_kernel<kBF16>, static_cast<const uint8_t*>(d),
                                             static_cast<const uint8_t*>(t), c_star, rows, V, slice,
                                             status);
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
    return dt == DSPARK_BF16 ? launch_tv<true>(rows, V, d, t, c_star, st, s)
                             : launch_tv<false>(rows, V, d, t, c_star, st, s);
}
