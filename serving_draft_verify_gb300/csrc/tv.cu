// dspark_accept_rate_tv: c* = 1 - 1/2 ||softmax(d) - softmax(t)||_1 per row
// (DeepSpec walkthrough, section 3.3, paper eq. 8 / `_compute_accept_rate_3d`),
// computed as sum_v min(p_d(v), p_t(v)).
//
// One HBM pass per row.  A thread-block cluster of kCS CTAs owns one row at a
// time; each CTA bulk-copies its 1/kCS slice of d and t into shared memory
// (double-buffered, so the next row streams in while this one is reduced):
//   A. slice max of d and t;
//   B. e_d = 2^(d log2e - m_d), e_t likewise, kept in registers; slice sums;
//   -- cluster exchange of (m, s) through distributed shared memory --
//   C. sum min(e_d 2^(m_d - L_d), e_t 2^(m_t - L_t)) from registers (no exp);
//   -- cluster exchange of the partial sums; rank 0 writes c*.
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
    static constexpr int kStages = kBF16 ? 2 : 1;
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

// Block-wide reductions over kThreads threads; `red` holds 2 * kWarps floats.
__device__ __forceinline__ float2 block_max2(float2 v, float* red) {
    v.x = warp_max(v.x);
    v.y = warp_max(v.y);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) { red[w] = v.x; red[kWarps + w] = v.y; }
    __syncthreads();
    float a = -INFINITY, b = -INFINITY;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) { a = fmaxf(a, red[i]); b = fmaxf(b, red[kWarps + i]); }
    return make_float2(a, b);
}
__device__ __forceinline__ float2 block_sum2(float2 v, float* red) {
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) { red[w] = v.x; red[kWarps + w] = v.y; }
    __syncthreads();
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) { a += red[i]; b += red[kWarps + i]; }
    return make_float2(a, b);
}

struct Slot {
    float md, sd, mt, st;   // slice max (log2 units) and sum of 2^(y - m)
    float p;                // slice partial of sum min(p_d, p_t)
    float pad[3];
};

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
tv_kernel(const uint8_t* __restrict__ d, const uint8_t* __restrict__ t, float* __restrict__ c_star,
          int64_t rows, int V, int slice, StatusBlock* status) {
    using Tr = TVTraits<kBF16>;
    constexpr int EPG = Tr::kEPG, ESZ = Tr::kESZ, STAGES = Tr::kStages, GMAX = Tr::kGMax;
    extern __shared__ __align__(128) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const uint32_t rank = cluster.block_rank();
    const int64_t cid = blockIdx.x / kCS;
    const int64_t ncl = gridDim.x / kCS;
    const int lo = static_cast<int>(rank) * slice;
    const int len = max(0, min(V, lo + slice) - lo);
    const uint32_t bytes = static_cast<uint32_t>(len) * ESZ;
    const int ngroups = len / EPG;
    const size_t stage_bytes = static_cast<size_t>(slice) * ESZ;

    uint8_t* buf = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * 2 * stage_bytes);
    float* red = reinterpret_cast<float*>(bars + STAGES);
    Slot* slot = reinterpret_cast<Slot*>(red + 2 * kWarps);

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

        // A: slice maxima
        float2 m = make_float2(-INFINITY, -INFINITY);
        if (!failed) {
            for (int g = tid; g < ngroups; g += kThreads) {
                float a[EPG], b[EPG];
                unpack<kBF16>(dg[g], a);
                unpack<kBF16>(tg[g], b);
#pragma unroll
                for (int e = 0; e < EPG; ++e) { m.x = fmaxf(m.x, a[e]); m.y = fmaxf(m.y, b[e]); }
            }
        }
        m = block_max2(m, red);
        // y = x log2e is rounded before the max is subtracted: rounding is monotone,
        // so max(y) is exactly md2 and y - md2 <= 0 even for |x| near the float range
        // a slice with no finite logit keeps reference 0 so that its terms are 2^-inf = 0
        const float md2 = (m.x > -INFINITY) ? __fmul_rn(m.x, kLog2e) : 0.f;
        const float mt2 = (m.y > -INFINITY) ? __fmul_rn(m.y, kLog2e) : 0.f;

        // B: exponentials in registers, slice sums
        float ed[GMAX * EPG], et[GMAX * EPG];
        float2 sum = make_float2(0.f, 0.f);
#pragma unroll
        for (int gi = 0; gi < GMAX; ++gi) {
            const int g = tid + gi * kThreads;
            if (!failed && g < ngroups) {
                float a[EPG], b[EPG];
                unpack<kBF16>(dg[g], a);
                unpack<kBF16>(tg[g], b);
#pragma unroll
                for (int e = 0; e < EPG; ++e) {
                    ed[gi * EPG + e] = exp2f(__fmul_rn(a[e], kLog2e) - md2);
                    et[gi * EPG + e] = exp2f(__fmul_rn(b[e], kLog2e) - mt2);
                    sum.x += ed[gi * EPG + e];
                    sum.y += et[gi * EPG + e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPG; ++e) { ed[gi * EPG + e] = 0.f; et[gi * EPG + e] = 0.f; }
            }
        }
        sum = block_sum2(sum, red);   // ends with every thread past its smem reads of this stage

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
        if (tid == 0) { slot->md = md2; slot->sd = sum.x; slot->mt = mt2; slot->st = sum.y; }
        cluster.sync();

        // every warp combines the kCS slots itself: lane r reads CTA r's slot
        const int lane = tid & 31;
        float rmd = -INFINITY, rsd = 0.f, rmt = -INFINITY, rst = 0.f;
        if (lane < kCS) {
            const Slot* rs = cluster.map_shared_rank(slot, lane);
            rsd = rs->sd; rst = rs->st;
            rmd = rsd > 0.f ? rs->md : -INFINITY;          // empty slices do not set the reference
            rmt = rst > 0.f ? rs->mt : -INFINITY;
        }
        const float Md = warp_max(rmd), Mt = warp_max(rmt);
        const float Sd = warp_sum(rsd > 0.f ? rsd * exp2f(rmd - Md) : 0.f);
        const float St = warp_sum(rst > 0.f ? rst * exp2f(rmt - Mt) : 0.f);
        const float Ld2 = Md + log2f(Sd), Lt2 = Mt + log2f(St);
        const float alpha = (sum.x > 0.f) ? exp2f(md2 - Ld2) : 0.f;
        const float beta = (sum.y > 0.f) ? exp2f(mt2 - Lt2) : 0.f;

        // C: sum of min(p_d, p_t) over this slice, from registers
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < GMAX * EPG; ++i) p += fminf(ed[i] * alpha, et[i] * beta);
        p = block_sum2(make_float2(p, 0.f), red).x;
        if (tid == 0) slot->p = p;
        cluster.sync();
        if (rank == 0 && tid < 32) {
            const float pr = (tid < kCS) ? cluster.map_shared_rank(slot, tid)->p : 0.f;
            const float c = warp_sum(pr);
            if (tid == 0 && !failed) c_star[row] = c;
        }
    }
    // no CTA leaves while a peer may still read its shared memory
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
    return static_cast<size_t>(Tr::kStages) * 2 * slice * Tr::kESZ + Tr::kStages * 8 +
           2 * kWarps * sizeof(float) + sizeof(Slot) + 128;
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_status(workspace, s) != DSPARK_OK) return DSPARK_ERR_CUDA;
    StatusBlock* st = static_cast<StatusBlock*>(workspace);
    return dt == DSPARK_BF16 ? launch_tv<true>(rows, V, d, t, c_star, st, s)
                             : launch_tv<false>(rows, V, d, t, c_star, st, s);
}
