// C-ABI helpers that belong to no single operation: status strings, the
// device status read-back, and the test hooks of the sampler's noise.
#include "common.cuh"
#include "host_common.h"
#include "../../include/dspark_debug.h"

namespace dspark {
namespace {
__global__ void debug_exp_draws(const uint32_t* __restrict__ w, float* __restrict__ E, int64_t n) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        E[i] = exp_draw(w[i]);
}
__global__ void debug_philox_rows(uint64_t seed, uint32_t k, uint32_t b, uint32_t stream, uint32_t q0, int64_t n,
                                  uint32_t* __restrict__ out) {
    const PhiloxRow pr = philox_row_setup(seed, k, b, stream);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const U4 r = philox_row(pr, q0 + static_cast<uint32_t>(i));
        out[4 * i] = r.x;
        out[4 * i + 1] = r.y;
        out[4 * i + 2] = r.z;
        out[4 * i + 3] = r.w;
    }
}
}  // namespace
}  // namespace dspark

extern "C" dspark_status_t dspark_debug_exp_draws(const uint32_t* words, float* E, int64_t n,
                                                  dspark_stream_t stream) {
    if (n < 0 || (n > 0 && (words == nullptr || E == nullptr))) return DSPARK_ERR_INVALID_ARGUMENT;
    dspark::clear_stale_error();
    if (n == 0) return DSPARK_OK;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    dspark::debug_exp_draws<<<static_cast<int>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(words, E, n);
    return dspark::launch_status();
}

extern "C" dspark_status_t dspark_debug_philox_rows(uint64_t seed, uint32_t k, uint32_t b, uint32_t stream,
                                                    uint32_t q0, int64_t n, uint32_t* out, dspark_stream_t stream_) {
    if (n < 0 || (n > 0 && out == nullptr)) return DSPARK_ERR_INVALID_ARGUMENT;
    dspark::clear_stale_error();
    if (n == 0) return DSPARK_OK;
    const int64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    dspark::debug_philox_rows<<<static_cast<int>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream_)>>>(
        seed, k, b, stream, q0, n, out);
    return dspark::launch_status();
}

extern "C" const char* dspark_status_string(dspark_status_t s) {
    switch (s) {
        case DSPARK_OK: return "DSPARK_OK";
        case DSPARK_ERR_INVALID_ARGUMENT: return "DSPARK_ERR_INVALID_ARGUMENT";
        case DSPARK_ERR_UNSUPPORTED: return "DSPARK_ERR_UNSUPPORTED";
        case DSPARK_ERR_WORKSPACE_TOO_SMALL: return "DSPARK_ERR_WORKSPACE_TOO_SMALL";
        case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
        case DSPARK_ERR_TIMEOUT: return "DSPARK_ERR_TIMEOUT";
        case DSPARK_ERR_DEVICE_CHECK: return "DSPARK_ERR_DEVICE_CHECK";
    }
    return "DSPARK_ERR_UNKNOWN";
}

extern "C" dspark_status_t dspark_workspace_status(const void* workspace, dspark_stream_t stream) {
    if (workspace == nullptr) return DSPARK_ERR_INVALID_ARGUMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t code = 0;
    if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
    return static_cast<dspark_status_t>(code);
}

namespace dspark {
namespace {
std::mutex g_stage_mu;
cudaMemPool_t g_stage_pool[64] = {};

// The library's own pool on device `dev` (created on first use), which keeps its
// memory between calls rather than returning it at every synchronisation.
cudaMemPool_t stage_pool(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_stage_mu);
    if (g_stage_pool[dev] != nullptr) return g_stage_pool[dev];
    cudaMemPoolProps pp{};
    pp.allocType = cudaMemAllocationTypePinned;
    pp.location.type = cudaMemLocationTypeDevice;
    pp.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &pp) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    uint64_t keep = ~static_cast<uint64_t>(0);
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
        cudaGetLastError();
        cudaMemPoolDestroy(pool);
        return nullptr;
    }
    g_stage_pool[dev] = pool;
    return pool;
}
}  // namespace

std::atomic<uint64_t> g_staged_bytes{0};

void* stage_to_device(const void* host, size_t bytes, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone || bytes == 0) return nullptr;
    cudaMemPool_t pool = stage_pool(current_device());
    if (pool == nullptr) return nullptr;
    void* d = nullptr;
    if (cudaMallocFromPoolAsync(&d, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cudaMemcpyAsync(d, host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        cudaFreeAsync(d, s);
        return nullptr;
    }
    g_staged_bytes.fetch_add(bytes);
    return d;
}

void stage_release(void* p, cudaStream_t s) {
    if (p != nullptr) cudaFreeAsync(p, s);
}

std::atomic<size_t> g_l2_resident_bytes{0};
std::atomic<size_t> g_l2_window_max{0};
namespace {
std::mutex g_l2_mu;
bool g_l2_saved = false;
size_t g_l2_prev_limit = 0;
}  // namespace
}  // namespace dspark

extern "C" dspark_status_t dspark_set_l2_residency(size_t bytes) {
    using namespace dspark;
    std::lock_guard<std::mutex> lock(g_l2_mu);
    clear_stale_error();
    if (bytes == 0) {
        g_l2_resident_bytes.store(0);
        if (g_l2_saved) {
            // W2's lines back to normal, then the set-aside back to what it was
            if (cudaCtxResetPersistingL2Cache() != cudaSuccess) {
                cudaGetLastError();
                return DSPARK_ERR_CUDA;
            }
            if (cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, g_l2_prev_limit) != cudaSuccess) {
                cudaGetLastError();
                return DSPARK_ERR_CUDA;
            }
            g_l2_saved = false;
        }
        return DSPARK_OK;
    }
    const int dev = current_device();
    int maxp = 0, maxw = 0;
    if (cudaDeviceGetAttribute(&maxp, cudaDevAttrMaxPersistingL2CacheSize, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&maxw, cudaDevAttrMaxAccessPolicyWindowSize, dev) != cudaSuccess || maxp <= 0 ||
        maxw <= 0) {
        cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    if (!g_l2_saved) {
        if (cudaDeviceGetLimit(&g_l2_prev_limit, cudaLimitPersistingL2CacheSize) != cudaSuccess) {
            cudaGetLastError();
            return DSPARK_ERR_CUDA;
        }
        g_l2_saved = true;
    }
    const size_t keep = bytes < static_cast<size_t>(maxp) ? bytes : static_cast<size_t>(maxp);
    if (cudaDeviceSetLimit(cudaLimitPersistingL2CacheSize, keep) != cudaSuccess) {
        cudaGetLastError();
        return DSPARK_ERR_CUDA;
    }
    g_l2_window_max.store(static_cast<size_t>(maxw));
    g_l2_resident_bytes.store(keep);
    return DSPARK_OK;
}

extern "C" uint64_t dspark_debug_staged_bytes(void) { return dspark::g_staged_bytes.load(); }
