// Host-side helpers shared by the C-ABI entry points: argument checks,
// per-device caches, launch error mapping.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/dspark.h"

namespace dspark {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// W2's L2 residency (dspark_set_l2_residency): the bytes of persisting L2 the
// context now sets aside (0: off) and the largest access-policy window.
extern std::atomic<size_t> g_l2_resident_bytes;
extern std::atomic<size_t> g_l2_window_max;

// Adds to `attr` an access-policy window that marks the lines of [base, base +
// bytes) persisting, when residency is on; returns whether it did.  The window
// covers min(bytes, the largest window) and a fraction hitRatio of it is
// persisting, so that what persists fits the set-aside.
inline bool l2_window(cudaLaunchAttribute* attr, const void* base, size_t bytes) {
    const size_t keep = g_l2_resident_bytes.load(), wmax = g_l2_window_max.load();
    if (keep == 0 || wmax == 0 || base == nullptr || bytes == 0) return false;
    const size_t nb = bytes < wmax ? bytes : wmax;
    attr->id = cudaLaunchAttributeAccessPolicyWindow;
    attr->val.accessPolicyWindow.base_ptr = const_cast<void*>(base);
    attr->val.accessPolicyWindow.num_bytes = nb;
    attr->val.accessPolicyWindow.hitRatio = keep >= nb ? 1.f : static_cast<float>(keep) / static_cast<float>(nb);
    attr->val.accessPolicyWindow.hitProp = cudaAccessPropertyPersisting;
    attr->val.accessPolicyWindow.missProp = cudaAccessPropertyStreaming;
    return true;
}

// Current device and its SM count (cached per device; calls from several host
// threads may fill an entry at once, all with the same value).
inline int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}
inline int sm_count(int dev) {
    static std::atomic<int> cache[64];                    // static storage: starts at 0
    if (dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Launch-error check mapped to a status.
// Drops an error left by an earlier, unrelated runtime call (not a sticky one:
// those persist and fail the next launch), so that launch_status() reports
// this library's launches only.  Called at the top of each entry point.
inline void clear_stale_error() { cudaGetLastError(); }

inline dspark_status_t launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// Clears the status block at the head of a workspace (async on `stream`).
inline dspark_status_t clear_status(void* workspace, cudaStream_t stream) {
    return cudaMemsetAsync(workspace, 0, 16, stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// The address kernels use for `p`: p itself for device (or managed) memory, the
// mapping's device address for page-locked host memory registered with CUDA (the
// kernels then read it over the host link, only the bytes they touch), and false
// for ordinary host memory, which a kernel cannot reach.
inline bool device_view(const void* p, const void** out) {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (pa.type == cudaMemoryTypeUnregistered) return false;
    if (pa.type == cudaMemoryTypeHost) {
        if (pa.devicePointer == nullptr || !aligned16(pa.devicePointer)) return false;
        *out = pa.devicePointer;
        return true;
    }
    *out = p;
    return true;
}

// True if p (or the device address of a mapping) lies in page-locked host memory.
inline bool in_host_memory(const void* p) {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return pa.type == cudaMemoryTypeHost;
}

// Device memory holding a copy of `bytes` of page-locked host memory at `host`,
// written by one copy-engine transfer on `s` (the host link's full rate; a
// kernel's own scattered reads of a mapping reach less).  The memory comes,
// stream-ordered, from a pool private to the library that keeps what it has
// allocated between calls, until the process exits.  nullptr where that is not
// possible -- `s` is being captured into a graph, or the allocation fails --
// and the caller's kernels then read the mapping themselves.
void* stage_to_device(const void* host, size_t bytes, cudaStream_t s);
// Returns a stage_to_device buffer to the pool once the work queued on `s` so far
// is done.
void stage_release(void* p, cudaStream_t s);

// dspark_draft_block with `stage` choosing whether U and h in host memory are first
// copied to the device (stage_to_device) or read over the link by the kernels; the
// no-allocation entry point passes false.
dspark_status_t draft_block_entry(int B, int gamma, int V, int H, int r, dspark_dtype_t dt, const void* U,
                                  const void* h, const void* W1, const void* W2, const void* w, float bias,
                                  const int32_t* x0, float temperature, uint64_t seed, int32_t* x, float* lse_d,
                                  float* logp_d, float* c, float* a, void* workspace, size_t workspace_bytes,
                                  dspark_stream_t stream, bool stage);

// Once-per-device flag for one-time kernel attribute setup.
struct OncePerDevice {
    std::mutex mu;
    bool done[64] = {false};
    template <class F>
    cudaError_t run(int dev, F&& f) {
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        if (done[dev]) return cudaSuccess;
        const cudaError_t e = f();
        if (e == cudaSuccess) done[dev] = true;
        return e;
    }
};

}  // namespace dspark
