// dspark_draft_block_noalloc: dspark_draft_block for callers that cannot
// allocate device memory.  Some hosts of this library own every byte of GPU
// memory through their own pool or arena and forbid cudaMalloc (and allocating
// library calls) from plug-in code: an inference server that pre-reserves its
// memory at start-up, or a runtime that must not allocate inside a step.  They
// can pass inputs and outputs, but not the scratch workspace that
// dspark_draft_block wants.  This entry point uses a fixed scratch array that
// lives in the library's own device image instead.
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace {

// Scratch for one draft block call: status block, per-position winner words,
// per-chunk (max, sum) partials and the y of each chunk's best token.  Every GPU
// that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
static __device__ __align__(256) unsigned char g_draft_scratch[kNoAllocScratchBytes];

// Device address of g_draft_scratch, looked up once per device with that
// device current.  The host-side name g_draft_scratch is only a stand-in; a
// kernel must be given the address returned by cudaGetSymbolAddress.
constexpr int kMaxDevices = 64;   // device ordinals 0 .. 63 (more than any one node has)
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

void* scratch_address(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_draft_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" dspark_status_t dspark_draft_block_noalloc(int B, int gamma, int V, int H, int r, dspark_dtype_t dt,
                                                      const void* U, const void* h, const void* W1, const void* W2,
                                                      const void* w, float bias, const int32_t* x0,
                                                      float temperature, uint64_t seed, int32_t* x, float* lse_d,
                                                      float* logp_d, float* c, float* a, dspark_stream_t stream) {
    // the size checks of dspark_draft_block first, so that a malformed call is an
    // argument error whatever its size
    if (B <= 0 || B > 65535 || gamma <= 0 || gamma > DSPARK_MAX_GAMMA || V <= 0 || H < 0 || r <= 0 || r > 256)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (dspark_draft_block_workspace_size(B, gamma, V, r) > kNoAllocScratchBytes) return DSPARK_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (dev >= kMaxDevices) return DSPARK_ERR_UNSUPPORTED;
    void* scratch = scratch_address(dev);
    if (scratch == nullptr) return DSPARK_ERR_CUDA;
    // dspark_draft_block's path clears the status block and the per-position words
    // itself; inputs in host memory are read over the link (no staging copy, which
    // would allocate)
    return dspark::draft_block_entry(B, gamma, V, H, r, dt, U, h, W1, W2, w, bias, x0, temperature, seed, x, lse_d,
                                     logp_d, c, a, scratch, kNoAllocScratchBytes, stream, /*stage=*/false);
}
