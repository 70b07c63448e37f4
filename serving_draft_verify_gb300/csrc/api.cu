// C-ABI helpers that belong to no single operation: status strings and the
// device status read-back.
#include "common.cuh"
#include "host_common.h"

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
