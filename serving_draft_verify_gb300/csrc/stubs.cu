// Entry points not yet implemented: they return DSPARK_ERR_UNSUPPORTED.
#include "common.cuh"
#include "host_common.h"

extern "C" size_t dspark_verify_workspace_size(int, int, int, int) { return dspark::kStatusBytes; }
extern "C" dspark_status_t dspark_verify(int, int, int, int, dspark_dtype_t, const void*, const void*, const void*,
                                         const void*, const int32_t*, const int32_t*, const float*, const float*,
                                         const int32_t*, float, uint64_t, int32_t*, int32_t*, void*, size_t,
                                         dspark_stream_t) {
    return DSPARK_ERR_UNSUPPORTED;
}
