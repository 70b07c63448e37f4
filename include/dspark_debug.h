/*
 * dspark_debug.h -- test hooks of libdspark.so.  Not part of the draft /
 * schedule / verify path; they expose one internal stage so that tests can
 * check it on its own.
 */
#ifndef DSPARK_DEBUG_H
#define DSPARK_DEBUG_H

#include "dspark.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The draft logits of one position through the tensor-core path (the same
 * kernel, tiles and accumulation as dspark_draft_block's bf16 path):
 *   z[b][v] = U_k[b][v] + sum_j W2[v][j] * W1[prev[b]][j]
 * (DeepSpec walkthrough section 3.2, VanillaMarkovHead, eq. 5).
 *   U_k [B][V], W1 [V][r], W2 [V][r] bf16 (r % 64 == 0, r <= 256, V % 8 == 0);
 *   prev [B] int32 in [0, V); z [B][V] float32 out.
 * workspace: dspark_draft_block_workspace_size(B, 1, V, r) bytes.
 * Returns DSPARK_ERR_UNSUPPORTED if r is not a tensor-core rank. */
dspark_status_t dspark_debug_draft_logits(int B, int V, int r, const void* U_k, const void* W1,
                                          const void* W2, const int32_t* prev, float* z,
                                          void* workspace, size_t workspace_bytes,
                                          dspark_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_DEBUG_H */
