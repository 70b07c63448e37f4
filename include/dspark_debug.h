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

/* Measurement hook: while enabled, dspark_draft_block records a pair of CUDA
 * events (created by the library on the current device at the first enable)
 * around every launch of its vocabulary-wide pass: the one cooperative
 * tensor-core launch that covers all gamma positions, or, on the per-position
 * path, each position's phase kernel.  dspark_debug_phase_times() waits for
 * the last recorded event and writes the duration in ms of each such launch
 * of the most recent dspark_draft_block call into ms[0..n-1]; it returns the
 * number of launches recorded (1 for the cooperative launch, gamma on the
 * per-position path, 0 if timing is off).  Not thread-safe; meant for
 * benchmarks, one device at a time. */
dspark_status_t dspark_debug_enable_phase_timing(int enable);
int dspark_debug_phase_times(float* ms, int n);

/* Test hook: while enabled, the tensor-core draft path launches one engine
 * kernel and one winner kernel per position instead of the single
 * cooperative launch (the path it takes anyway when its grid cannot be
 * co-resident).  Results are identical either way.  Process-wide flag. */
dspark_status_t dspark_debug_force_phase_launches(int enable);

/* Test hook: which path dspark_draft_block takes for bf16 weights with the
 * Markov head (r % 64 == 0, r <= 256).  mode 0 (default): by batch size -- the
 * small-batch GEMV path (W2 streamed once per position for all requests,
 * warp-level MMAs) for B <= 8, where it measured faster, and the tcgen05
 * engine above; 1: always the tcgen05 engine; 2: the GEMV path wherever it
 * applies (B <= 16), the calls it cannot take returning
 * DSPARK_ERR_UNSUPPORTED.  Both paths draw the same tokens from the same
 * Philox words; their logits differ only in the summation order of the
 * rank-r product.  Process-wide flag; DSPARK_ERR_INVALID_ARGUMENT for other
 * modes. */
dspark_status_t dspark_debug_set_draft_path(int mode);

/* Test hook for the bounded waits: one thread waits at the grid barrier kept
 * in a draft workspace (dspark_draft_block_workspace_size(1, 1, 1, 8) bytes,
 * 256-byte aligned) for an arrival that never comes, giving up after
 * limit_ns nanoseconds (1 .. 100 ms) with DSPARK_ERR_TIMEOUT in the
 * workspace's status block -- the same wait routine and status path the
 * cooperative draft and verify launches use.  The device context stays
 * usable.  Asynchronous on `stream`. */
dspark_status_t dspark_debug_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                          dspark_stream_t stream);

/* Test hook for the sampler's noise: E[i] = -ln u_i for u_i = ((words[i] >> 9)
 * + 1/2) 2^-23, computed on the GPU by the same routine the draws use (the
 * Gumbel variate of the draw is -ln E).  words [n] uint32, E [n] float32,
 * device pointers; n >= 0.  Asynchronous on `stream`. */
dspark_status_t dspark_debug_exp_draws(const uint32_t* words, float* E, int64_t n, dspark_stream_t stream);

/* Test hook for the per-row Philox4x32-10 of the draws: out[4 i + j] = word j
 * of Philox(key (seed_lo, seed_hi); counter (q0 + i, k, b, stream)) for
 * i < n, computed on the GPU by the routine the draws use.  out [4 n] uint32
 * device pointer; n >= 0.  Asynchronous on `stream`. */
dspark_status_t dspark_debug_philox_rows(uint64_t seed, uint32_t k, uint32_t b, uint32_t stream, uint32_t q0,
                                         int64_t n, uint32_t* out, dspark_stream_t stream_);

/* Measurement hook: the bytes of host inputs the library has copied to the
 * device with a copy-engine transfer so far in this process (dspark_draft_block
 * stages U and h in pinned host memory that way, outside stream capture);
 * inputs the kernels read over the host link are not counted. */
uint64_t dspark_debug_staged_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_DEBUG_H */
