// dspark_decode_rounds: several speculative-decoding rounds in a row on one
// stream (DeepSpec walkthrough sections 8.1 / 8.3, `generate_decoding_sample`:
// propose a draft block, verify it, emit the accepted tokens and the verifier's
// token, continue from the new context).  Each round is the draft block, the
// prefix scheduler (Algorithm 1, section 3.3) and verification (section 8.2),
// followed by round_update, which records what the round emitted and carries
// the anchor: the next round's x_0 is the last token emitted.  Nothing here
// synchronises with the host, so a caller can capture all rounds in one CUDA
// graph.
#include "common.cuh"
#include "host_common.h"

namespace dspark {
namespace {

constexpr int kUpdThreads = 1024;

struct TraceArgs {
    int32_t* x;
    float* lse_d;
    float* logp_d;
    float* c;
    float* a;
    int32_t* ell;
    int32_t* n_accept;
    int32_t* next_token;
};

// Round i's bookkeeping, one CTA: the emitted tokens (accepted draft tokens, the
// verifier's token, then -1), their count, the next anchor, E[tau] and the
// realised tokens per request, the sub-calls' device status, and the optional
// per-round trace of the draft / schedule / verify outputs.
__global__ void __launch_bounds__(kUpdThreads)
round_update(int round, int B, int gamma, const int32_t* __restrict__ x, const float* __restrict__ lse_d,
             const float* __restrict__ logp_d, const float* __restrict__ c, const float* __restrict__ a,
             const int32_t* __restrict__ ell, const int32_t* __restrict__ n_accept,
             const int32_t* __restrict__ next_token, int32_t* anchor, int32_t* tokens, int32_t* n_emitted,
             double* stats, TraceArgs tr, StatusBlock* status, const StatusBlock* st_draft,
             const StatusBlock* st_sched, const StatusBlock* st_verify) {
    __shared__ double e_part[kUpdThreads / 32];
    __shared__ long long n_part[kUpdThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bg = static_cast<size_t>(B) * gamma;
    double e_sum = 0.0;
    long long n_sum = 0;
    for (int b = tid; b < B; b += kUpdThreads) {
        int n = n_accept[b];
        int l = ell[b];
        if (n < 0 || n > gamma) {                    // cannot come from dspark_verify; guarded anyway
            set_status(status, DSPARK_ERR_DEVICE_CHECK, 40);
            n = n < 0 ? 0 : gamma;
        }
        if (l < 0 || l > gamma) {
            set_status(status, DSPARK_ERR_DEVICE_CHECK, 41);
            l = l < 0 ? 0 : gamma;
        }
        const int y = next_token[b];
        int32_t* out = tokens + (static_cast<size_t>(round) * B + b) * (gamma + 1);
        for (int k = 0; k <= gamma; ++k) out[k] = k < n ? x[static_cast<size_t>(b) * gamma + k] : (k == n ? y : -1);
        n_emitted[static_cast<size_t>(round) * B + b] = n + 1;
        anchor[b] = y;
        double e = 1.0;
        for (int j = 0; j < l; ++j) e += static_cast<double>(a[static_cast<size_t>(b) * gamma + j]);
        e_sum += e;
        n_sum += n + 1;
    }
    // block sums in a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        e_sum += __shfl_xor_sync(0xffffffffu, e_sum, o);
        n_sum += __shfl_xor_sync(0xffffffffu, n_sum, o);
    }
    if (lane == 0) {
        e_part[warp] = e_sum;
        n_part[warp] = n_sum;
    }
    if (tr.x || tr.lse_d || tr.logp_d || tr.c || tr.a) {
        const size_t o = static_cast<size_t>(round) * bg;
        for (size_t i = tid; i < bg; i += kUpdThreads) {
            if (tr.x) tr.x[o + i] = x[i];
            if (tr.lse_d) tr.lse_d[o + i] = lse_d[i];
            if (tr.logp_d) tr.logp_d[o + i] = logp_d[i];
            if (tr.c) tr.c[o + i] = c[i];
            if (tr.a) tr.a[o + i] = a[i];
        }
    }
    if (tr.ell || tr.n_accept || tr.next_token) {
        const size_t o = static_cast<size_t>(round) * B;
        for (int b = tid; b < B; b += kUpdThreads) {
            if (tr.ell) tr.ell[o + b] = ell[b];
            if (tr.n_accept) tr.n_accept[o + b] = n_accept[b];
            if (tr.next_token) tr.next_token[o + b] = next_token[b];
        }
    }
    __syncthreads();
    if (tid == 0) {
        double E = 0.0;
        long long N = 0;
        for (int w = 0; w < kUpdThreads / 32; ++w) {
            E += e_part[w];
            N += n_part[w];
        }
        stats[2 * round] = E / B;
        stats[2 * round + 1] = static_cast<double>(N) / B;
        // the first error of a sub-call, tagged with its stage (1 draft, 2 schedule, 3 verify)
        const StatusBlock* subs[3] = {st_draft, st_sched, st_verify};
        for (int s = 0; s < 3; ++s) {
            const uint32_t code = subs[s]->code;
            if (code != 0u) set_status(status, code, 1000u * (s + 1) + subs[s]->detail);
        }
    }
}

struct RoundsLayout {
    size_t draft, sched, verify;                          // sub-workspaces (each 256-byte aligned)
    size_t draft_bytes, sched_bytes, verify_bytes;
    size_t x, lse_d, logp_d, c, a, ell, n_sched, theta, n_accept, next_token;
    size_t total;
};

RoundsLayout rounds_layout(int B, int gamma, int V, int r) {
    RoundsLayout L{};
    const size_t bg = static_cast<size_t>(B) * gamma;
    size_t o = kStatusBytes;
    auto take = [&o](size_t bytes) {
        const size_t at = o;
        o = round_up(o + bytes, 256);
        return at;
    };
    L.draft_bytes = dspark_draft_block_workspace_size(B, gamma, V, r);
    L.sched_bytes = dspark_schedule_prefix_workspace_size(B, gamma);
    L.verify_bytes = dspark_verify_workspace_size(B, gamma, V, r);
    L.draft = take(L.draft_bytes);
    L.sched = take(L.sched_bytes);
    L.verify = take(L.verify_bytes);
    L.x = take(bg * 4);
    L.lse_d = take(bg * 4);
    L.logp_d = take(bg * 4);
    L.c = take(bg * 4);
    L.a = take(bg * 4);
    L.ell = take(static_cast<size_t>(B) * 4);
    L.n_sched = take(4);
    L.theta = take(8);
    L.n_accept = take(static_cast<size_t>(B) * 4);
    L.next_token = take(static_cast<size_t>(B) * 4);
    L.total = o;
    return L;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_decode_rounds_workspace_size(int B, int gamma, int V, int r) {
    if (B <= 0 || gamma <= 0 || V <= 0 || r <= 0) return kStatusBytes;
    return rounds_layout(B, gamma, V, r).total;
}

extern "C" dspark_status_t dspark_decode_rounds(int rounds, int pool, int B, int gamma, int V, int H, int r,
                                                dspark_dtype_t dt, const void* U, const void* h,
                                                const void* t_logits, const void* W1, const void* W2,
                                                const void* w, float bias, const double* sps, int32_t* anchor,
                                                float temperature, uint64_t seed, int32_t* tokens,
                                                int32_t* n_emitted, double* stats, const dspark_round_trace_t* trace,
                                                void* workspace, size_t workspace_bytes, dspark_stream_t stream) {
    if (rounds < 0 || pool < 1 || B <= 0 || gamma <= 0 || V <= 0 || H <= 0 || r <= 0)
        return DSPARK_ERR_INVALID_ARGUMENT;
    if (dt != DSPARK_F32 && dt != DSPARK_BF16) return DSPARK_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || !aligned256(workspace)) return DSPARK_ERR_INVALID_ARGUMENT;
    const RoundsLayout L = rounds_layout(B, gamma, V, r);
    if (workspace_bytes < L.total) return DSPARK_ERR_WORKSPACE_TOO_SMALL;
    clear_stale_error();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (clear_status(workspace, s) != DSPARK_OK) return DSPARK_ERR_CUDA;
    if (rounds == 0) return DSPARK_OK;
    if (U == nullptr || h == nullptr || t_logits == nullptr || W1 == nullptr || W2 == nullptr || w == nullptr ||
        sps == nullptr || anchor == nullptr || tokens == nullptr || n_emitted == nullptr || stats == nullptr)
        return DSPARK_ERR_INVALID_ARGUMENT;

    uint8_t* base = static_cast<uint8_t*>(workspace);
    auto at = [base](size_t off) { return static_cast<void*>(base + off); };
    int32_t* x = static_cast<int32_t*>(at(L.x));
    float* lse_d = static_cast<float*>(at(L.lse_d));
    float* logp_d = static_cast<float*>(at(L.logp_d));
    float* c = static_cast<float*>(at(L.c));
    float* a = static_cast<float*>(at(L.a));
    int32_t* ell = static_cast<int32_t*>(at(L.ell));
    int32_t* n_sched = static_cast<int32_t*>(at(L.n_sched));
    double* theta = static_cast<double*>(at(L.theta));
    int32_t* n_accept = static_cast<int32_t*>(at(L.n_accept));
    int32_t* next_token = static_cast<int32_t*>(at(L.next_token));
    TraceArgs tr{};
    if (trace != nullptr) {
        tr.x = trace->x;
        tr.lse_d = trace->lse_d;
        tr.logp_d = trace->logp_d;
        tr.c = trace->c;
        tr.a = trace->a;
        tr.ell = trace->ell;
        tr.n_accept = trace->n_accept;
        tr.next_token = trace->next_token;
    }

    const size_t esz = dt == DSPARK_BF16 ? 2 : 4;
    const size_t u_slot = static_cast<size_t>(B) * gamma * V * esz;
    const size_t h_slot = static_cast<size_t>(B) * gamma * H * esz;
    const size_t t_slot = static_cast<size_t>(B) * (gamma + 1) * V * esz;
    for (int i = 0; i < rounds; ++i) {
        const size_t p = static_cast<size_t>(i % pool);
        const void* Ui = static_cast<const uint8_t*>(U) + p * u_slot;
        const void* hi = static_cast<const uint8_t*>(h) + p * h_slot;
        const void* ti = static_cast<const uint8_t*>(t_logits) + p * t_slot;
        const uint64_t si = seed + static_cast<uint64_t>(i);   // each round its own Philox key
        dspark_status_t st = dspark_draft_block(B, gamma, V, H, r, dt, Ui, hi, W1, W2, w, bias, anchor, temperature,
                                                si, x, lse_d, logp_d, c, a, at(L.draft), L.draft_bytes, stream);
        if (st != DSPARK_OK) return st;
        st = dspark_schedule_prefix(B, gamma, a, sps, ell, n_sched, theta, at(L.sched), L.sched_bytes, stream);
        if (st != DSPARK_OK) return st;
        st = dspark_verify(B, gamma, V, r, dt, ti, Ui, W1, W2, anchor, x, lse_d, logp_d, ell, temperature, si,
                           n_accept, next_token, at(L.verify), L.verify_bytes, stream);
        if (st != DSPARK_OK) return st;
        round_update<<<1, kUpdThreads, 0, s>>>(i, B, gamma, x, lse_d, logp_d, c, a, ell, n_accept, next_token, anchor,
                                               tokens, n_emitted, stats, tr, static_cast<StatusBlock*>(workspace),
                                               static_cast<const StatusBlock*>(at(L.draft)),
                                               static_cast<const StatusBlock*>(at(L.sched)),
                                               static_cast<const StatusBlock*>(at(L.verify)));
        if (launch_status() != DSPARK_OK) return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}
