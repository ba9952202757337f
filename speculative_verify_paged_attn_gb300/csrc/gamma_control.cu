// gamma_control.cu -- acceptance telemetry and the adaptive draft length.
//
// "Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM Serving"
// (dynamic lookahead from a moving-average acceptance rate: above 0.85 -> 5
// drafts, above 0.70 -> 4, above 0.50 -> 3, otherwise 2); "The Sub-Millisecond
// Speculative Decoding Meltdown", production failure scenarios (below 0.25 the
// engine falls back to one token); "LOW-LATENCY INFERENCE: SPECULATIVE
// DECODING & PAGING", acceptance math (E[K] = sum_{i<=gamma} alpha^i, speed-up
// (E[K] + 1) / (gamma r + 1)).
//
// A sequence that accepted k of g drafts ran k + (k < g) acceptance tests, so
// accepted / tests estimates the per-token rate.  Moving averages in fp32,
// every product and sum rounded on its own: A = d*A + k, N = d*N + tests,
// alpha = A / N.  The batch keeps its own (A, N) over the step's integer totals,
// so its draft length does not depend on a summation order.
//
// One CTA: each thread updates sequences, integer totals are reduced in shared
// memory, thread 0 updates the batch state and writes the telemetry.  The call
// reads the step's accepted lengths where they already are (device memory), so
// the next step's draft length is decided without a host round trip.
#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kGammaThreads = 256;

__device__ __forceinline__ int gamma_from_alpha(float alpha) {
    if (alpha > 0.85f) return 5;
    if (alpha > 0.70f) return 4;
    if (alpha > 0.50f) return 3;
    if (alpha >= 0.25f) return 2;
    return 1;
}

__global__ void __launch_bounds__(kGammaThreads) gamma_update_kernel(const __grid_constant__ GammaArgs a) {
    __shared__ unsigned long long s_k, s_t;
    __shared__ int s_bad;
    if (threadIdx.x == 0) {
        s_k = 0ull;
        s_t = 0ull;
        s_bad = 0;
    }
    __syncthreads();
    unsigned long long my_k = 0ull, my_t = 0ull;
    for (int b = threadIdx.x; b < a.B; b += kGammaThreads) {
        const int k = a.accepted_len[b];
        if (k < 0 || k > a.gamma) {
            s_bad = 1;
            continue;
        }
        const int tests = k + (k < a.gamma ? 1 : 0);
        my_k += (unsigned long long)k;
        my_t += (unsigned long long)tests;
        if (a.seq_state) {
            const float A = __fadd_rn(__fmul_rn(a.decay, a.seq_state[2 * b]), (float)k);
            const float N = __fadd_rn(__fmul_rn(a.decay, a.seq_state[2 * b + 1]), (float)tests);
            a.seq_state[2 * b] = A;
            a.seq_state[2 * b + 1] = N;
            if (a.seq_gamma_next) a.seq_gamma_next[b] = gamma_from_alpha(__fdiv_rn(A, N));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        my_k += __shfl_xor_sync(0xffffffffu, my_k, o);
        my_t += __shfl_xor_sync(0xffffffffu, my_t, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&s_k, my_k);
        atomicAdd(&s_t, my_t);
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    if (s_bad) {
        raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        return;
    }
    const float A = __fadd_rn(__fmul_rn(a.decay, a.batch_state[0]), (float)s_k);
    const float N = __fadd_rn(__fmul_rn(a.decay, a.batch_state[1]), (float)s_t);
    a.batch_state[0] = A;
    a.batch_state[1] = N;
    const float alpha = __fdiv_rn(A, N);
    const int g = gamma_from_alpha(alpha);
    *a.batch_gamma_next = g;
    float ek = 0.f, prod = 1.f;
    for (int i = 0; i < g; ++i) {
        prod = __fmul_rn(prod, alpha);
        ek = __fadd_rn(ek, prod);
    }
    const float eta = __fdiv_rn(__fadd_rn(ek, 1.f), __fadd_rn(__fmul_rn((float)g, a.r), 1.f));
    a.telemetry[0] = alpha;
    a.telemetry[1] = __fdiv_rn((float)s_k, (float)a.B);
    a.telemetry[2] = ek;
    a.telemetry[3] = eta;
}

}  // namespace

cudaError_t launch_gamma_update(const GammaArgs &a, cudaStream_t stream) {
    gamma_update_kernel<<<1, kGammaThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace svpa
