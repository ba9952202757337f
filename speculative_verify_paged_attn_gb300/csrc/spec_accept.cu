// spec_accept.cu -- draft/target rejection samplers for sm_103a.
//
// Linear sampler ("LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING",
// section "Verification Acceptance Probabilities and Speedup Math":
// alpha_i = min(1, P(x_i)/Q(x_i)); architecture diagram: "Rejection Recovery
// (Resample)"): draft i is accepted iff u_i * Q_i(x_i) <= P_i(x_i) with the
// product rounded once to fp32; the first rejected position k is resampled
// from max(0, P_k - Q_k), or a bonus token is drawn from P_gamma when every
// draft is accepted.  The draw is the first token whose running residual
// mass exceeds u * (total mass).
//
// GB300 layout: one 1024-thread CTA per row.  Warp 0 runs the gamma
// acceptance tests (gathered loads and a warp ballot); then every thread sums
// its contiguous segment of the residual row in fp32 (vector loads, token
// order), a block-wide fp64 exclusive scan gives each segment's offset and
// the total S, and the thread whose segment holds u*S walks it again to
// find the token.  One pass over the row, no inter-CTA protocol.
//
// This file is compiled with -fmad=false; the acceptance product also uses
// __fmul_rn, which is never contracted.
#include <math_constants.h>

#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kRowThreads = 1024;
constexpr double kNearBand = 1e-6;

// Block-wide exclusive scan of one double per thread; returns this thread's
// exclusive prefix and writes the block total to *total.
__device__ double block_exclusive_scan(double v, double *total, double *s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        double w = lane < nw ? s_warp[lane] : 0.0;
        double wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) s_warp[32 + lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == nw - 1) s_warp[64] = wi;
    }
    __syncthreads();
    const double ex = s_warp[32 + warp] + (inc - v);
    *total = s_warp[64];
    __syncthreads();
    return ex;
}

// Residual weight of token t: max(0, P - Q) (fp32), or P when q == nullptr.
__device__ __forceinline__ float weight(const float *p, const float *q, int t) {
    const float pv = __ldg(p + t);
    if (!q) return pv;
    const float d = pv - __ldg(q + t);
    return d > 0.f ? d : 0.f;
}

// fp32 sum of the weights of tokens [s0, s1) in token order; 16-byte vector
// loads when the segment allows them.
__device__ float segment_sum(const float *p, const float *q, int s0, int s1) {
    float acc = 0.f;
    const bool vec = ((s1 - s0) & 3) == 0 && ((reinterpret_cast<uintptr_t>(p + s0) & 15) == 0) &&
                     (!q || (reinterpret_cast<uintptr_t>(q + s0) & 15) == 0);
    if (vec) {
        const float4 *p4 = reinterpret_cast<const float4 *>(p + s0);
        const float4 *q4 = q ? reinterpret_cast<const float4 *>(q + s0) : nullptr;
        const int n4 = (s1 - s0) >> 2;
#pragma unroll 8
        for (int i = 0; i < n4; ++i) {
            float4 w = __ldg(p4 + i);
            if (q4) {
                const float4 v = __ldg(q4 + i);
                w.x = fmaxf(w.x - v.x, 0.f);
                w.y = fmaxf(w.y - v.y, 0.f);
                w.z = fmaxf(w.z - v.z, 0.f);
                w.w = fmaxf(w.w - v.w, 0.f);
            }
            acc += w.x;
            acc += w.y;
            acc += w.z;
            acc += w.w;
        }
        return acc;
    }
    for (int t = s0; t < s1; ++t) acc += weight(p, q, t);
    return acc;
}

__global__ void __launch_bounds__(kRowThreads) spec_accept_kernel(const __grid_constant__ AcceptArgs a) {
    __shared__ double s_warp[72];
    __shared__ double s_c[2];
    __shared__ int s_k, s_tok;
    const int b = blockIdx.x;
    const int gamma = a.gamma, V = a.V;

    // ---- acceptance tests
    if (threadIdx.x < 32) {
        const int i = threadIdx.x;
        bool rejected = false;
        if (i < gamma) {
            int x = a.tokens[(size_t)b * gamma + i];
            if (x < 0 || x >= V) {
                raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                x = 0;
            }
            const float qx = __ldg(a.q + ((size_t)b * gamma + i) * V + x);
            const float px = __ldg(a.p + ((size_t)b * (gamma + 1) + i) * V + x);
            const float u = __ldg(a.u_acc + (size_t)b * gamma + i);
            rejected = !(__fmul_rn(u, qx) <= px);
        }
        const unsigned rej = __ballot_sync(0xffffffffu, rejected);
        if (i == 0) {
            s_k = rej ? __ffs(rej) - 1 : gamma;
            s_tok = -1;
        }
    }
    __syncthreads();
    const int k = s_k;
    const float *prow = a.p + ((size_t)b * (gamma + 1) + k) * V;
    const float *qrow = k < gamma ? a.q + ((size_t)b * gamma + k) * V : nullptr;

    // ---- residual mass of this thread's segment and the row total
    const int per = ((V + blockDim.x - 1) / blockDim.x + 3) & ~3;
    const int s0 = min(V, (int)threadIdx.x * per), s1 = min(V, s0 + per);
    float part = segment_sum(prow, qrow, s0, s1);
    double S;
    double ex = block_exclusive_scan((double)part, &S, s_warp);
    if (!(S > 0.0) && qrow) {
        // empty residual: draw from the target row instead
        qrow = nullptr;
        part = segment_sum(prow, nullptr, s0, s1);
        ex = block_exclusive_scan((double)part, &S, s_warp);
    }
    const float u = __ldg(a.u_s + b);
    const double target = (double)u * S;
    if (S > 0.0 && ex <= target && target < ex + (double)part) {
        float run = 0.f;
        for (int t = s0; t < s1; ++t) {
            const float w = weight(prow, qrow, t);
            const float prev = run;
            run += w;
            if (ex + (double)run > target) {
                s_tok = t;
                s_c[0] = ex + (double)prev;
                s_c[1] = ex + (double)run;
                break;
            }
        }
    }
    __syncthreads();
    int tok = s_tok;
    bool near = false;
    if (tok >= 0) {
        near = fabs(s_c[0] / S - (double)u) < kNearBand || fabs(s_c[1] / S - (double)u) < kNearBand;
    } else {
        // u*S at or past the total (rounding): the last token with mass
        int best = -1;
        for (int t = threadIdx.x; t < V; t += blockDim.x)
            if (weight(prow, qrow, t) > 0.f) best = t;
        if (best >= 0) atomicMax(&s_tok, best);
        __syncthreads();
        tok = s_tok;
        near = true;
        if (tok < 0) {
            if (threadIdx.x == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);  // a row with no mass
            tok = 0;
        }
    }
    if (threadIdx.x <= gamma) {
        const int i = threadIdx.x;
        int v;
        if (i < k) v = a.tokens[(size_t)b * gamma + i];
        else if (i == k) v = tok;
        else v = -1;
        a.out_tokens[(size_t)b * (gamma + 1) + i] = v;
    }
    if (threadIdx.x == 0) {
        a.accepted_len[b] = k;
        if (a.near) a.near[b] = near ? 1 : 0;
    }
}

// ---------------------------------------------------------------- tree
constexpr int kTreeThreads = 1024;

// Block sum (fp64) of fp32 per-thread partials.
__device__ double block_sum(double v, double *s_warp) {
    double tot;
    block_exclusive_scan(v, &tot, s_warp);
    return tot;
}

// Inverse-CDF draw from the residual R held in shared memory (fp32, V
// entries): thread i owns a contiguous segment.
__device__ int smem_draw(const float *R, int V, double u, double *s_warp, int *s_tok, double *s_c,
                         bool *near) {
    const int seg = (V + blockDim.x - 1) / blockDim.x;
    const int s0 = threadIdx.x * seg, s1 = min(V, s0 + seg);
    float part = 0.f;
    for (int t = s0; t < s1; ++t) part += R[t];
    double S;
    const double ex = block_exclusive_scan((double)part, &S, s_warp);
    if (threadIdx.x == 0) *s_tok = -1;
    __syncthreads();
    if (!(S > 0.0)) return -2;
    const double target = u * S;
    if (ex <= target && target < ex + (double)part) {
        float run = 0.f;
        for (int t = s0; t < s1; ++t) {
            const float prev = run;
            run += R[t];
            if (ex + (double)run > target) {
                *s_tok = t;
                s_c[0] = (ex + (double)prev) / S;
                s_c[1] = (ex + (double)run) / S;
                break;
            }
        }
    }
    __syncthreads();
    int tok = *s_tok;
    if (tok >= 0) {
        *near = fabs(s_c[0] - u) < kNearBand || fabs(s_c[1] - u) < kNearBand;
    } else {
        __syncthreads();
        int best = -1;
        for (int t = threadIdx.x; t < V; t += blockDim.x)
            if (R[t] > 0.f) best = t;
        if (best >= 0) atomicMax(s_tok, best);
        __syncthreads();
        tok = *s_tok;
        *near = true;
    }
    __syncthreads();
    return tok;
}

__global__ void __launch_bounds__(kTreeThreads) spec_accept_tree_kernel(const __grid_constant__ TreeArgs a) {
    extern __shared__ float R[];  // V fp32 residual weights
    __shared__ double s_warp[72];
    __shared__ double s_c[2];
    __shared__ int s_tok;
    const int b = blockIdx.x;
    const int V = a.V;
    const int32_t *tok = a.tokens + (size_t)b * a.n_nodes;
    int node = 0, depth = 0;
    bool near = false;
    int final_tok = -1;
    while (true) {
        const float *Pn = a.p + ((size_t)b * a.n_nodes + node) * V;
        const int qr = a.qrow[node];
        if (qr < 0) {
            for (int t = threadIdx.x; t < V; t += blockDim.x) R[t] = __ldg(Pn + t);
            __syncthreads();
            bool nb = false;
            final_tok = smem_draw(R, V, (double)__ldg(a.u_s + b), s_warp, &s_tok, s_c, &nb);
            near |= nb;
            break;
        }
        const float *Qn = a.q + ((size_t)b * a.n_internal + qr) * V;
        double Z = 1.0;
        int accepted = -1, tested = 0;
        for (int cnode = node + 1; cnode < a.n_nodes; ++cnode) {
            if (a.parent[cnode] != node) continue;
            int x = tok[cnode];
            if (x < 0 || x >= V) {
                if (threadIdx.x == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                x = 0;
            }
            const float u = __ldg(a.u_acc + (size_t)b * a.n_nodes + cnode);
            bool ok;
            if (tested == 0) {
                ok = __fmul_rn(u, __ldg(Qn + x)) <= __ldg(Pn + x);
            } else {
                const double lhs = (double)u * (double)__ldg(Qn + x) * Z;
                const double rx = (double)R[x];
                ok = lhs <= rx;
                if (Z > 0.0 && fabs(lhs - rx) / Z < kNearBand) near = true;
            }
            if (ok) {
                accepted = cnode;
                break;
            }
            // reject: R <- max(0, R - Z * Q), Z <- sum(R)
            const float zf = (float)Z;
            float part = 0.f;
            for (int t = threadIdx.x; t < V; t += blockDim.x) {
                const float prev = tested == 0 ? __ldg(Pn + t) : R[t];
                const float v = prev - zf * __ldg(Qn + t);
                const float r = v > 0.f ? v : 0.f;
                R[t] = r;
                part += r;
            }
            ++tested;
            Z = block_sum((double)part, s_warp);
        }
        if (accepted >= 0) {
            ++depth;
            if (threadIdx.x == 0) {
                a.path_nodes[(size_t)b * a.width + depth] = accepted;
                a.out_tokens[(size_t)b * a.width + depth - 1] = tok[accepted];
            }
            node = accepted;
            continue;
        }
        bool nb = false;
        final_tok = smem_draw(R, V, (double)__ldg(a.u_s + b), s_warp, &s_tok, s_c, &nb);
        if (final_tok == -2) {  // empty residual: draw from the node's target row
            for (int t = threadIdx.x; t < V; t += blockDim.x) R[t] = __ldg(Pn + t);
            __syncthreads();
            final_tok = smem_draw(R, V, (double)__ldg(a.u_s + b), s_warp, &s_tok, s_c, &nb);
        }
        near |= nb;
        break;
    }
    if (final_tok < 0) {
        if (threadIdx.x == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        final_tok = 0;
    }
    if (threadIdx.x == 0) {
        int32_t *path = a.path_nodes + (size_t)b * a.width;
        int32_t *out = a.out_tokens + (size_t)b * a.width;
        path[0] = 0;
        for (int d = depth + 1; d < a.width; ++d) path[d] = -1;
        out[depth] = final_tok;
        for (int d = depth + 1; d < a.width; ++d) out[d] = -1;
        a.accepted_len[b] = depth;
        if (a.near) a.near[b] = near ? 1 : 0;
    }
}

}  // namespace

cudaError_t launch_spec_accept(const AcceptArgs &a, cudaStream_t stream) {
    spec_accept_kernel<<<a.B, kRowThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// The row sampler keeps no state between CTAs: its workspace is a stub.
int spec_accept_chunks(int vocab) {
    (void)vocab;
    return 1;
}

cudaError_t launch_spec_accept_tree(const TreeArgs &a, cudaStream_t stream) {
    const size_t smem = (size_t)a.V * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(spec_accept_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    spec_accept_tree_kernel<<<a.B, kTreeThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace svpa
