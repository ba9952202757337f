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
// GB300 layout.  A row is one sequence: a few gathered loads for the
// acceptance tests, then one pass over a V-token residual row.  One CTA per
// row leaves most SMs idle and caps a row at what one SM can pull from
// memory, so the row is split across a thread-block cluster of up to 8 CTAs
// (one contiguous slice each).  Each CTA runs the acceptance tests itself
// (the same loads, hence the same k), sums its slice with coalesced 16-byte
// loads (fp32 per 4-token lane group, fp32 per warp, fp64 across warps), and
// the CTA totals are exchanged through distributed shared memory.  The CTA
// whose slice holds u*S narrows the target down warp -> 128-token step ->
// lane -> token, re-reading only the 128 tokens of one step.  The GB300 fp64
// pipe retires two lanes per clock per SM, so fp64 is kept to a handful of
// scalar operations per CTA.  Vocabularies beyond 262144 tokens take a
// one-CTA-per-row kernel.
//
// Also here: the draft-tree sampler on the same cluster split, the linear
// sampler fed by logits (softmax rows formed in the kernels: slab
// statistics, then the cluster sampler on a logits weight source), and the
// draft-tree sampler fed by logits (the statistics of the visited rows only,
// formed by the cluster at each node of the walk).
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

// ---------------------------------------------------------------- cluster rows
// A row is split into n_ctas <= 8 contiguous slices of kClWarps * NI * 128
// tokens, one per CTA of a cluster.  Warp w of CTA c owns NI steps of 128
// tokens; in step i lane l owns tokens [base + 128 i + 4 l, +4).
constexpr int kClWarps = 8;
constexpr int kClThreads = kClWarps * 32;
constexpr int kClMaxCtas = 8;
constexpr int kStep = 128;
constexpr int kClMaxSteps = 32;
constexpr int kLoadBatch = 4;
constexpr int kClCtasPerSm = 4;  // resident CTAs per SM the kernels are built for
constexpr int kClMaxVocab = kClMaxCtas * kClWarps * kClMaxSteps * kStep;  // 262144

enum : int { kDrawFound = 0, kDrawPastEnd = 1, kDrawNoMass = 2 };

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// The cluster's start-up barrier, split: every CTA arrives on entry and waits
// before its first store into a peer's shared memory, by which time every
// CTA of the cluster has started (the wait is normally long satisfied).
__device__ __forceinline__ void cluster_arrive_on_entry() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_started() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    return remote;
}

// Stores into the word at the same shared-memory offset as `p` in the CTA of
// cluster rank `rank`.  The exchanges push every CTA's values into every
// peer before a cluster barrier (release / acquire), so that after the
// barrier each CTA reads them from its own shared memory, and no CTA touches
// a peer's shared memory after the cluster's last barrier (a CTA may then
// exit without waiting for its peers).
__device__ __forceinline__ void st_peer_f64(double *p, uint32_t rank, double v) {
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(peer_addr(p, rank)), "d"(v) : "memory");
}
__device__ __forceinline__ void st_peer_f32(float *p, uint32_t rank, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(peer_addr(p, rank)), "f"(v) : "memory");
}

__device__ __forceinline__ float lane_sum(float4 w) { return ((w.x + w.y) + w.z) + w.w; }

__device__ __forceinline__ float warp_incl_scan(float s) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
    }
    return s;
}

__device__ __forceinline__ float relu(float d) { return d > 0.f ? d : 0.f; }

// Weight sources.  operator()(t0) gives the weights of tokens t0..t0+3 (t0 a
// multiple of 4; 0 past V); at(t) the weight of one token.
// max(0, P - Q) in fp32, or P when q == nullptr, read from global memory.
struct SrcGlobal {
    const float *p, *q;
    int V;
    bool vec;  // rows 16-byte aligned and V % 4 == 0
    __device__ float4 operator()(int t0) const {
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vec) {
            if (t0 < V) {
                w = __ldg(reinterpret_cast<const float4 *>(p + t0));
                if (q) {
                    const float4 v = __ldg(reinterpret_cast<const float4 *>(q + t0));
                    w = make_float4(relu(w.x - v.x), relu(w.y - v.y), relu(w.z - v.z), relu(w.w - v.w));
                }
            }
        } else {
            if (t0 < V) w.x = at(t0);
            if (t0 + 1 < V) w.y = at(t0 + 1);
            if (t0 + 2 < V) w.z = at(t0 + 2);
            if (t0 + 3 < V) w.w = at(t0 + 3);
        }
        return w;
    }
    __device__ float at(int t) const { return weight(p, q, t); }
};

// A residual slice held in shared memory (tokens [lo, lo + slice)).
struct SrcSmem {
    const float *R;
    int lo;
    __device__ float4 operator()(int t0) const { return *reinterpret_cast<const float4 *>(R + (t0 - lo)); }
    __device__ float at(int t) const { return R[t - lo]; }
};

// Tree rejection update R <- max(0, prev - zf * Q) in fp32 (product rounded,
// never fused), prev = P on a node's first rejection, else R; stores the new
// R slice and returns it.
struct SrcUpdate {
    float *R;
    const float *p;  // nullptr: prev = R
    const float *q;
    int lo, V;
    float zf;
    bool vec;
    __device__ float4 operator()(int t0) const {
        float4 prev, qv;
        if (vec) {
            prev = make_float4(0.f, 0.f, 0.f, 0.f);
            qv = prev;
            if (t0 < V) {
                prev = p ? __ldg(reinterpret_cast<const float4 *>(p + t0))
                         : *reinterpret_cast<const float4 *>(R + (t0 - lo));
                qv = __ldg(reinterpret_cast<const float4 *>(q + t0));
            }
        } else {
            float pv[4], qq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pv[j] = 0.f;
                qq[j] = 0.f;
                if (t0 + j < V) {
                    pv[j] = p ? __ldg(p + t0 + j) : R[t0 + j - lo];
                    qq[j] = __ldg(q + t0 + j);
                }
            }
            prev = make_float4(pv[0], pv[1], pv[2], pv[3]);
            qv = make_float4(qq[0], qq[1], qq[2], qq[3]);
        }
        const float4 r = make_float4(relu(prev.x - __fmul_rn(zf, qv.x)), relu(prev.y - __fmul_rn(zf, qv.y)),
                                     relu(prev.z - __fmul_rn(zf, qv.z)), relu(prev.w - __fmul_rn(zf, qv.w)));
        *reinterpret_cast<float4 *>(R + (t0 - lo)) = r;
        return r;
    }
};

// Per-CTA state of the cluster-wide sums and draw of one row.
template <int NI>
struct ClusterRow {
    float g[kClWarps][NI];        // per-step sums (fp32)
    float wsum[kClWarps];         // per-warp sums (fp32, steps in order)
    double wincl[kClWarps];       // inclusive fp64 prefix of the warp sums
    double total;                 // this CTA's slice total
    double peer[2][kClMaxCtas];   // every CTA's slice total by exchange parity, pushed by each CTA
    double pincl[kClMaxCtas];     // inclusive prefix of the last exchange's totals (rank order)
    float probe[2];               // R at a probed token by exchange parity, pushed by its owner
    double S, r;
    float probe_val;
    int cta, mode, warp, tok, near, slot, last;
};

// The weights a thread loaded for its NI steps in cluster_sum, kept in
// registers for cluster_draw when the row is short enough (KEEP); the draw
// then scans its step from these instead of loading it again.
template <int NI, bool KEEP>
struct Kept {
    float4 v[KEEP ? NI : 1];
};
template <int NI>
constexpr bool kKeepWeights = NI <= 4;

struct ClusterGeom {
    int rank, n_ctas, cta_lo, cta_hi, wbase;
};

// Sums the row's weights over the cluster; returns the row total S (the same
// double in every CTA).  When probe >= 0 the CTA owning token `probe` also
// publishes R[probe] from `R` (after the sums), readable as st.probe_val.
// Every thread of every CTA of the cluster calls this, with the same parity.
template <int NI, class Src, bool KEEP = false>
__device__ __forceinline__ double cluster_sum(ClusterRow<NI> &st, const Src &src, const ClusterGeom &g,
                                              int parity, int probe, const float *R, Kept<NI, KEEP> &keep) {
    constexpr int nb = NI < kLoadBatch ? NI : kLoadBatch;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float G = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < NI; i0 += nb) {
        float4 wv[nb];
#pragma unroll
        for (int j = 0; j < nb; ++j) wv[j] = src(g.wbase + (i0 + j) * kStep + 4 * lane);
#pragma unroll
        for (int j = 0; j < nb; ++j) {
            const float s = __shfl_sync(0xffffffffu, warp_incl_scan(lane_sum(wv[j])), 31);
            if (lane == 0) st.g[warp][i0 + j] = s;
            G += s;
            if constexpr (KEEP) keep.v[i0 + j] = wv[j];
        }
    }
    if (lane == 0) st.wsum[warp] = G;
    __syncthreads();
    const int owner = probe >= 0 ? probe / (kClWarps * NI * kStep) : -1;
    if (threadIdx.x < 32) {
        // inclusive fp64 prefix of the warp sums (a 3-step scan over lanes
        // 0..7); the CTA total is its last entry
        double v = lane < kClWarps ? (double)st.wsum[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < kClWarps; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane < kClWarps) st.wincl[lane] = v;
        const double total = __shfl_sync(0xffffffffu, v, kClWarps - 1);
        if (lane == 0) {
            st.total = total;
            st.last = parity;
        }
        // push this CTA's total (and the probed R value from its owner) into every CTA
        if (lane < g.n_ctas) {
            st_peer_f64(&st.peer[parity][g.rank], (uint32_t)lane, total);
            if (owner == g.rank) st_peer_f32(&st.probe[parity], (uint32_t)lane, R[probe - g.cta_lo]);
        }
    }
    cluster_sync_all();
    if (threadIdx.x < 32) {
        // the totals in rank order, by the same scan in every CTA: the row
        // total S is the last entry of the prefix
        double v = lane < g.n_ctas ? st.peer[parity][lane] : 0.0;
#pragma unroll
        for (int o = 1; o < kClMaxCtas; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane < kClMaxCtas) st.pincl[lane] = v;
        const double S = __shfl_sync(0xffffffffu, v, kClMaxCtas - 1);
        if (lane == 0) {
            st.S = S;
            if (owner >= 0) st.probe_val = st.probe[parity];
        }
    }
    __syncthreads();
    return st.S;
}

template <int NI, class Src>
__device__ __forceinline__ double cluster_sum(ClusterRow<NI> &st, const Src &src, const ClusterGeom &g,
                                              int parity, int probe = -1, const float *R = nullptr) {
    Kept<NI, false> none;
    return cluster_sum<NI, Src, false>(st, src, g, parity, probe, R, none);
}

// Last token in [lo, hi) with positive weight, or -1 (the whole CTA calls it).
template <class Src>
__device__ int cta_last_positive(const Src &src, int lo, int hi, int *s_slot) {
    if (threadIdx.x == 0) *s_slot = -1;
    __syncthreads();
    int best = -1;
    for (int t = lo + (int)threadIdx.x; t < hi; t += blockDim.x)
        if (src.at(t) > 0.f) best = t;
    if (best >= 0) atomicMax(s_slot, best);
    __syncthreads();
    return *s_slot;
}

// Inverse-CDF draw after cluster_sum over the same weights: the first token
// whose running mass exceeds u*S.  Returns true in the one CTA that made the
// draw (tok, near set there); tok = -1 there when the row has no mass (then
// it is CTA 0).  near: u*S within 1e-6 * S of a running sum, or within
// band_abs when that is given.  Every thread of every CTA calls this.
template <int NI, class Src, bool KEEP = false>
__device__ bool cluster_draw(ClusterRow<NI> &st, const Src &src, const ClusterGeom &g, float u, int *tok_out,
                             bool *near_out, double band_abs, const Kept<NI, KEEP> &keep) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // which CTA holds u*S: the first whose running total exceeds it (warp 0,
    // all ranks compared at once)
    if (threadIdx.x < 32) {
        const double S = st.S, target = (double)u * S;
        int mode = kDrawNoMass, cta = 0;
        double before = 0.0;
        if (S > 0.0) {
            const unsigned hit = __ballot_sync(0xffffffffu, lane < g.n_ctas && st.pincl[lane] > target);
            if (hit) {
                cta = __ffs(hit) - 1;
                before = cta > 0 ? st.pincl[cta - 1] : 0.0;
                mode = kDrawFound;
            } else {  // u*S at or past S (rounding): the last CTA with mass
                const unsigned pos = __ballot_sync(0xffffffffu, lane < g.n_ctas && st.peer[st.last][lane] > 0.0);
                cta = pos ? 31 - __clz(pos) : -1;
                mode = kDrawPastEnd;
            }
        }
        if (lane == 0) {
            st.mode = mode;
            st.cta = cta;
            st.r = target - before;
        }
    }
    __syncthreads();
    const int mode = st.mode;
    if (g.rank != st.cta) return false;
    if (mode == kDrawNoMass) {
        *tok_out = -1;
        *near_out = true;
        return true;
    }
    int tok;
    bool near = true;
    if (mode == kDrawFound) {
        // warp (all eight compared at once), then 128-token step, then lane,
        // then token
        if (threadIdx.x < 32) {
            const double r1 = st.r;
            const unsigned hit = __ballot_sync(0xffffffffu, lane < kClWarps && st.wincl[lane] > r1);
            const int ws = hit ? __ffs(hit) - 1 : -1;
            if (lane == 0) {
                st.warp = ws;
                st.r = r1 - (ws > 0 ? st.wincl[ws - 1] : 0.0);
                st.tok = -2;
                st.near = 1;
            }
        }
        __syncthreads();
        const int ws = st.warp;
        const int wlo = g.cta_lo + (ws < 0 ? 0 : ws) * NI * kStep;
        if (warp == ws) {
            // the running fp32 sums over the steps in cluster_sum's order, the
            // comparisons independent of one another
            const double r2 = st.r;
            float G = 0.f, Gs = 0.f;
            int step = -1;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const float Gn = G + st.g[ws][i];
                if (step < 0 && (double)Gn > r2) {
                    step = i;
                    Gs = G;
                }
                G = Gn;
            }
            G = Gs;
            if (step >= 0) {
                const int t0 = wlo + step * kStep + 4 * lane;
                float4 wv;
                if constexpr (KEEP) {  // this lane loaded these weights in cluster_sum
                    wv = keep.v[0];
#pragma unroll
                    for (int i = 1; i < NI; ++i)
                        if (i == step) wv = keep.v[i];
                } else {
                    wv = src(t0);
                }
                const float incl = warp_incl_scan(lane_sum(wv));
                float excl = __shfl_up_sync(0xffffffffu, incl, 1);
                if (lane == 0) excl = 0.f;
                const unsigned hit = __ballot_sync(0xffffffffu, (double)(G + incl) > r2);
                const int l = hit ? __ffs(hit) - 1 : 31;
                if (lane == l) {
                    const float wj[4] = {wv.x, wv.y, wv.z, wv.w};
                    const double band = band_abs >= 0.0 ? band_abs : kNearBand * st.S;
                    float c = G + excl;
                    int found = -1, lastpos = -1;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (wj[j] > 0.f) lastpos = j;
                        const float cn = c + wj[j];
                        if (found < 0 && (double)cn > r2) {
                            found = j;
                            st.near = (fabs((double)c - r2) < band || fabs((double)cn - r2) < band) ? 1 : 0;
                        }
                        c = cn;
                    }
                    // found < 0: a rounding gap between levels (u*S within
                    // a few fp32 ulps of this group's end): its last token
                    st.tok = found >= 0 ? t0 + found : (lastpos >= 0 ? t0 + lastpos : -2);
                }
            }
        }
        __syncthreads();
        tok = st.tok;
        near = st.near != 0;
        if (tok == -2) {
            // rounding gap at the CTA or warp level: the last token with mass
            // in that range
            const int lo = ws < 0 ? g.cta_lo : wlo;
            const int hi = ws < 0 ? g.cta_hi : min(g.cta_hi, wlo + NI * kStep);
            tok = cta_last_positive(src, lo, hi, &st.slot);
            near = true;
        }
    } else {  // kDrawPastEnd
        tok = cta_last_positive(src, g.cta_lo, g.cta_hi, &st.slot);
    }
    *tok_out = tok;
    *near_out = near;
    return true;
}

template <int NI, class Src>
__device__ __forceinline__ bool cluster_draw(ClusterRow<NI> &st, const Src &src, const ClusterGeom &g, float u,
                                             int *tok_out, bool *near_out, double band_abs = -1.0) {
    const Kept<NI, false> none{};
    return cluster_draw<NI, Src, false>(st, src, g, u, tok_out, near_out, band_abs, none);
}

template <int NI>
__device__ __forceinline__ ClusterGeom cluster_geom(int V, int n_ctas) {
    ClusterGeom g;
    g.rank = (int)(blockIdx.x % (unsigned)n_ctas);
    g.n_ctas = n_ctas;
    g.cta_lo = g.rank * (kClWarps * NI * kStep);
    g.cta_hi = min(V, g.cta_lo + kClWarps * NI * kStep);
    g.wbase = g.cta_lo + (int)(threadIdx.x >> 5) * NI * kStep;
    return g;
}

// ---------------------------------------------------------------- linear, cluster per row
template <int NI>
__global__ void __launch_bounds__(kClThreads, kClCtasPerSm)
    spec_accept_cluster_kernel(const __grid_constant__ AcceptArgs a, int n_ctas) {
    __shared__ ClusterRow<NI> st;
    __shared__ int s_k;
    __shared__ float s_u;
    const ClusterGeom g = cluster_geom<NI>(a.V, n_ctas);
    const int b = (int)(blockIdx.x / (unsigned)n_ctas);
    const int gamma = a.gamma, V = a.V;
    const int lane = threadIdx.x & 31;
    cluster_arrive_on_entry();

    // acceptance tests: every CTA of the cluster makes the same loads and
    // reaches the same k
    if (threadIdx.x < 32) {
        bool rejected = false;
        if (lane < gamma) {
            int x = a.tokens[(size_t)b * gamma + lane];
            if (x < 0 || x >= V) {
                if (g.rank == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                x = 0;
            }
            const float qx = __ldg(a.q + ((size_t)b * gamma + lane) * V + x);
            const float px = __ldg(a.p + ((size_t)b * (gamma + 1) + lane) * V + x);
            const float u = __ldg(a.u_acc + (size_t)b * gamma + lane);
            rejected = !(__fmul_rn(u, qx) <= px);
        }
        const unsigned rej = __ballot_sync(0xffffffffu, rejected);
        if (lane == 0) {
            s_k = rej ? __ffs(rej) - 1 : gamma;
            s_u = __ldg(a.u_s + b);
        }
    }
    __syncthreads();
    const int k = s_k;
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.p) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
    SrcGlobal src{a.p + ((size_t)b * (gamma + 1) + k) * V, k < gamma ? a.q + ((size_t)b * gamma + k) * V : nullptr,
                  V, vec};
    cluster_wait_started();
    Kept<NI, kKeepWeights<NI>> keep;
    double S = cluster_sum(st, src, g, 0, -1, nullptr, keep);
    if (!(S > 0.0) && src.q) {
        // empty residual: draw from the target row instead (S is the same in
        // every CTA, so the whole cluster takes this branch)
        src.q = nullptr;
        S = cluster_sum(st, src, g, 1, -1, nullptr, keep);
    }
    int tok;
    bool near;
    if (cluster_draw(st, src, g, s_u, &tok, &near, -1.0, keep) && threadIdx.x == 0) {
        if (tok < 0) {  // a row with no mass
            raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            tok = 0;
        }
        a.out_tokens[(size_t)b * (gamma + 1) + k] = tok;
        if (a.near) a.near[b] = near ? 1 : 0;
    }
    if (g.rank == 0) {
        const int i = threadIdx.x;
        if (i <= gamma && i != k)
            a.out_tokens[(size_t)b * (gamma + 1) + i] = i < k ? a.tokens[(size_t)b * gamma + i] : -1;
        if (i == 0) a.accepted_len[b] = k;
    }
    // no peer touches this CTA's shared memory after the last exchange: no
    // closing cluster barrier
}

// ---------------------------------------------------------------- tree, cluster per row
// Multi-draft recursion along the tree ("Tree Attention Mechanism" and the
// rejection-recovery step of the same page): at a node with children
// c_1..c_m (node order) and draft distribution Q, child c_1 is accepted iff
// u * Q(x) <= P(x) (fp32, as in the linear sampler); after a rejection the
// residual becomes R <- max(0, R - Z * Q) with Z = sum(R) (R = P before the
// first rejection, Z = 1), and child c_j (j > 1) is accepted iff
// u * Q(x) * Z <= R(x).  An accepted child becomes the node; when every
// child is rejected the token is drawn from R (from P when R is empty), and a
// leaf draws its bonus token from its own P.  The residual slice lives in
// each CTA's shared memory; R(x) for the next sibling is published by the
// CTA that owns x along with the slice sums.
template <int NI>
__global__ void __launch_bounds__(kClThreads, kClCtasPerSm)
    spec_accept_tree_cluster_kernel(const __grid_constant__ TreeArgs a, int n_ctas) {
    extern __shared__ float4 dyn_smem[];
    float *R = reinterpret_cast<float *>(dyn_smem);  // this CTA's residual slice
    __shared__ ClusterRow<NI> st;
    const ClusterGeom g = cluster_geom<NI>(a.V, n_ctas);
    const int b = (int)(blockIdx.x / (unsigned)n_ctas);
    const int V = a.V, n_nodes = a.n_nodes;
    const int32_t *ntok = a.tokens + (size_t)b * n_nodes;
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.p) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
    const bool lead = g.rank == 0 && threadIdx.x == 0;
    cluster_arrive_on_entry();
    // the row's node tokens and uniforms, and for every node c > 0 Q(x_c) and
    // P(x_c) in the rows of its parent (the tree is known up front, so these
    // gathers are made once, all in flight together, rather than one
    // dependent round of loads per visited node; parents precede their
    // children and every parent has a draft row)
    __shared__ int s_x[kMaxNq];
    __shared__ float s_ua[kMaxNq], s_qx[kMaxNq], s_px[kMaxNq];
    if (threadIdx.x < (unsigned)n_nodes) {
        const int c = (int)threadIdx.x;
        int x = ntok[c];
        if (x < 0 || x >= V) {
            if (g.rank == 0 && c > 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            x = 0;
        }
        s_x[c] = x;
        s_ua[c] = __ldg(a.u_acc + (size_t)b * n_nodes + c);
        if (c > 0) {
            const int pn = a.parent[c];
            s_qx[c] = __ldg(a.q + ((size_t)b * a.n_internal + a.qrow[pn]) * V + x);
            s_px[c] = __ldg(a.p + ((size_t)b * n_nodes + pn) * V + x);
        }
    }
    const float u_s = __ldg(a.u_s + b);
    __syncthreads();
    cluster_wait_started();
    int node = 0, depth = 0, parity = 0;
    bool near = false;
    int tok = -1;
    bool drew;
    while (true) {
        const float *Pn = a.p + ((size_t)b * n_nodes + node) * V;
        const int qr = a.qrow[node];
        if (qr < 0) {  // leaf: bonus token from its own P
            const SrcGlobal src{Pn, nullptr, V, vec};
            Kept<NI, kKeepWeights<NI>> keep;
            cluster_sum(st, src, g, parity, -1, nullptr, keep);
            parity ^= 1;
            bool nb = false;
            drew = cluster_draw(st, src, g, u_s, &tok, &nb, -1.0, keep);
            near |= nb;
            break;
        }
        const float *Qn = a.q + ((size_t)b * a.n_internal + qr) * V;
        double Z = 1.0;
        float rx = 0.f;  // R(x) of the child under test, after a rejection
        int accepted = -1, tested = 0;
        for (int c = node + 1; c < n_nodes; ++c) {
            if (a.parent[c] != node) continue;
            const float u = s_ua[c];
            bool ok;
            if (tested == 0) {
                ok = __fmul_rn(u, s_qx[c]) <= s_px[c];
            } else {
                const double lhs = (double)u * (double)s_qx[c] * Z;
                ok = lhs <= (double)rx;
                // within 1e-6 of the threshold in normalised units (no fp64 division)
                if (Z > 0.0 && fabs(lhs - (double)rx) < kNearBand * Z) near = true;
            }
            if (ok) {
                accepted = c;
                break;
            }
            int xn = -1;  // the next sibling's token: R is probed there
            for (int c2 = c + 1; c2 < n_nodes; ++c2)
                if (a.parent[c2] == node) {
                    xn = s_x[c2];
                    break;
                }
            const SrcUpdate upd{R, tested == 0 ? Pn : nullptr, Qn, g.cta_lo, V, (float)Z, vec};
            Z = cluster_sum(st, upd, g, parity, xn, R);
            parity ^= 1;
            rx = st.probe_val;
            ++tested;
        }
        if (accepted >= 0) {
            ++depth;
            if (lead) {
                a.path_nodes[(size_t)b * a.width + depth] = accepted;
                a.out_tokens[(size_t)b * a.width + depth - 1] = s_x[accepted];
            }
            node = accepted;
            continue;
        }
        bool nb = false;
        if (Z > 0.0) {
            drew = cluster_draw(st, SrcSmem{R, g.cta_lo}, g, u_s, &tok, &nb);
        } else {  // empty residual: draw from the node's target row
            const SrcGlobal src{Pn, nullptr, V, vec};
            Kept<NI, kKeepWeights<NI>> keep;
            cluster_sum(st, src, g, parity, -1, nullptr, keep);
            parity ^= 1;
            drew = cluster_draw(st, src, g, u_s, &tok, &nb, -1.0, keep);
        }
        near |= nb;
        break;
    }
    if (drew && threadIdx.x == 0) {
        if (tok < 0) {  // a row with no mass
            raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            tok = 0;
        }
        a.out_tokens[(size_t)b * a.width + depth] = tok;
        if (a.near) a.near[b] = near ? 1 : 0;
    }
    if (lead) {
        int32_t *path = a.path_nodes + (size_t)b * a.width;
        int32_t *out = a.out_tokens + (size_t)b * a.width;
        path[0] = 0;
        for (int d = depth + 1; d < a.width; ++d) {
            path[d] = -1;
            out[d] = -1;
        }
        a.accepted_len[b] = depth;
    }
    // no peer touches this CTA's shared memory after the last exchange
}

// ---------------------------------------------------------------- logits front-end
// The sampler fed by logits: P_i = softmax(Lp_i / T), Q_i = softmax(Lq_i /
// T_draft) are never written out.  "Speculative Decoding and KV-Cache
// Compression", section 2.3 (the acceptance ratio takes softmax(logits)[x]);
// "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING", architecture
// (target logits checked against draft logits).
//
// Two kernels.  logit_stats_kernel reads every logit once, one CTA per
// 8192-token slab of a row (independent CTAs, so the read runs at memory
// speed whatever the batch), and writes the slab's max m and sum s of
// 2^((l - m) c), c = log2(e) / T.  The sampler kernel, launched as its
// programmatic dependent, is the linear sampler's cluster kernel: it loads
// the draft tokens, their logits and the uniforms while the statistics grid
// runs, then each CTA merges every row's slab pairs in a fixed order (a
// half-warp butterfly per row), so all CTAs of a cluster hold the same
// maxima and normalisers; the acceptance tests use P(x) = 2^((l_x - m) c) /
// S formed in fp32 exactly as the residual's weights, and the residual row k
// is read again (from L2) with its weights formed in fp32 for the cluster
// sum and draw.  The GB300 fp64 pipe has a 64-cycle dependent latency and a
// ~1400-cycle division, so nothing on this latency chain but the cluster
// sums is fp64.
//
// fp32 formation errs by ~1.2e-7 * |log2 P| relative per probability (the
// exponent's rounding; <= 1.3e-5 down to 2^-100) plus <= ~1e-5 in the
// normaliser (partial sums of 16 terms per thread, fp32 merges within a
// slab and across at most 32 slabs), so decisions within 5e-5 of their thresholds are
// reported as near: a test with |u Q - P| <= 5e-5 * max(P, u Q) (or both below
// 2^-100), a residual with mass below 5e-5, a draw within 5e-5 (absolute) of a
// running sum.
constexpr int kMaxLogitRows = 2 * 32 + 1;
constexpr int kSlab = 8192;                          // tokens per statistics CTA
constexpr int kMaxSlabs = kClMaxVocab / kSlab;       // 32
constexpr double kLogitBand = 5e-5;
constexpr double kLogitTiny = 7.888609052210118e-31;  // 2^-100
constexpr float kLogitBandF = 5e-5f;
constexpr float kLogitTinyF = 7.888609052210118e-31f;  // 2^-100, a normal fp32 value

// Four logits of a row from token t0 (a multiple of 4); -inf past V.
__device__ __forceinline__ float4 load_logits4(const float *row, int t0, int V, bool vec) {
    float4 w = make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
    if (vec) {
        if (t0 < V) w = __ldg(reinterpret_cast<const float4 *>(row + t0));
    } else {
        if (t0 < V) w.x = __ldg(row + t0);
        if (t0 + 1 < V) w.y = __ldg(row + t0 + 1);
        if (t0 + 2 < V) w.z = __ldg(row + t0 + 2);
        if (t0 + 3 < V) w.w = __ldg(row + t0 + 3);
    }
    return w;
}

// (m, s) of sixteen logits (four float4): the max of all sixteen, then their
// exponentials (independent of one another) summed as a tree.  -inf entries
// add nothing; an all -inf group gives (-inf, 0).
__device__ __forceinline__ void group_stats16(const float4 (&w)[4], float c, float &m, float &s) {
    m = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fmaxf(w[i].x, w[i].y), fmaxf(w[i].z, w[i].w)));
    s = 0.f;
    if (m > -CUDART_INF_F) {
        float e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            e[i] = (ex2_approx((w[i].x - m) * c) + ex2_approx((w[i].y - m) * c)) +
                   (ex2_approx((w[i].z - m) * c) + ex2_approx((w[i].w - m) * c));
        s = (e[0] + e[1]) + (e[2] + e[3]);
    }
}

// (m, s) <- the merge of (m, s) and (m2, s2).
__device__ __forceinline__ void online_merge(float &m, float &s, float m2, float s2, float c) {
    if (m2 > m) {
        s = s * ex2_approx((m - m2) * c) + s2;
        m = m2;
    } else if (m2 > -CUDART_INF_F) {
        s = s + s2 * ex2_approx((m2 - m) * c);
    }
}

// Row r of sequence b: target rows 0..gamma, draft rows gamma+1..2 gamma.
__device__ __forceinline__ const float *logit_row(const LogitsArgs &a, int b, int r) {
    return r <= a.gamma ? a.lp + ((size_t)b * (a.gamma + 1) + r) * a.V
                        : a.lq + ((size_t)b * a.gamma + (r - a.gamma - 1)) * a.V;
}

// One CTA of 128 threads per (sequence, row, slab): the slab's (max, sum)
// into a.stats.  Each thread reduces 64 logits in two batches of eight
// float4 loads (a batch's loads all in flight together).  At 48 registers
// ten CTAs fit on an SM, so the 7B sampler shape's 1152 slabs run as one
// wave.
constexpr int kStatThreads = 128;
constexpr int kStatWarps = kStatThreads / 32;
static_assert(kSlab == kStatThreads * 64, "a statistics CTA covers one slab");
__global__ void __launch_bounds__(kStatThreads) logit_stats_kernel(const __grid_constant__ LogitsArgs a) {
    // the sampler may be scheduled now; it waits for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ float s_wm[kStatWarps], s_ws[kStatWarps];
    const int rows = 2 * a.gamma + 1;
    const int slab = (int)(blockIdx.x % (unsigned)a.n_slabs);
    const int br = (int)(blockIdx.x / (unsigned)a.n_slabs);  // b * rows + r
    const int b = br / rows, r = br - b * rows;
    const float *row = logit_row(a, b, r);
    const float c = r <= a.gamma ? a.c_target : a.c_draft;
    const bool vec = (a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.lp) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.lq) & 15) == 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float m = -CUDART_INF_F, s = 0.f, m2, s2;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 w[2][4];
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[g][i] = load_logits4(row, slab * kSlab + 4 * ((int)threadIdx.x + (8 * h + 4 * g + i) * kStatThreads),
                                       a.V, vec);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            group_stats16(w[g], c, m2, s2);
            online_merge(m, s, m2, s2, c);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        m2 = __shfl_xor_sync(0xffffffffu, m, o);
        s2 = __shfl_xor_sync(0xffffffffu, s, o);
        online_merge(m, s, m2, s2, c);
    }
    if (lane == 0) {
        s_wm[warp] = m;
        s_ws[warp] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = s_wm[0], ss = s_ws[0];
        for (int i = 1; i < kStatWarps; ++i) online_merge(mm, ss, s_wm[i], s_ws[i], c);
        a.stats[(size_t)br * a.n_slabs + slab] = make_float2(mm, ss);
    }
}

// Residual weights from logits: max(0, P - Q) in fp32 with P = 2^((l - mp)
// cp) * ip (ip = 1/S rounded to fp32), likewise Q; P alone when q == nullptr.
struct SrcLogits {
    const float *p, *q;
    int V;
    bool vec;
    float mp, cp, ip, mq, cq, iq;
    __device__ float prob_p(float l) const { return ex2_approx((l - mp) * cp) * ip; }
    __device__ float prob_q(float l) const { return ex2_approx((l - mq) * cq) * iq; }
    __device__ float4 operator()(int t0) const {
        if (t0 >= V) return make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 lp = load_logits4(p, t0, V, vec);
        float4 w = make_float4(prob_p(lp.x), prob_p(lp.y), prob_p(lp.z), prob_p(lp.w));
        if (q) {
            const float4 lq = load_logits4(q, t0, V, vec);
            w = make_float4(relu(w.x - prob_q(lq.x)), relu(w.y - prob_q(lq.y)), relu(w.z - prob_q(lq.z)),
                            relu(w.w - prob_q(lq.w)));
        }
        return w;
    }
    __device__ float at(int t) const {
        const float pv = prob_p(__ldg(p + t));
        return q ? relu(pv - prob_q(__ldg(q + t))) : pv;
    }
};

template <int NI>
__global__ void __launch_bounds__(kClThreads, kClCtasPerSm)
    spec_accept_logits_cluster_kernel(const __grid_constant__ LogitsArgs a, int n_ctas) {
    __shared__ ClusterRow<NI> st;
    __shared__ float s_m[kMaxLogitRows], s_inv[kMaxLogitRows];  // row max, 1 / row sum (fp32)
    __shared__ int s_k, s_near;
    __shared__ float s_u;
    const ClusterGeom g = cluster_geom<NI>(a.V, n_ctas);
    const int b = (int)(blockIdx.x / (unsigned)n_ctas);
    const int gamma = a.gamma, V = a.V, rows = 2 * gamma + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.lp) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.lq) & 15) == 0;
    cluster_arrive_on_entry();
    // the inputs the statistics grid does not write (draft tokens, their two
    // logits, the uniforms) are loaded while that grid still runs
    float lpx = 0.f, lqx = 0.f, ua = 0.f;
    if (threadIdx.x < 32 && lane < gamma) {
        int x = a.tokens[(size_t)b * gamma + lane];
        if (x < 0 || x >= V) {
            if (g.rank == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            x = 0;
        }
        lpx = __ldg(logit_row(a, b, lane) + x);
        lqx = __ldg(logit_row(a, b, gamma + 1 + lane) + x);
        ua = __ldg(a.u_acc + (size_t)b * gamma + lane);
    }
    if (threadIdx.x == 32) s_u = __ldg(a.u_s + b);
    // the slab statistics are complete once the statistics grid is
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- row maxima and normalisers: half-warp h of the CTA merges rows h,
    // h + 16, ...; lane l of the half holds slabs l and l + 16; max by
    // butterfly, then the rescaled sums by butterfly (fp32, the same order in
    // every CTA; at most 32 terms, so the sum errs by < 2e-6 relative)
    const int nsl = a.n_slabs;
    const int hl = lane & 15;
    // the loop is uniform over the warp (both halves run every iteration and
    // every shuffle; a half past the last row works on an empty row)
    for (int r0 = 2 * warp; r0 < rows; r0 += 2 * kClWarps) {
        const int r = r0 + (lane >> 4);
        const bool row_ok = r < rows;
        const float c = r <= gamma ? a.c_target : a.c_draft;
        const float2 *ps = a.stats + ((size_t)b * rows + r) * nsl;
        const float2 p0 = row_ok && hl < nsl ? ps[hl] : make_float2(-CUDART_INF_F, 0.f);
        const float2 p1 = row_ok && hl + 16 < nsl ? ps[hl + 16] : make_float2(-CUDART_INF_F, 0.f);
        float m = fmaxf(p0.x, p1.x);
#pragma unroll
        for (int o = 8; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float S = 0.f;
        if (m > -CUDART_INF_F) {
            if (p0.x > -CUDART_INF_F) S += p0.y * ex2_approx((p0.x - m) * c);
            if (p1.x > -CUDART_INF_F) S += p1.y * ex2_approx((p1.x - m) * c);
        }
#pragma unroll
        for (int o = 8; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
        if (row_ok && hl == 0) {
            s_m[r] = m;
            s_inv[r] = __frcp_rn(S);
            // a row with no finite logit, or with NaN / +inf
            if (!(S > 0.f) || !(S < CUDART_INF_F) || !(m > -CUDART_INF_F) || !(m < CUDART_INF_F))
                if (g.rank == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        }
    }
    __syncthreads();

    // ---- acceptance tests (fp32: P and Q formed as for the residual, the
    // product u Q rounded once; they err by ~1e-7 relative, far inside the
    // band); every CTA makes the same loads on the same statistics and
    // reaches the same k
    if (threadIdx.x < 32) {
        bool rejected = false, close = false;
        if (lane < gamma) {
            const int rq = gamma + 1 + lane;
            const float P = ex2_approx((lpx - s_m[lane]) * a.c_target) * s_inv[lane];
            const float Q = ex2_approx((lqx - s_m[rq]) * a.c_draft) * s_inv[rq];
            const float uq = __fmul_rn(ua, Q);
            const float hi = fmaxf(P, uq);
            rejected = !(uq <= P);
            close = fabsf(uq - P) <= kLogitBandF * hi || hi < kLogitTinyF;
        }
        const unsigned rej = __ballot_sync(0xffffffffu, rejected);
        const unsigned cl = __ballot_sync(0xffffffffu, close);
        if (lane == 0) {
            const int k = rej ? __ffs(rej) - 1 : gamma;
            const unsigned ran = k >= 31 ? 0xffffffffu : (2u << k) - 1u;  // tests 0..k
            s_k = k;
            s_near = (cl & ran) ? 1 : 0;
        }
    }
    __syncthreads();

    // ---- the draw from the residual of row k (or the bonus row)
    const int k = s_k;
    SrcLogits src;
    src.p = logit_row(a, b, k);
    src.q = k < gamma ? logit_row(a, b, gamma + 1 + k) : nullptr;
    src.V = V;
    src.vec = vec;
    src.mp = s_m[k];
    src.cp = a.c_target;
    src.ip = s_inv[k];
    src.mq = k < gamma ? s_m[gamma + 1 + k] : 0.f;
    src.cq = a.c_draft;
    src.iq = k < gamma ? s_inv[gamma + 1 + k] : 0.f;
    bool near = s_near != 0;
    cluster_wait_started();
    Kept<NI, kKeepWeights<NI>> keep;
    double S = cluster_sum(st, src, g, 0, -1, nullptr, keep);
    if (src.q) {
        if (S < kLogitBand) near = true;
        if (!(S > 0.0)) {  // empty residual: draw from the target row (S is the same in every CTA)
            src.q = nullptr;
            S = cluster_sum(st, src, g, 1, -1, nullptr, keep);
        }
    }
    int tok;
    bool nd;
    if (cluster_draw(st, src, g, s_u, &tok, &nd, kLogitBand, keep) && threadIdx.x == 0) {
        if (tok < 0) {  // a row with no mass
            raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            tok = 0;
        }
        a.out_tokens[(size_t)b * (gamma + 1) + k] = tok;
        if (a.near) a.near[b] = (near || nd) ? 1 : 0;
    }
    if (g.rank == 0) {
        const int i = threadIdx.x;
        if (i <= gamma && i != k)
            a.out_tokens[(size_t)b * (gamma + 1) + i] = i < k ? a.tokens[(size_t)b * gamma + i] : -1;
        if (i == 0) a.accepted_len[b] = k;
    }
    // no peer touches this CTA's shared memory after the last exchange
}

// ---------------------------------------------------------------- tree, fed by logits
// The draft-tree recursion of spec_accept_tree_cluster_kernel on P[node] =
// softmax(Lp[node] / T) and Q[node] = softmax(Lq[qrow(node)] / T_draft)
// ("Speculative Decoding and KV-Cache Compression", section 2.3; "The
// Sub-Millisecond Speculative Decoding Meltdown", tree attention).  The walk
// visits one node per level, so the softmax statistics are formed for the
// visited rows only, by the cluster at each node: every CTA reduces its slice
// of the node's target row and draft row to (max, sum of 2^((l - max) c)),
// the pairs are exchanged through distributed shared memory and merged in
// rank order (fp32), so every CTA holds the same normalisers.  The tests are
// fp32 on probabilities formed as the residual's weights: the first child
// u Q(x) <= P(x), a later child u Q(x) Z <= R(x) with the fp32 residual R
// probed at x by the CTA that owns x.
//
// Near band after j rejected siblings: s_j = 2^(j+1) * 5e-5.  Each fp32
// probability errs by at most ~2.5e-5 relative; carried through the
// recursion R <- max(0, R - Z Q), Z = sum R, a residual entry errs by at most
// eps (P + a_j Q) and its mass by eps (1 + a_j) with a_1 = 1, a_{j+1} = 2 a_j + 2,
// so a test after j rejections is off by at most eps (P + a_{j+1} Q) <= s_j
// max(P, Q), and a draw's running sums by at most s_j.

// Residual update from logits: R <- max(0, prev - zf * Q) in fp32, prev = P
// (formed from its logits) on a node's first rejection, else R.
struct SrcUpdateLogits {
    float *R;
    const float *p;  // nullptr: prev = R
    const float *q;
    int lo, V;
    float zf;
    bool vec;
    float mp, cp, ip, mq, cq, iq;
    __device__ float4 operator()(int t0) const {
        float4 prev = make_float4(0.f, 0.f, 0.f, 0.f), qv = prev;
        if (t0 < V) {
            if (p) {
                const float4 l = load_logits4(p, t0, V, vec);
                prev = make_float4(ex2_approx((l.x - mp) * cp) * ip, ex2_approx((l.y - mp) * cp) * ip,
                                   ex2_approx((l.z - mp) * cp) * ip, ex2_approx((l.w - mp) * cp) * ip);
            } else {
                prev = *reinterpret_cast<const float4 *>(R + (t0 - lo));
            }
            const float4 l = load_logits4(q, t0, V, vec);
            qv = make_float4(ex2_approx((l.x - mq) * cq) * iq, ex2_approx((l.y - mq) * cq) * iq,
                             ex2_approx((l.z - mq) * cq) * iq, ex2_approx((l.w - mq) * cq) * iq);
        }
        const float4 r = make_float4(relu(prev.x - __fmul_rn(zf, qv.x)), relu(prev.y - __fmul_rn(zf, qv.y)),
                                     relu(prev.z - __fmul_rn(zf, qv.z)), relu(prev.w - __fmul_rn(zf, qv.w)));
        *reinterpret_cast<float4 *>(R + (t0 - lo)) = r;
        return r;
    }
};

// Softmax statistics of a node's two rows (0: target, 1: draft), as every CTA
// of the cluster holds them after cluster_row_stats.
struct TreeRowStats {
    float2 peer[2][2][kClMaxCtas];  // every CTA's (max, sum) by exchange parity and row, pushed by each CTA
    float2 w[2][kClWarps];
    float m[2];
    float inv[2];       // 1 / S (fp32)
    int bad;
};

// (max, sum) of this CTA's slice of `row` at scale c, merged over warp w's
// steps (groups of 16 logits), then over the warp's lanes; lane 0 stores the
// warp's pair in w[warp].
template <int NI>
__device__ __forceinline__ void warp_row_stats(const float *row, float c, const ClusterGeom &g, int V, bool vec,
                                               float2 *w) {
    const int lane = threadIdx.x & 31;
    float m = -CUDART_INF_F, s = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < NI; i0 += 4) {
        float4 x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            x[j] = i0 + j < NI ? load_logits4(row, g.wbase + (i0 + j) * kStep + 4 * lane, V, vec)
                               : make_float4(-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F);
        float m2, s2;
        group_stats16(x, c, m2, s2);
        online_merge(m, s, m2, s2, c);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        online_merge(m, s, m2, s2, c);
    }
    if (lane == 0) w[threadIdx.x >> 5] = make_float2(m, s);
}

// The softmax statistics of the target row p (scale cp) and, when q is not
// null, the draft row q (scale cq) over the whole cluster.  Every thread of
// every CTA calls this with the same parity; on return ts.m and ts.inv are
// the same in every CTA (the CTAs' pairs merged by the same fp32 butterfly),
// and ts.bad is set for a row with no finite logit, a NaN or +inf.
template <int NI>
__device__ void cluster_row_stats(TreeRowStats &ts, const float *p, const float *q, float cp, float cq,
                                  const ClusterGeom &g, int V, bool vec, int parity) {
    const int lane = threadIdx.x & 31;
    warp_row_stats<NI>(p, cp, g, V, vec, ts.w[0]);
    if (q) warp_row_stats<NI>(q, cq, g, V, vec, ts.w[1]);
    __syncthreads();
    if (threadIdx.x < 32) {
        // lane r < 2 merges the warps' pairs of row r, in warp order
        float m = -CUDART_INF_F, s = 0.f;
        if (lane < 2 && (lane == 0 || q)) {
            const float c = lane == 0 ? cp : cq;
            for (int w = 0; w < kClWarps; ++w) online_merge(m, s, ts.w[lane][w].x, ts.w[lane][w].y, c);
        }
        // push both rows' pairs into every CTA (lane t: peer t)
        const float m0 = __shfl_sync(0xffffffffu, m, 0), s0 = __shfl_sync(0xffffffffu, s, 0);
        const float m1 = __shfl_sync(0xffffffffu, m, 1), s1 = __shfl_sync(0xffffffffu, s, 1);
        if (lane < g.n_ctas) {
            st_peer_f32(&ts.peer[parity][0][g.rank].x, (uint32_t)lane, m0);
            st_peer_f32(&ts.peer[parity][0][g.rank].y, (uint32_t)lane, s0);
            st_peer_f32(&ts.peer[parity][1][g.rank].x, (uint32_t)lane, m1);
            st_peer_f32(&ts.peer[parity][1][g.rank].y, (uint32_t)lane, s1);
        }
    }
    cluster_sync_all();
    if (threadIdx.x < 32) {
        // half r of warp 0 merges row r: lane c of the half holds CTA c's pair
        const int r = lane >> 4, c16 = lane & 15;
        const bool have = c16 < g.n_ctas && (r == 0 || q);
        const float c = r == 0 ? cp : cq;
        const float2 v = have ? ts.peer[parity][r][c16] : make_float2(-CUDART_INF_F, 0.f);
        float m = v.x;
#pragma unroll
        for (int o = 8; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float S = (m > -CUDART_INF_F && v.x > -CUDART_INF_F) ? v.y * ex2_approx((v.x - m) * c) : 0.f;
#pragma unroll
        for (int o = 8; o; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
        if (c16 == 0 && (r == 0 || q)) {
            ts.m[r] = m;
            ts.inv[r] = __frcp_rn(S);
            if (!(S > 0.f) || !(S < CUDART_INF_F) || !(m > -CUDART_INF_F) || !(m < CUDART_INF_F)) ts.bad = 1;
        }
    }
    __syncthreads();
}

template <int NI>
__global__ void __launch_bounds__(kClThreads, kClCtasPerSm)
    spec_accept_tree_logits_cluster_kernel(const __grid_constant__ TreeArgs a, int n_ctas) {
    extern __shared__ float4 dyn_smem[];
    float *R = reinterpret_cast<float *>(dyn_smem);  // this CTA's residual slice
    __shared__ ClusterRow<NI> st;
    __shared__ TreeRowStats ts;
    const ClusterGeom g = cluster_geom<NI>(a.V, n_ctas);
    const int b = (int)(blockIdx.x / (unsigned)n_ctas);
    const int V = a.V, n_nodes = a.n_nodes;
    const int32_t *ntok = a.tokens + (size_t)b * n_nodes;
    const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(a.p) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
    const bool lead = g.rank == 0 && threadIdx.x == 0;
    cluster_arrive_on_entry();
    // node tokens and uniforms; per child of the node being visited P and Q
    // of its token (fp32, formed as for the residual)
    __shared__ int s_x[kMaxNq];
    __shared__ float s_ua[kMaxNq], s_px[kMaxNq], s_qx[kMaxNq];
    if (threadIdx.x < (unsigned)n_nodes) {
        int x = ntok[threadIdx.x];
        if (x < 0 || x >= V) {
            if (g.rank == 0 && threadIdx.x > 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            x = 0;
        }
        s_x[threadIdx.x] = x;
        s_ua[threadIdx.x] = __ldg(a.u_acc + (size_t)b * n_nodes + threadIdx.x);
    }
    if (threadIdx.x == 0) ts.bad = 0;
    const float u_s = __ldg(a.u_s + b);
    __syncthreads();
    cluster_wait_started();
    int node = 0, depth = 0, parity = 0;
    bool near = false, drew = false;
    int tok = -1;
    while (true) {
        const float *Pn = a.p + ((size_t)b * n_nodes + node) * V;
        const int qr = a.qrow[node];
        const float *Qn = qr >= 0 ? a.q + ((size_t)b * a.n_internal + qr) * V : nullptr;
        cluster_row_stats<NI>(ts, Pn, Qn, a.c_target, a.c_draft, g, V, vec, parity);
        parity ^= 1;
        SrcLogits srcp;
        srcp.p = Pn;
        srcp.q = nullptr;
        srcp.V = V;
        srcp.vec = vec;
        srcp.mp = ts.m[0];
        srcp.cp = a.c_target;
        srcp.ip = ts.inv[0];
        srcp.mq = 0.f;
        srcp.cq = a.c_draft;
        srcp.iq = 0.f;
        if (qr < 0) {  // leaf: bonus token from its own P
            Kept<NI, kKeepWeights<NI>> keep;
            cluster_sum(st, srcp, g, parity, -1, nullptr, keep);
            parity ^= 1;
            bool nb = false;
            drew = cluster_draw(st, srcp, g, u_s, &tok, &nb, kLogitBand, keep);
            near |= nb;
            break;
        }
        {
            const int c = node + 1 + (int)threadIdx.x;
            if (c < n_nodes && a.parent[c] == node) {
                s_px[c] = ex2_approx((__ldg(Pn + s_x[c]) - ts.m[0]) * a.c_target) * ts.inv[0];
                s_qx[c] = ex2_approx((__ldg(Qn + s_x[c]) - ts.m[1]) * a.c_draft) * ts.inv[1];
            }
            __syncthreads();
        }
        // the tests in fp32 (they err by ~1e-7 relative, far inside the band):
        // the first child u Q <= P, a later one u Q Z <= R(x)
        double Z = 1.0;
        float zf = 1.f;
        float rx = 0.f;  // R(x) of the child under test, after a rejection
        int accepted = -1, j = 0;
        for (int c = node + 1; c < n_nodes; ++c) {
            if (a.parent[c] != node) continue;
            const float P = s_px[c], Qx = s_qx[c];
            const float band = kLogitBandF * (float)(2u << min(j, 29));
            const float lhs = __fmul_rn(__fmul_rn(s_ua[c], Qx), zf);
            const float Rx = j == 0 ? P : rx;  // the residual at x: P before any rejection
            const float hi = fmaxf(P, Qx);
            const bool ok = lhs <= Rx;
            const bool close = fabsf(lhs - Rx) <= band * hi || hi < kLogitTinyF;
            near |= close;
            if (ok) {
                accepted = c;
                break;
            }
            int xn = -1;  // the next sibling's token: R is probed there
            for (int c2 = c + 1; c2 < n_nodes; ++c2)
                if (a.parent[c2] == node) {
                    xn = s_x[c2];
                    break;
                }
            SrcUpdateLogits upd;
            upd.R = R;
            upd.p = j == 0 ? Pn : nullptr;
            upd.q = Qn;
            upd.lo = g.cta_lo;
            upd.V = V;
            upd.zf = (float)Z;
            upd.vec = vec;
            upd.mp = ts.m[0];
            upd.cp = a.c_target;
            upd.ip = ts.inv[0];
            upd.mq = ts.m[1];
            upd.cq = a.c_draft;
            upd.iq = ts.inv[1];
            Z = cluster_sum(st, upd, g, parity, xn, R);
            zf = (float)Z;
            parity ^= 1;
            rx = st.probe_val;
            ++j;
        }
        if (accepted >= 0) {
            ++depth;
            if (lead) {
                a.path_nodes[(size_t)b * a.width + depth] = accepted;
                a.out_tokens[(size_t)b * a.width + depth - 1] = s_x[accepted];
            }
            node = accepted;
            continue;
        }
        const double s = kLogitBand * (double)(2u << min(j, 29));
        if (Z < s) near = true;
        bool nb = false;
        if (Z > 0.0) {
            drew = cluster_draw(st, SrcSmem{R, g.cta_lo}, g, u_s, &tok, &nb, s);
        } else {  // empty residual: draw from the node's target row
            Kept<NI, kKeepWeights<NI>> keep;
            cluster_sum(st, srcp, g, parity, -1, nullptr, keep);
            parity ^= 1;
            drew = cluster_draw(st, srcp, g, u_s, &tok, &nb, kLogitBand, keep);
        }
        near |= nb;
        break;
    }
    if (drew && threadIdx.x == 0) {
        if (tok < 0) {  // a row with no mass
            raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
            tok = 0;
        }
        a.out_tokens[(size_t)b * a.width + depth] = tok;
        if (a.near) a.near[b] = near ? 1 : 0;
    }
    if (lead) {
        if (ts.bad) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        int32_t *path = a.path_nodes + (size_t)b * a.width;
        int32_t *out = a.out_tokens + (size_t)b * a.width;
        path[0] = 0;
        for (int d = depth + 1; d < a.width; ++d) {
            path[d] = -1;
            out[d] = -1;
        }
        a.accepted_len[b] = depth;
    }
    // no peer touches this CTA's shared memory after the last exchange
}

int sm_count_cached() {
    static DeviceMemo<int> memo;
    int n = 0;
    const cudaError_t e = memo.get(&n, [](int *v) {
        int dev = 0;
        cudaError_t r = cudaGetDevice(&dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
        return r == cudaSuccess && *v <= 0 ? cudaErrorInvalidValue : r;
    });
    return e == cudaSuccess ? n : 152;
}

// Steps per warp (a power of two) for B rows of V tokens, or 0 when V is
// beyond the cluster kernels: the fewest steps that cover a row with 8 CTAs,
// then more steps (fewer CTAs per row) while the grid would not be resident
// in one wave.  Depends on (B, V) only, so both samplers split a row alike.
int cluster_steps(int B, int V) {
    constexpr int per_step_row = kClWarps * kStep * kClMaxCtas;
    const int need = (V + per_step_row - 1) / per_step_row;
    int ni = 1;
    while (ni < need) ni <<= 1;
    if (ni > kClMaxSteps) return 0;
    const long long slots = (long long)sm_count_cached() * kClCtasPerSm;
    auto ctas = [&](int n) { return (V + kClWarps * n * kStep - 1) / (kClWarps * n * kStep); };
    while (ni < kClMaxSteps && ctas(ni) > 1 && (long long)B * ctas(ni) > slots) ni <<= 1;
    return ni;
}

template <class Args>
cudaError_t launch_cluster(void (*const *kernels)(Args, int), const Args &a, int V, int B, size_t dyn_smem_per_step,
                           cudaStream_t stream, bool programmatic = false) {
    const int ni = cluster_steps(B, V);
    const int chunk = kClWarps * ni * kStep;
    const int n = (V + chunk - 1) / chunk;
    int idx = 0;
    while ((1 << idx) < ni) ++idx;
    void (*kern)(Args, int) = kernels[idx];
    const size_t smem = dyn_smem_per_step * (size_t)ni;
    if (smem > 0) {
        // the shared-memory opt-in of each step count, once per device
        static DeviceMemo<size_t> opted[8];
        size_t have = 0;
        auto opt_in = [&](size_t *v) {
            *v = smem;
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        };
        cudaError_t e = opted[idx & 7].get(&have, opt_in);
        if (e == cudaSuccess && have < smem) e = opt_in(&have);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * n));
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)n;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // a programmatic dependent of the previous kernel on the stream: it may
    // start early and waits (griddepcontrol.wait) before reading its results
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a, n);
}

}  // namespace

cudaError_t launch_spec_accept(const AcceptArgs &a, cudaStream_t stream) {
    if (a.B <= 0) return cudaSuccess;
    if (cluster_steps(a.B, a.V) == 0 || (long long)a.B * kClMaxCtas > 0x7fffffffLL) {
        spec_accept_kernel<<<a.B, kRowThreads, 0, stream>>>(a);
        return cudaGetLastError();
    }
    static void (*const kernels[])(AcceptArgs, int) = {
        spec_accept_cluster_kernel<1>, spec_accept_cluster_kernel<2>,  spec_accept_cluster_kernel<4>,
        spec_accept_cluster_kernel<8>, spec_accept_cluster_kernel<16>, spec_accept_cluster_kernel<32>};
    return launch_cluster(kernels, a, a.V, a.B, 0, stream);
}

int spec_accept_tree_max_vocab() { return kClMaxVocab; }

size_t spec_accept_logits_stats_bytes(int B, int gamma, int V) {
    return (size_t)B * (size_t)(2 * gamma + 1) * (size_t)((V + kSlab - 1) / kSlab) * sizeof(float2);
}

cudaError_t launch_spec_accept_logits(const LogitsArgs &a, cudaStream_t stream) {
    if (a.B <= 0) return cudaSuccess;
    if (a.gamma < 1 || 2 * a.gamma + 1 > kMaxLogitRows || cluster_steps(a.B, a.V) == 0 ||
        (long long)a.B * kClMaxCtas > 0x7fffffffLL || !a.stats)
        return cudaErrorInvalidValue;
    LogitsArgs b = a;
    b.n_slabs = (a.V + kSlab - 1) / kSlab;
    const long long stat_ctas = (long long)a.B * (2 * a.gamma + 1) * b.n_slabs;
    if (b.n_slabs > kMaxSlabs || stat_ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    logit_stats_kernel<<<(unsigned)stat_ctas, kStatThreads, 0, stream>>>(b);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    static void (*const kernels[])(LogitsArgs, int) = {
        spec_accept_logits_cluster_kernel<1>, spec_accept_logits_cluster_kernel<2>,
        spec_accept_logits_cluster_kernel<4>, spec_accept_logits_cluster_kernel<8>,
        spec_accept_logits_cluster_kernel<16>, spec_accept_logits_cluster_kernel<32>};
    return launch_cluster(kernels, b, a.V, a.B, 0, stream, /*programmatic=*/true);
}

cudaError_t launch_spec_accept_tree(const TreeArgs &a, cudaStream_t stream) {
    if (a.B <= 0) return cudaSuccess;
    if (cluster_steps(a.B, a.V) == 0) return cudaErrorInvalidValue;
    static void (*const kernels[])(TreeArgs, int) = {
        spec_accept_tree_cluster_kernel<1>, spec_accept_tree_cluster_kernel<2>,
        spec_accept_tree_cluster_kernel<4>, spec_accept_tree_cluster_kernel<8>,
        spec_accept_tree_cluster_kernel<16>, spec_accept_tree_cluster_kernel<32>};
    return launch_cluster(kernels, a, a.V, a.B, (size_t)kClWarps * kStep * sizeof(float), stream);
}


cudaError_t launch_spec_accept_tree_logits(const TreeArgs &a, cudaStream_t stream) {
    if (a.B <= 0) return cudaSuccess;
    if (cluster_steps(a.B, a.V) == 0) return cudaErrorInvalidValue;
    static void (*const kernels[])(TreeArgs, int) = {
        spec_accept_tree_logits_cluster_kernel<1>,  spec_accept_tree_logits_cluster_kernel<2>,
        spec_accept_tree_logits_cluster_kernel<4>,  spec_accept_tree_logits_cluster_kernel<8>,
        spec_accept_tree_logits_cluster_kernel<16>, spec_accept_tree_logits_cluster_kernel<32>};
    return launch_cluster(kernels, a, a.V, a.B, (size_t)kClWarps * kStep * sizeof(float), stream);
}

}  // namespace svpa
