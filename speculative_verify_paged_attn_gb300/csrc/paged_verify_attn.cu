// paged_verify_attn.cu -- paged verification attention for sm_103a.
//
// What it computes ("The Sub-Millisecond Speculative Decoding Meltdown",
// section "Speculative Decoding Mechanics & The K-Token Penalty"): for every
// sequence, the n_q verification queries (last committed token + drafts, or
// the nodes of a draft tree) attend over the sequence's K/V history with a
// causal or ancestor (tree) mask, A = softmax(Q K^T * scale + M) V.  The
// history is read page by page through the block table ("Triton CUDA Fused
// Speculative Tree-Verification Kernel" on the same page: per-page physical
// block lookup, K/V cache [blocks, heads, 16, dim], per-(block, head) FP8
// scales, running max/sum softmax).
//
// GB300 design (differs from the page's per-query Triton program):
//  * work unit = (sequence, kv head, KV split): all G*n_q query rows of a kv
//    head share each K/V page, so every page is read from HBM exactly once;
//  * persistent CTAs, several per SM; a producer warp takes units from an
//    atomic counter (unsplit units longest sequence first, ranked by
//    seq_order_kernel below) and streams their (K, V) page tiles -- and, at each
//    unit's first page, the unit's query tile -- into a ring of shared-memory
//    stages with tiled bulk tensor copies (TMA, 128-byte swizzle, one
//    mbarrier pair per stage), gathering pages by block id.  The ring runs
//    across unit boundaries, so a CTA never drains between units;
//  * consumer warps (one per 16 query rows): m16n8k16 tensor-core MMAs (bf16,
//    or f16 on exactly decoded FP8 bytes) for S = Q K^T and O += P V, online
//    softmax in fp32 registers with exp2 and quad shuffles, the rescale of O
//    skipped while no row maximum moves;
//  * long contexts are cut into splits; each split writes (max, sum, acc)
//    partials and the last CTA of a (sequence, kv head) to finish -- an
//    atomic ticket, never a spin -- merges them with a log-sum-exp combine.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kBarConsumers = 1;  // named barrier id used by the consumer warps

template <int D, bool FP8>
struct Geo {
    static constexpr int EB = FP8 ? 1 : 2;
    static constexpr int ROW = D * EB;             // bytes of one token row of one kv head
    static constexpr int SLABS = ROW / 128;         // 128-byte swizzle slabs per row
    static constexpr int TILE = 16 * ROW;           // one page of K (or V) for one kv head
    static constexpr int STAGE = 2 * TILE;          // K tile then V tile
    static constexpr int ACC = D / 2;               // fp32 accumulators per thread (16 rows x D / 32)
    static constexpr int QSLABS = D * 2 / 128;      // queries are bf16
};

template <int MT>
struct Occ {  // resident CTAs per SM the register budget is sized for
    static constexpr int MINB = MT == 1 ? 6 : (MT <= 3 ? 3 : (MT == 4 ? 2 : 1));
};

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagEnd = 4;

struct StageMeta {
    int32_t b, h, split, i, n, L, nsplit, flags, qb;
    float ks, vs;
    int32_t pad;
};

// Byte offset of 16-byte chunk `ch` of row `t` inside a swizzled tile whose
// 128-byte slabs are `slab` bytes apart; chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t swz(int t, int ch, int slab) {
    return (uint32_t)((ch >> 3) * slab + (t << 7) + (((ch & 7) ^ (t & 7)) << 4));
}

// Column (head-dim index) held by accumulator register i of lane quad index c.
template <bool FP8>
__device__ __forceinline__ int acc_col(int i, int c) {
    const int e = i & 3;
    if constexpr (!FP8) {
        return (i >> 2) * 8 + 2 * c + (e & 1);
    } else {
        const int par = (i >> 2) & 1, ch = i >> 3;
        return ch * 16 + 4 * c + 2 * (e & 1) + par;
    }
}

// Merge the split partials of (b, h) into the final output; run by the
// consumer warps of the CTA that finished the last split.
template <int D, int NCW>
__device__ void combine_splits(const AttnArgs &a, int b, int h, int nsplit, int warp, int lane) {
    constexpr int PER = D / 32;  // head-dim columns per lane
    const int unit = b * a.Hkv + h;
    const int G = a.G;
    for (int R = warp; R < a.M; R += NCW) {
        const size_t base = (size_t)unit * a.max_splits * a.M + R;
        float mx = -CUDART_INF_F;
        for (int s2 = 0; s2 < nsplit; ++s2) mx = fmaxf(mx, __ldcg(&a.part_ml[(base + (size_t)s2 * a.M) * 2]));
        const float msafe = mx == -CUDART_INF_F ? 0.f : mx;
        float o[PER];
#pragma unroll
        for (int x = 0; x < PER; ++x) o[x] = 0.f;
        float l = 0.f;
        for (int s2 = 0; s2 < nsplit; ++s2) {
            const size_t pr = base + (size_t)s2 * a.M;
            const float w = exp2f(__ldcg(&a.part_ml[pr * 2]) - msafe);
            l += w * __ldcg(&a.part_ml[pr * 2 + 1]);
            const float *prow = a.part_acc + pr * D + lane * PER;
            if constexpr (PER == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(prow));
                o[0] += w * v.x; o[1] += w * v.y; o[2] += w * v.z; o[3] += w * v.w;
            } else {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(prow));
                o[0] += w * v.x; o[1] += w * v.y;
            }
        }
        const int j = R / G, gi = R - j * G;
        const size_t od = (((size_t)b * a.n_q + j) * a.Hq + (size_t)h * G + gi);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16 *orow = a.out + od * D + lane * PER;
        if constexpr (PER == 4) {
            uint2 pk;
            pk.x = pack_bf16x2(o[0] * inv, o[1] * inv);
            pk.y = pack_bf16x2(o[2] * inv, o[3] * inv);
            *reinterpret_cast<uint2 *>(orow) = pk;
        } else {
            *reinterpret_cast<uint32_t *>(orow) = pack_bf16x2(o[0] * inv, o[1] * inv);
        }
        if (a.lse && lane == 0) a.lse[od] = (mx + log2f(l)) * 0.69314718055994530942f;
    }
}

template <int D, bool FP8, int MT>
__global__ void __launch_bounds__((MT + 1) * 32, Occ<MT>::MINB)
    pva_kernel(const __grid_constant__ CUtensorMap mk0, const __grid_constant__ CUtensorMap mk1,
               const __grid_constant__ CUtensorMap mv0, const __grid_constant__ CUtensorMap mv1,
               const __grid_constant__ CUtensorMap mq0, const __grid_constant__ CUtensorMap mq1,
               const __grid_constant__ AttnArgs a) {
    using G_ = Geo<D, FP8>;
    constexpr int NCW = MT;
    constexpr int NCT = NCW * 32;
    constexpr int ACC = G_::ACC;
    constexpr int QSLAB = MT * 16 * 128;           // bytes of one 128-byte column slab of Q
    constexpr int QBUF = QSLAB * G_::QSLABS;
    const int NS = a.n_stages;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qbuf = smem;                                 // 2 query buffers
    uint8_t *stages = qbuf + 2 * QBUF;
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + (size_t)NS * G_::STAGE);
    uint64_t *empty = full + NS;
    uint64_t *qempty = empty + NS;                        // [2]
    StageMeta *meta = reinterpret_cast<StageMeta *>(qempty + 2);
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        mbar_init(&qempty[0], NCW);
        mbar_init(&qempty[1], NCW);
        fence_mbar_init();
    }
    // query rows past M are never written by the copies: keep them finite
    for (int x = threadIdx.x; x < 2 * QBUF / 16; x += blockDim.x)
        reinterpret_cast<uint4 *>(qbuf)[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    __syncthreads();

    if (warp == NCW) {
        // ================================================= producer warp
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&mk0);
            prefetch_tensormap(&mv0);
            prefetch_tensormap(&mq0);
            if constexpr (G_::QSLABS > 1) prefetch_tensormap(&mq1);
        }
        int slot = 0, issued = 0, units = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint32_t qbytes = (uint32_t)(a.M * 128 * G_::QSLABS);
        while (ok) {
            int u = 0;
            if (lane == 0) u = atomicAdd(&a.sched[0], 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u >= a.total_units) break;
            const int bh = u / a.max_splits, split = u - bh * a.max_splits;
            const int rb = bh / a.Hkv, h = bh - rb * a.Hkv;
            const int b = a.order ? __ldg(a.order + rb) : rb;  // longest sequences first
            const int L = __ldg(a.context_lens + b);
            const int npages = (L + a.n_q + kBlockSize - 1) / kBlockSize;
            if (L < 0 || npages > a.max_blocks) {
                if (lane == 0 && split == 0 && h == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                continue;
            }
            const int nsplit = (npages + a.split_pages - 1) / a.split_pages;
            if (split >= nsplit) continue;
            const int page0 = split * a.split_pages;
            const int n = min(a.split_pages, npages - page0);
            const int qb = units & 1;
            const int32_t *bt = a.block_table + (size_t)b * a.max_blocks + page0;
            for (int i0 = 0; i0 < n && ok; i0 += 32) {
                int blk = 0;
                float ks = 1.f, vs = 1.f;
                if (i0 + lane < n) {
                    blk = __ldg(bt + i0 + lane);
                    if (blk < 0 || blk >= a.num_blocks) {
                        raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
                        blk = 0;
                    }
                    if constexpr (FP8) {
                        ks = __ldg(a.k_scale + (size_t)blk * a.Hkv + h);
                        vs = __ldg(a.v_scale + (size_t)blk * a.Hkv + h);
                    }
                }
                const int cnt = min(32, n - i0);
                for (int j = 0; j < cnt; ++j) {
                    const int bj = __shfl_sync(0xffffffffu, blk, j);
                    const float ksj = __shfl_sync(0xffffffffu, ks, j);
                    const float vsj = __shfl_sync(0xffffffffu, vs, j);
                    if (lane == 0) {
                        const int i = i0 + j;
                        if (issued >= NS) ok = mbar_wait(&empty[slot], phase ^ 1u, a.err);
                        if (ok && i == 0 && units >= 2)
                            ok = mbar_wait(&qempty[qb], (uint32_t)(((units >> 1) & 1) ^ 1), a.err);
                        if (ok) {
                            StageMeta &m = meta[slot];
                            m.b = b; m.h = h; m.split = split; m.i = i; m.n = n; m.L = L;
                            m.nsplit = nsplit; m.qb = qb; m.ks = ksj; m.vs = vsj;
                            m.flags = (i == 0 ? kFlagFirst : 0) | (i == n - 1 ? kFlagLast : 0);
                            uint8_t *st = stages + (size_t)slot * G_::STAGE;
                            mbar_arrive_expect_tx(&full[slot], G_::STAGE + (i == 0 ? qbytes : 0u));
                            if (i == 0) {
                                uint8_t *qd = qbuf + qb * QBUF;
                                tma_load_4d(qd, &mq0, 0, h * a.G, 0, b, &full[slot], pol);
                                if constexpr (G_::QSLABS > 1)
                                    tma_load_4d(qd + QSLAB, &mq1, 0, h * a.G, 0, b, &full[slot], pol);
                            }
                            if constexpr (G_::SLABS > 1) {
                                // both slabs of the page in one copy (5-D box)
                                tma_load_5d(st, &mk0, 0, 0, 0, h, bj, &full[slot], pol);
                                tma_load_5d(st + G_::TILE, &mv0, 0, 0, 0, h, bj, &full[slot], pol);
                            } else {
                                tma_load_4d(st, &mk0, 0, 0, h, bj, &full[slot], pol);
                                tma_load_4d(st + G_::TILE, &mv0, 0, 0, h, bj, &full[slot], pol);
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
                    if (!ok) break;
                    ++issued;
                    if (++slot == NS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            ++units;
        }
        if (lane == 0) {
            // end-of-work marker for the consumers
            if (ok && issued >= NS) ok = mbar_wait(&empty[slot], phase ^ 1u, a.err);
            if (ok) {
                meta[slot].flags = kFlagEnd;
                mbar_arrive(&full[slot]);
            }
            // no copy may still be in flight when the CTA exits: wait (bounded)
            // for the last stages to land.  The stage the end marker reused
            // (page issued - NS) was already known complete when its empty
            // barrier was passed, and its full barrier has moved on since.
            const int first = issued >= NS ? issued - NS + 1 : 0;
            for (int i = first; i < issued && ok; ++i)
                ok = mbar_wait(&full[i % NS], (uint32_t)((i / NS) & 1), a.err);
            // the last CTA to finish resets the scheduler for the next call
            __threadfence();
            const int done = atomicAdd(&a.sched[1], 1);
            if (done == (int)gridDim.x - 1) {
                a.sched[0] = 0;
                a.sched[1] = 0;
            }
        }
        return;
    }

    // ===================================================== consumer warps
    const int mt = warp;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const int G = a.G;
    unsigned long long mrow[2];
    mrow[0] = r0 < a.M ? a.anc[r0 / G] : 0ull;
    mrow[1] = r1 < a.M ? a.anc[r1 / G] : 0ull;

    float acc[ACC / 4][4];
    float m_run[2], l_run[2];
    float s_ref = 0.f;            // FP8: running max of the V scales seen in this unit
    uint32_t qa[FP8 ? D / 16 : 1][4];  // FP8: f16 query fragments held in registers

    int slot = 0;
    uint32_t phase = 0;
    while (true) {
        if (!mbar_wait(&full[slot], phase, a.err)) break;
        const StageMeta md = meta[slot];
        if (md.flags & kFlagEnd) break;
        const uint8_t *qd = qbuf + md.qb * QBUF;
        if (md.flags & kFlagFirst) {
#pragma unroll
            for (int i = 0; i < ACC / 4; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
            m_run[0] = m_run[1] = -CUDART_INF_F;
            l_run[0] = l_run[1] = 0.f;
            s_ref = 0.f;
            if constexpr (FP8) {
                // f16 fragments, head-dim order permuted to match the byte
                // order ldmatrix delivers from FP8 rows: thread (g, c) holds
                // columns 4c..4c+3 of each 16-column step
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int r = x ? r1 : r0;
                        const int ch = 2 * kk + (c >> 1);
                        const uint2 v = *reinterpret_cast<const uint2 *>(
                            qd + swz(r, ch, QSLAB) + (c & 1) * 8);
                        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
                        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
                        qa[kk][x] = pack_f16x2(f0.x, f0.y);
                        qa[kk][2 + x] = pack_f16x2(f1.x, f1.y);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&qempty[md.qb]);
            }
        }
        uint8_t *kt = stages + (size_t)slot * G_::STAGE;
        uint8_t *vt = kt + G_::TILE;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
        const int L = md.L, T = L + a.n_q;
        const int pos0 = (md.split * a.split_pages + md.i) * kBlockSize;

        // slots past the last token may hold anything: zero their V rows so
        // that 0 * garbage cannot reach the accumulators
        const bool tail = pos0 + kBlockSize > T;
        if (tail) {
            const int tv = T - pos0;
            const int nz = (kBlockSize - tv) * G_::SLABS * 8;
            for (int z = lane; z < nz; z += 32) {
                const int row = tv + z / (G_::SLABS * 8);
                const int rem = z % (G_::SLABS * 8);
                *reinterpret_cast<uint4 *>(vt + ((rem >> 3) << 11) + (row << 7) + ((rem & 7) << 4)) =
                    make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        // ---- S = Q K^T (16 rows x 16 tokens)
        float s[2][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[x][e] = 0.f;
        if constexpr (!FP8) {
            const uint32_t qbase = smem_u32(qd);
            const int qrow = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int qpar = lane >> 4;
            const int tok = ((lane >> 4) << 3) + (lane & 7);
            const int par = (lane >> 3) & 1;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t q4[4];
                ldmatrix_x4(qbase + swz(qrow, 2 * kk + qpar, QSLAB), q4[0], q4[1], q4[2], q4[3]);
                uint32_t b00, b01, b10, b11;
                ldmatrix_x4(kbase + swz(tok, 2 * kk + par, 2048), b00, b01, b10, b11);
                mma_bf16_16816(s[0], q4, b00, b01);
                mma_bf16_16816(s[1], q4, b10, b11);
            }
        } else {
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                uint32_t r0k, r1k, r2k, r3k;
                ldmatrix_x4(kbase + swz(tok, 2 * kp + par, 2048), r0k, r1k, r2k, r3k);
                mma_f16_16816(s[0], qa[2 * kp], e4m3x2_to_f16x2(r0k & 0xffff), e4m3x2_to_f16x2(r0k >> 16));
                mma_f16_16816(s[1], qa[2 * kp], e4m3x2_to_f16x2(r1k & 0xffff), e4m3x2_to_f16x2(r1k >> 16));
                mma_f16_16816(s[0], qa[2 * kp + 1], e4m3x2_to_f16x2(r2k & 0xffff), e4m3x2_to_f16x2(r2k >> 16));
                mma_f16_16816(s[1], qa[2 * kp + 1], e4m3x2_to_f16x2(r3k & 0xffff), e4m3x2_to_f16x2(r3k >> 16));
            }
        }
        float sc = a.scale_log2;
        if constexpr (FP8) sc *= md.ks;
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[x][e] *= sc;
        if (pos0 + kBlockSize > L) {
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int p = pos0 + x * 8 + 2 * c + (e & 1);
                    const int sidx = p - L;
                    const unsigned long long mk = mrow[e >> 1];
                    const bool vis = sidx < 0 || (sidx < a.n_q && ((mk >> sidx) & 1ull));
                    if (!vis) s[x][e] = -CUDART_INF_F;
                }
        }

        // ---- online softmax (rows g and g+8 of this m-tile)
        float alpha[2];
        float pv_scale = 1.f;
        if constexpr (FP8) {
            // fold the page's V scale into P relative to the running maximum
            // scale of the unit (so P * ratio <= P never overflows f16)
            const float vs = md.vs;
            if (vs > s_ref) {
                const float ratio = s_ref / vs;
                s_ref = vs;
                alpha[0] = alpha[1] = ratio;  // folded into the rescale below
            } else {
                alpha[0] = alpha[1] = 1.f;
            }
            pv_scale = s_ref > 0.f ? vs / s_ref : 0.f;
        } else {
            alpha[0] = alpha[1] = 1.f;
        }
        uint32_t pa[4];
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
            float mx = fmaxf(fmaxf(s[0][2 * rh], s[0][2 * rh + 1]), fmaxf(s[1][2 * rh], s[1][2 * rh + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(m_run[rh], mx);
            const float msafe = mnew == -CUDART_INF_F ? 0.f : mnew;
            const float al = exp2f(m_run[rh] - msafe);
            m_run[rh] = mnew;
            const float p00 = exp2f(s[0][2 * rh] - msafe), p01 = exp2f(s[0][2 * rh + 1] - msafe);
            const float p10 = exp2f(s[1][2 * rh] - msafe), p11 = exp2f(s[1][2 * rh + 1] - msafe);
            l_run[rh] = l_run[rh] * al + (p00 + p01) + (p10 + p11);
            alpha[rh] *= al;
            if constexpr (!FP8) {
                pa[rh] = pack_bf16x2(p00, p01);
                pa[2 + rh] = pack_bf16x2(p10, p11);
            } else {
                pa[rh] = pack_f16x2(p00 * pv_scale, p01 * pv_scale);
                pa[2 + rh] = pack_f16x2(p10 * pv_scale, p11 * pv_scale);
            }
        }
        // rescale O only when some row's maximum (or the FP8 scale) moved
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int x = 0; x < ACC / 4; ++x)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[x][e] *= alpha[e >> 1];
        }

        // ---- O += P V
        if constexpr (!FP8) {
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(vbase + swz(tok, 2 * np + par, 2048), v0, v1, v2, v3);
                mma_bf16_16816(acc[2 * np], pa, v0, v1);
                mma_bf16_16816(acc[2 * np + 1], pa, v2, v3);
            }
        } else {
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int cp = 0; cp < D / 32; ++cp) {
                uint32_t r0v, r1v, r2v, r3v;
                ldmatrix_x4_trans(vbase + swz(tok, 2 * cp + par, 2048), r0v, r1v, r2v, r3v);
                // chunk 2cp from (r0v, r1v), chunk 2cp+1 from (r2v, r3v);
                // even / odd head-dim columns of each chunk are separate n-tiles
                const uint32_t ev0 = __byte_perm(r0v, r1v, 0x6420), od0 = __byte_perm(r0v, r1v, 0x7531);
                const uint32_t ev1 = __byte_perm(r2v, r3v, 0x6420), od1 = __byte_perm(r2v, r3v, 0x7531);
                mma_f16_16816(acc[4 * cp + 0], pa, e4m3x2_to_f16x2(ev0 & 0xffff), e4m3x2_to_f16x2(ev0 >> 16));
                mma_f16_16816(acc[4 * cp + 1], pa, e4m3x2_to_f16x2(od0 & 0xffff), e4m3x2_to_f16x2(od0 >> 16));
                mma_f16_16816(acc[4 * cp + 2], pa, e4m3x2_to_f16x2(ev1 & 0xffff), e4m3x2_to_f16x2(ev1 >> 16));
                mma_f16_16816(acc[4 * cp + 3], pa, e4m3x2_to_f16x2(od1 & 0xffff), e4m3x2_to_f16x2(od1 >> 16));
            }
        }

        __syncwarp();
        if (tail) fence_proxy_async_smem();
        if (lane == 0) {
            mbar_arrive(&empty[slot]);
            if (!FP8 && (md.flags & kFlagLast)) mbar_arrive(&qempty[md.qb]);
        }
        if (++slot == NS) {
            slot = 0;
            phase ^= 1u;
        }
        if (!(md.flags & kFlagLast)) continue;

        // ---- the unit is complete: output, or split partial + combine
        float lr[2];
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
            lr[rh] = l_run[rh];
            lr[rh] += __shfl_xor_sync(0xffffffffu, lr[rh], 1);
            lr[rh] += __shfl_xor_sync(0xffffffffu, lr[rh], 2);
        }
        const float oscale = FP8 ? s_ref : 1.f;
        const int b = md.b, h = md.h;
        const int rows[2] = {r0, r1};
        if (md.nsplit == 1) {
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int R = rows[rh];
                if (R >= a.M) continue;
                const int j = R / G, gi = R - j * G;
                const size_t o = (((size_t)b * a.n_q + j) * a.Hq + (size_t)h * G + gi);
                const float inv = lr[rh] > 0.f ? oscale / lr[rh] : 0.f;
                __nv_bfloat16 *orow = a.out + o * D;
                if constexpr (!FP8) {
#pragma unroll
                    for (int x = 0; x < ACC / 4; ++x)
                        *reinterpret_cast<uint32_t *>(orow + x * 8 + 2 * c) =
                            pack_bf16x2(acc[x][2 * rh] * inv, acc[x][2 * rh + 1] * inv);
                } else {
#pragma unroll
                    for (int ch = 0; ch < D / 16; ++ch) {
                        uint2 pk;
                        pk.x = pack_bf16x2(acc[2 * ch][2 * rh] * inv, acc[2 * ch + 1][2 * rh] * inv);
                        pk.y = pack_bf16x2(acc[2 * ch][2 * rh + 1] * inv, acc[2 * ch + 1][2 * rh + 1] * inv);
                        *reinterpret_cast<uint2 *>(orow + ch * 16 + 4 * c) = pk;
                    }
                }
                if (a.lse && c == 0) a.lse[o] = (m_run[rh] + log2f(lr[rh])) * 0.69314718055994530942f;
            }
            continue;
        }
        const int unit = b * a.Hkv + h;
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
            const int R = rows[rh];
            if (R >= a.M) continue;
            const size_t pr = ((size_t)unit * a.max_splits + md.split) * a.M + R;
            float *prow = a.part_acc + pr * D;
#pragma unroll
            for (int x = 0; x < ACC; ++x)
                if (((x & 2) >> 1) == rh) prow[acc_col<FP8>(x, c)] = acc[x >> 2][x & 3] * oscale;
            if (c == 0) {
                a.part_ml[pr * 2] = m_run[rh];
                a.part_ml[pr * 2 + 1] = lr[rh];
            }
        }
        __threadfence();
        named_barrier_sync(kBarConsumers, NCT);
        if (threadIdx.x == 0) {
            const int t = atomicAdd(&a.tickets[unit], 1);
            s_last = (t == md.nsplit - 1);
            if (s_last) a.tickets[unit] = 0;  // self-cleaning for the next call
        }
        named_barrier_sync(kBarConsumers, NCT);
        const int last = s_last;
        named_barrier_sync(kBarConsumers, NCT);  // s_last may be rewritten by the next unit
        if (!last) continue;
        __threadfence();
        combine_splits<D, NCW>(a, b, h, md.nsplit, warp, lane);
    }
}

template <int D, bool FP8, int MT>
cudaError_t plan_mt_uncached(AttnLaunch *out) {
    using G_ = Geo<D, FP8>;
    constexpr int THREADS = (MT + 1) * 32;
    auto kern = pva_kernel<D, FP8, MT>;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // registers are allocated per warp in units of 256
    const int per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
    int ctas = 65536 / (per_warp * (THREADS / 32));
    // up to 6 CTAs per SM (measured on the 7B shape: 4 -> 226 us, 5 -> 223, 6 -> 218; 7 and 8,
    // at 128 registers and fewer stages each, 223 and 221)
    ctas = ctas < 1 ? 1 : (ctas > 6 ? 6 : ctas);
    const int qbuf = 2 * MT * 16 * 128 * G_::QSLABS;
    const int fixed = 1024 + qbuf + 16 + 64;
    const int per_cta = 233472 / ctas - 1024 - (int)fa.sharedSizeBytes;
    int ns = (per_cta - fixed) / (G_::STAGE + 16 + (int)sizeof(StageMeta));
    ns = ns > 24 ? 24 : ns;
    if (ns < 2) ns = 2;
    out->n_stages = ns;
    out->smem = (size_t)fixed + (size_t)ns * (G_::STAGE + 16 + sizeof(StageMeta));
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)out->smem);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, THREADS, out->smem);
    if (e != cudaSuccess) return e;
    out->ctas_per_sm = nb < 1 ? 1 : nb;
    return cudaSuccess;
}

// Stage count, shared memory and residency of one instantiation, computed
// once per device (the attribute set on the first call stays set).
template <int D, bool FP8, int MT>
cudaError_t plan_mt(AttnLaunch *out) {
    static DeviceMemo<AttnLaunch> memo;
    return memo.get(out, plan_mt_uncached<D, FP8, MT>);
}

template <int D, bool FP8, int MT>
cudaError_t launch_mt(const AttnMaps &m, const AttnArgs &a, int grid, size_t smem, cudaStream_t st) {
    constexpr int THREADS = (MT + 1) * 32;
    // D 128 bf16 pages travel as one 5-D box per page (the slab maps are unused)
    const bool whole = D * (FP8 ? 1 : 2) > 128;
    pva_kernel<D, FP8, MT><<<grid, THREADS, smem, st>>>(whole ? m.kslabs : m.k[0], m.k[1], whole ? m.vslabs : m.v[0],
                                                         m.v[1], m.q[0], m.q[1], a);
    return cudaGetLastError();
}

inline int mt_of(int M) {
    const int mt = (M + 15) / 16;
    return mt <= 4 ? mt : (mt <= 6 ? 6 : 8);
}

template <int D, bool FP8>
cudaError_t plan_d(int M, AttnLaunch *o) {
    switch (mt_of(M)) {
        case 1: return plan_mt<D, FP8, 1>(o);
        case 2: return plan_mt<D, FP8, 2>(o);
        case 3: return plan_mt<D, FP8, 3>(o);
        case 4: return plan_mt<D, FP8, 4>(o);
        case 6: return plan_mt<D, FP8, 6>(o);
        default: return plan_mt<D, FP8, 8>(o);
    }
}

template <int D, bool FP8>
cudaError_t launch_d(const AttnMaps &m, const AttnArgs &a, int grid, size_t smem, cudaStream_t st) {
    switch (mt_of(a.M)) {
        case 1: return launch_mt<D, FP8, 1>(m, a, grid, smem, st);
        case 2: return launch_mt<D, FP8, 2>(m, a, grid, smem, st);
        case 3: return launch_mt<D, FP8, 3>(m, a, grid, smem, st);
        case 4: return launch_mt<D, FP8, 4>(m, a, grid, smem, st);
        case 6: return launch_mt<D, FP8, 6>(m, a, grid, smem, st);
        default: return launch_mt<D, FP8, 8>(m, a, grid, smem, st);
    }
}

}  // namespace

namespace {

// Rank of each sequence by decreasing length (ties by index): one CTA, each
// thread counts the sequences that go before its own (B <= kMaxOrderedSeqs).
__global__ void __launch_bounds__(1024) seq_order_kernel(const int32_t *context_lens, int B, int32_t *order) {
    __shared__ int32_t s_len[kMaxOrderedSeqs];
    for (int i = threadIdx.x; i < B; i += blockDim.x) s_len[i] = context_lens[i];
    __syncthreads();
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int li = s_len[i];
        int rank = 0;
        for (int j = 0; j < B; ++j) {
            const int lj = s_len[j];
            rank += (lj > li) || (lj == li && j < i);
        }
        order[rank] = i;
    }
}

}  // namespace

cudaError_t launch_seq_order(const int32_t *context_lens, int B, int32_t *order, cudaStream_t stream) {
    seq_order_kernel<<<1, 1024, 0, stream>>>(context_lens, B, order);
    return cudaGetLastError();
}

cudaError_t attn_plan_launch(int head_dim, bool fp8, int M, AttnLaunch *out) {
    if (head_dim == 128) return fp8 ? plan_d<128, true>(M, out) : plan_d<128, false>(M, out);
    return plan_d<64, false>(M, out);
}

cudaError_t launch_paged_verify_attn(const AttnMaps &maps, const AttnArgs &a, int head_dim, bool fp8,
                                     int grid, size_t smem, cudaStream_t stream) {
    if (head_dim == 128)
        return fp8 ? launch_d<128, true>(maps, a, grid, smem, stream)
                   : launch_d<128, false>(maps, a, grid, smem, stream);
    return launch_d<64, false>(maps, a, grid, smem, stream);
}

}  // namespace svpa
