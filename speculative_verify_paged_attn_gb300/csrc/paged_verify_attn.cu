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
//  * one CTA per (KV split, kv head, sequence): all G*n_q query rows of a kv
//    head share each K/V page, so every page is read from HBM exactly once;
//  * a producer warp streams (K, V) page tiles into a ring of shared-memory
//    stages with 2-D tiled bulk tensor copies (TMA, 128-byte swizzle), one
//    mbarrier pair per stage; pages are gathered by block id from the table;
//  * consumer warps: m16n8k16 tensor-core MMAs (bf16, or f16 on exactly
//    decoded FP8 bytes) for S = Q K^T and O += P V, online softmax in fp32
//    registers with exp2, quad shuffles for the row reductions;
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
};

// Byte offset of 16-byte chunk `ch` of token row `t` inside a swizzled tile:
// each 128-byte slab holds 16 rows of 128 bytes; chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t swz(int t, int ch) {
    return (uint32_t)(((ch >> 3) << 11) + (t << 7) + (((ch & 7) ^ (t & 7)) << 4));
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

template <int D, bool FP8, int MT, int TG>
__global__ void __launch_bounds__((MT * TG + 1) * 32, 1)
    pva_kernel(const __grid_constant__ CUtensorMap mk0, const __grid_constant__ CUtensorMap mk1,
               const __grid_constant__ CUtensorMap mv0, const __grid_constant__ CUtensorMap mv1,
               const __grid_constant__ AttnArgs a) {
    using G_ = Geo<D, FP8>;
    constexpr int NCW = MT * TG;
    constexpr int NCT = NCW * 32;
    constexpr int ACC = G_::ACC;

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int L = a.context_lens[b];
    const int T = L + a.n_q;
    const int npages = (T + kBlockSize - 1) / kBlockSize;
    if (L < 0 || npages > a.max_blocks) {
        if (split == 0 && h == 0 && threadIdx.x == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        return;
    }
    const int nsplit = (npages + a.split_pages - 1) / a.split_pages;
    if (split >= nsplit) return;
    const int page0 = split * a.split_pages;
    const int n = min(a.split_pages, npages - page0);
    const int NS = a.n_stages;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + (size_t)NS * G_::STAGE);
    uint64_t *empty = full + NS;
    int32_t *s_blk = reinterpret_cast<int32_t *>(empty + NS);
    float *s_ks = reinterpret_cast<float *>(s_blk + a.split_pages);
    float *s_vs = s_ks + a.split_pages;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], MT);
        }
        fence_mbar_init();
    }
    // block ids (and FP8 scales) of this split, checked against the pool
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks + page0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int blk = bt[i];
        if (blk < 0 || blk >= a.num_blocks) {
            raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
            blk = 0;
        }
        s_blk[i] = blk;
        if constexpr (FP8) {
            s_ks[i] = a.k_scale[(size_t)blk * a.Hkv + h];
            s_vs[i] = a.v_scale[(size_t)blk * a.Hkv + h];
        }
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            prefetch_tensormap(&mk0);
            prefetch_tensormap(&mv0);
            if constexpr (G_::SLABS > 1) {
                prefetch_tensormap(&mk1);
                prefetch_tensormap(&mv1);
            }
            const uint64_t pol = policy_evict_first();
            int slot = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int i = 0; i < n && ok; ++i) {
                if (i >= NS) ok = mbar_wait(&empty[slot], phase ^ 1u, a.err);
                if (!ok) break;
                uint8_t *st = stages + (size_t)slot * G_::STAGE;
                mbar_arrive_expect_tx(&full[slot], G_::STAGE);
                const int blk = s_blk[i];
                tma_load_4d(st, &mk0, 0, 0, h, blk, &full[slot], pol);
                tma_load_4d(st + G_::TILE, &mv0, 0, 0, h, blk, &full[slot], pol);
                if constexpr (G_::SLABS > 1) {
                    tma_load_4d(st + 2048, &mk1, 0, 0, h, blk, &full[slot], pol);
                    tma_load_4d(st + G_::TILE + 2048, &mv1, 0, 0, h, blk, &full[slot], pol);
                }
                if (++slot == NS) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            // do not leave the CTA with copies in flight: wait (bounded) for
            // the last stages to land
            const int first = n > NS ? n - NS : 0;
            for (int i = first; i < n && ok; ++i) {
                const int sl = i % NS;
                ok = mbar_wait(&full[sl], (uint32_t)((i / NS) & 1), a.err);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    const int grp = warp / MT, mt = warp % MT;
    const int g = lane >> 2, c = lane & 3;
    const int r0 = mt * 16 + g, r1 = r0 + 8;
    const int G = a.G;

    // Q fragments (A operand of m16n8k16), kept in registers for the split
    uint32_t qa[D / 16][4];
    {
        const __nv_bfloat16 *qrow[2] = {nullptr, nullptr};
        const int rr[2] = {r0, r1};
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            if (rr[x] < a.M) {
                const int j = rr[x] / G, gi = rr[x] - j * G;
                qrow[x] = a.q + (((size_t)b * a.n_q + j) * a.Hq + (size_t)h * G + gi) * D;
            }
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                uint32_t lo = 0, hi = 0;
                if (qrow[x]) {
                    if constexpr (!FP8) {
                        lo = *reinterpret_cast<const uint32_t *>(qrow[x] + kk * 16 + 2 * c);
                        hi = *reinterpret_cast<const uint32_t *>(qrow[x] + kk * 16 + 8 + 2 * c);
                    } else {
                        // f16 operands, head-dim order permuted to match the
                        // byte order ldmatrix delivers from FP8 rows
                        const uint2 v = *reinterpret_cast<const uint2 *>(qrow[x] + kk * 16 + 4 * c);
                        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
                        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
                        const float2 f0 = __bfloat1622float2(p0), f1 = __bfloat1622float2(p1);
                        lo = pack_f16x2(f0.x, f0.y);
                        hi = pack_f16x2(f1.x, f1.y);
                    }
                }
                qa[kk][x] = lo;      // a0 (row g) / a1 (row g+8)
                qa[kk][2 + x] = hi;  // a2 / a3
            }
        }
    }
    unsigned long long mrow[2];
    mrow[0] = r0 < a.M ? a.anc[r0 / G] : 0ull;
    mrow[1] = r1 < a.M ? a.anc[r1 / G] : 0ull;

    float acc[ACC / 4][4];
#pragma unroll
    for (int i = 0; i < ACC / 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
    float l_run[2] = {0.f, 0.f};

    int slot = grp, phase = 0;
    for (int i = grp; i < n; i += TG) {
        // stage `slot` holds page i; its use count is i / NS
        while (slot >= NS) {
            slot -= NS;
            phase ^= 1;
        }
        if (!mbar_wait(&full[slot], (uint32_t)phase, a.err)) break;
        uint8_t *kt = stages + (size_t)slot * G_::STAGE;
        uint8_t *vt = kt + G_::TILE;
        const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
        const int pos0 = (page0 + i) * kBlockSize;

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
            const int tok = ((lane >> 4) << 3) + (lane & 7);
            const int par = (lane >> 3) & 1;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b00, b01, b10, b11;
                ldmatrix_x4(kbase + swz(tok, 2 * kk + par), b00, b01, b10, b11);
                mma_bf16_16816(s[0], qa[kk], b00, b01);
                mma_bf16_16816(s[1], qa[kk], b10, b11);
            }
        } else {
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                uint32_t r0k, r1k, r2k, r3k;
                ldmatrix_x4(kbase + swz(tok, 2 * kp + par), r0k, r1k, r2k, r3k);
                mma_f16_16816(s[0], qa[2 * kp], e4m3x2_to_f16x2(r0k & 0xffff), e4m3x2_to_f16x2(r0k >> 16));
                mma_f16_16816(s[1], qa[2 * kp], e4m3x2_to_f16x2(r1k & 0xffff), e4m3x2_to_f16x2(r1k >> 16));
                mma_f16_16816(s[0], qa[2 * kp + 1], e4m3x2_to_f16x2(r2k & 0xffff), e4m3x2_to_f16x2(r2k >> 16));
                mma_f16_16816(s[1], qa[2 * kp + 1], e4m3x2_to_f16x2(r3k & 0xffff), e4m3x2_to_f16x2(r3k >> 16));
            }
        }
        float sc = a.scale_log2;
        if constexpr (FP8) sc *= s_ks[i];
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
        uint32_t pa[4];
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
            float mx = fmaxf(fmaxf(s[0][2 * rh], s[0][2 * rh + 1]), fmaxf(s[1][2 * rh], s[1][2 * rh + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(m_run[rh], mx);
            const float msafe = mnew == -CUDART_INF_F ? 0.f : mnew;
            alpha[rh] = exp2f(m_run[rh] - msafe);
            m_run[rh] = mnew;
            const float p00 = exp2f(s[0][2 * rh] - msafe), p01 = exp2f(s[0][2 * rh + 1] - msafe);
            const float p10 = exp2f(s[1][2 * rh] - msafe), p11 = exp2f(s[1][2 * rh + 1] - msafe);
            l_run[rh] = l_run[rh] * alpha[rh] + (p00 + p01) + (p10 + p11);
            if constexpr (!FP8) {
                pa[rh] = pack_bf16x2(p00, p01);
                pa[2 + rh] = pack_bf16x2(p10, p11);
            } else {
                pa[rh] = pack_f16x2(p00, p01);
                pa[2 + rh] = pack_f16x2(p10, p11);
            }
        }

        // ---- O = alpha * O + P V
        if constexpr (!FP8) {
#pragma unroll
            for (int x = 0; x < ACC / 4; ++x)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[x][e] *= alpha[e >> 1];
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(vbase + swz(tok, 2 * np + par), v0, v1, v2, v3);
                mma_bf16_16816(acc[2 * np], pa, v0, v1);
                mma_bf16_16816(acc[2 * np + 1], pa, v2, v3);
            }
        } else {
            const float vs = s_vs[i];
            const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
            const int par = lane >> 4;
#pragma unroll
            for (int cp = 0; cp < D / 32; ++cp) {
                uint32_t r0v, r1v, r2v, r3v;
                ldmatrix_x4_trans(vbase + swz(tok, 2 * cp + par), r0v, r1v, r2v, r3v);
                // chunk 2cp from (r0v, r1v), chunk 2cp+1 from (r2v, r3v);
                // even / odd head-dim columns of each chunk are separate n-tiles
                const uint32_t ev0 = __byte_perm(r0v, r1v, 0x6420), od0 = __byte_perm(r0v, r1v, 0x7531);
                const uint32_t ev1 = __byte_perm(r2v, r3v, 0x6420), od1 = __byte_perm(r2v, r3v, 0x7531);
                float t[4][4];
#pragma unroll
                for (int y = 0; y < 4; ++y)
#pragma unroll
                    for (int e = 0; e < 4; ++e) t[y][e] = 0.f;
                mma_f16_16816(t[0], pa, e4m3x2_to_f16x2(ev0 & 0xffff), e4m3x2_to_f16x2(ev0 >> 16));
                mma_f16_16816(t[1], pa, e4m3x2_to_f16x2(od0 & 0xffff), e4m3x2_to_f16x2(od0 >> 16));
                mma_f16_16816(t[2], pa, e4m3x2_to_f16x2(ev1 & 0xffff), e4m3x2_to_f16x2(ev1 >> 16));
                mma_f16_16816(t[3], pa, e4m3x2_to_f16x2(od1 & 0xffff), e4m3x2_to_f16x2(od1 >> 16));
#pragma unroll
                for (int y = 0; y < 4; ++y)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float &dst = acc[(2 * cp) * 2 + y][e];
                        dst = fmaf(t[y][e], vs, dst * alpha[e >> 1]);
                    }
            }
        }

        __syncwarp();
        if (tail) fence_proxy_async_smem();
        if (lane == 0) mbar_arrive(&empty[slot]);
        slot += TG;
    }

    // full row sums
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
        l_run[rh] += __shfl_xor_sync(0xffffffffu, l_run[rh], 1);
        l_run[rh] += __shfl_xor_sync(0xffffffffu, l_run[rh], 2);
    }

    // ---- merge the token groups of this CTA (same rows, disjoint pages)
    if constexpr (TG > 1) {
        named_barrier_sync(kBarConsumers, NCT);
        float *red = reinterpret_cast<float *>(stages);
        constexpr int RS = ACC + 4;
        if (grp > 0) {
            float *dst = red + ((size_t)((grp - 1) * MT + mt) * RS) * 32 + lane;
#pragma unroll
            for (int x = 0; x < ACC; ++x) dst[x * 32] = acc[x >> 2][x & 3];
            dst[ACC * 32] = m_run[0];
            dst[(ACC + 1) * 32] = m_run[1];
            dst[(ACC + 2) * 32] = l_run[0];
            dst[(ACC + 3) * 32] = l_run[1];
        }
        named_barrier_sync(kBarConsumers, NCT);
        if (grp == 0) {
            for (int og = 1; og < TG; ++og) {
                const float *src = red + ((size_t)((og - 1) * MT + mt) * RS) * 32 + lane;
                float wa[2], wb[2];
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {
                    const float mb = src[(ACC + rh) * 32];
                    const float lb = src[(ACC + 2 + rh) * 32];
                    const float mnew = fmaxf(m_run[rh], mb);
                    const float msafe = mnew == -CUDART_INF_F ? 0.f : mnew;
                    wa[rh] = exp2f(m_run[rh] - msafe);
                    wb[rh] = exp2f(mb - msafe);
                    m_run[rh] = mnew;
                    l_run[rh] = l_run[rh] * wa[rh] + lb * wb[rh];
                }
#pragma unroll
                for (int x = 0; x < ACC; ++x) {
                    const int rh = (x & 2) >> 1;
                    acc[x >> 2][x & 3] = acc[x >> 2][x & 3] * wa[rh] + src[x * 32] * wb[rh];
                }
            }
        }
    }

    const int unit = b * a.Hkv + h;
    if (grp == 0) {
        const int rows[2] = {r0, r1};
        if (nsplit == 1) {
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int R = rows[rh];
                if (R >= a.M) continue;
                const int j = R / G, gi = R - j * G;
                const size_t o = (((size_t)b * a.n_q + j) * a.Hq + (size_t)h * G + gi);
                const float inv = l_run[rh] > 0.f ? 1.f / l_run[rh] : 0.f;
                __nv_bfloat16 *orow = a.out + o * D;
#pragma unroll
                for (int x = 0; x < ACC; ++x)
                    if (((x & 2) >> 1) == rh) orow[acc_col<FP8>(x, c)] = __float2bfloat16_rn(acc[x >> 2][x & 3] * inv);
                if (a.lse && c == 0)
                    a.lse[o] = (m_run[rh] + log2f(l_run[rh])) * 0.69314718055994530942f;
            }
        } else {
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int R = rows[rh];
                if (R >= a.M) continue;
                const size_t pr = ((size_t)unit * a.max_splits + split) * a.M + R;
                float *prow = a.part_acc + pr * D;
#pragma unroll
                for (int x = 0; x < ACC; ++x)
                    if (((x & 2) >> 1) == rh) prow[acc_col<FP8>(x, c)] = acc[x >> 2][x & 3];
                if (c == 0) {
                    a.part_ml[pr * 2] = m_run[rh];
                    a.part_ml[pr * 2 + 1] = l_run[rh];
                }
            }
            __threadfence();
        }
    }
    if (nsplit == 1) return;

    // ---- split-KV: the last CTA of this (sequence, kv head) combines
    named_barrier_sync(kBarConsumers, NCT);
    if (threadIdx.x == 0) {
        const int t = atomicAdd(&a.tickets[unit], 1);
        s_last = (t == nsplit - 1);
        if (s_last) a.tickets[unit] = 0;  // self-cleaning for the next call
    }
    named_barrier_sync(kBarConsumers, NCT);
    if (!s_last) return;
    __threadfence();
    constexpr int PER = D / 32;  // head-dim columns per lane
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
#pragma unroll
        for (int x = 0; x < PER; ++x) orow[x] = __float2bfloat16_rn(o[x] * inv);
        if (a.lse && lane == 0) a.lse[od] = (mx + log2f(l)) * 0.69314718055994530942f;
    }
}

template <int D, bool FP8, int MT>
cudaError_t launch_mt(const AttnMaps &m, const AttnArgs &a, cudaStream_t st) {
    constexpr int TG = MT == 1 ? 4 : (MT <= 4 ? 2 : 1);
    constexpr int THREADS = (MT * TG + 1) * 32;
    auto kern = pva_kernel<D, FP8, MT, TG>;
    const size_t smem = attn_smem_bytes(D, FP8, a.n_stages, a.split_pages);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.max_splits, a.Hkv, a.B);
    kern<<<grid, THREADS, smem, st>>>(m.k[0], m.k[1], m.v[0], m.v[1], a);
    return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_d(const AttnMaps &m, const AttnArgs &a, cudaStream_t st) {
    const int mt = (a.M + 15) / 16;
    switch (mt) {
        case 1: return launch_mt<D, FP8, 1>(m, a, st);
        case 2: return launch_mt<D, FP8, 2>(m, a, st);
        case 3: return launch_mt<D, FP8, 3>(m, a, st);
        case 4: return launch_mt<D, FP8, 4>(m, a, st);
        case 5:
        case 6: return launch_mt<D, FP8, 6>(m, a, st);
        default: return launch_mt<D, FP8, 8>(m, a, st);
    }
}

template <int D, bool FP8, int MT>
int stages_mt(int split_pages) {
    constexpr int TG = MT == 1 ? 4 : (MT <= 4 ? 2 : 1);
    constexpr int THREADS = (MT * TG + 1) * 32;
    using G_ = Geo<D, FP8>;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, pva_kernel<D, FP8, MT, TG>) != cudaSuccess) return -1;
    // registers are allocated per warp in units of 256
    const int per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
    int ctas = 65536 / (per_warp * (THREADS / 32));
    ctas = ctas < 1 ? 1 : (ctas > 4 ? 4 : ctas);
    const int per_cta = 232448 / ctas - 1024 - (int)fa.sharedSizeBytes;
    const int fixed = 1024 + 12 * split_pages + 64;
    int ns = (per_cta - fixed) / (G_::STAGE + 16);
    // the token-group merge reuses the stage ring
    const int red = (TG - 1) * MT * (G_::ACC + 4) * 32 * 4;
    const int ns_min = (red + G_::STAGE - 1) / G_::STAGE;
    ns = ns > 32 ? 32 : ns;
    if (ns < 4) ns = 4;
    if (ns < ns_min) ns = ns_min;
    return ns;
}

template <int D, bool FP8>
int stages_d(int M, int split_pages) {
    switch ((M + 15) / 16) {
        case 1: return stages_mt<D, FP8, 1>(split_pages);
        case 2: return stages_mt<D, FP8, 2>(split_pages);
        case 3: return stages_mt<D, FP8, 3>(split_pages);
        case 4: return stages_mt<D, FP8, 4>(split_pages);
        case 5:
        case 6: return stages_mt<D, FP8, 6>(split_pages);
        default: return stages_mt<D, FP8, 8>(split_pages);
    }
}

}  // namespace

int attn_pick_stages(int head_dim, bool fp8, int M, int split_pages) {
    if (head_dim == 128) return fp8 ? stages_d<128, true>(M, split_pages) : stages_d<128, false>(M, split_pages);
    return stages_d<64, false>(M, split_pages);
}

size_t attn_smem_bytes(int head_dim, bool fp8, int n_stages, int split_pages) {
    const size_t stage = 2 * 16 * (size_t)head_dim * (fp8 ? 1 : 2);
    return 1024 + stage * n_stages + 16 * (size_t)n_stages + 12 * (size_t)split_pages + 64;
}

cudaError_t launch_paged_verify_attn(const AttnMaps &maps, const AttnArgs &a, int head_dim, bool fp8,
                                     cudaStream_t stream) {
    if (head_dim == 128) return fp8 ? launch_d<128, true>(maps, a, stream) : launch_d<128, false>(maps, a, stream);
    return launch_d<64, false>(maps, a, stream);
}

}  // namespace svpa
