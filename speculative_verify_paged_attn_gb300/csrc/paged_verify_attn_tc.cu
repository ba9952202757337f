// paged_verify_attn_tc.cu -- paged verification attention on the 5th-generation
// tensor cores (tcgen05 + TMEM) for sm_103a, used when one kv head carries
// many query rows (grouped-query models, draft trees: G * n_q up to 128).
//
// Same computation as paged_verify_attn.cu ("The Sub-Millisecond Speculative
// Decoding Meltdown", section "Speculative Decoding Mechanics & The K-Token
// Penalty": A = softmax(Q K^T * scale + M_tree) V over a paged K/V history;
// "Triton CUDA Fused Speculative Tree-Verification Kernel": per-page block
// lookup, K/V cache [blocks, heads, 16, dim], running max / sum).
//
// Work unit = (sequence, kv head, KV split); persistent CTAs, one per SM
// (unsplit units are handed out longest sequence first, in the order a small
// ranking kernel leaves in the workspace).
// Warp roles:
//   warp 0     producer: takes units from an atomic counter and streams blocks
//              of 8 pages (128 tokens) of K -- with each unit's query tile on
//              its first block -- and, one block behind, of V, with tiled TMA
//              copies (128-byte swizzle) into 3-deep K and V rings; lanes 0..7
//              issue one page each; missing pages of a unit's last block are
//              fetched at an out-of-range block coordinate (zero fill);
//   warp 1     MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T
//              (M 128, N 128, K 128) into one of two TMEM S buffers, issued
//              ahead of PV_{j-1} when K_j has already landed, and
//              O += P_j V_j (M 128, N 128, K 128) with P_j read from TMEM,
//              into one of two TMEM O buffers (one per unit in flight);
//   warps 2-5  softmax, one thread per query row (TMEM lane): S row from
//              TMEM, mask (only on blocks that reach the speculative slots),
//              online softmax with a lazy reference maximum (O is rescaled in
//              TMEM only when a row maximum grows by more than 2^8), P row as
//              bf16 pairs written over the S columns it came from;
//   warps 6-9  epilogue, one thread per query row: a finished unit's O from
//              TMEM to the output (or a split partial, merged by the last
//              split's CTA with log-sum-exp weights, one warp per row) while
//              the softmax warps run the next unit.
// All waits are bounded; nothing spins forever.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstddef>
#include <type_traits>

#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kD = 128;
constexpr int kPagesPerBlock = 8;
constexpr int kNB = kPagesPerBlock * 16;       // tokens per block (128)
constexpr int kRows = 128;                      // MMA M
constexpr int kKVTile = kNB * 256;              // K (or V) block: 8 pages of 4 KB
constexpr int kNMeta = 8;                       // block descriptors in flight
constexpr int kBarEpi = 1;                      // named barrier of the epilogue warps

// Warps 0 producer, 1 MMA, 2-5 softmax, 6-9 epilogue; 3-deep K and V rings
// of bf16 blocks that the MMA reads directly.  (FP8 pages take
// paged_verify_attn_f8.cu's kernel.)
struct TcCfg {
    static constexpr int kThreads = 320;
    static constexpr int kNK = 3;               // tiles the MMA reads (K freed once S_j is done)
    static constexpr int kNV = 3;               // (V freed once PV_j is done)
    static constexpr int kQSlab = 128 * 128;    // one 64-column slab of the query buffer
    static constexpr int kQBuf = 2 * kQSlab;
    static constexpr int kSoftmaxWarp0 = 2;
    static constexpr int kSoftmaxWarps = 4;
    static constexpr int kEpiWarp0 = 6;
    static constexpr int kEpiWarps = 4;
};
constexpr float kRescaleLog2 = 8.f;             // rescale O when a maximum grows by > 2^8

// TMEM columns: O[0] 0..127, O[1] 128..255, S[0] 256..383, S[1] 384..511; the
// softmax overwrites the first 64 columns of S[x] with P (bf16 pairs), which
// the PV MMA reads as its A operand straight from TMEM.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 256;

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagEnd = 4;

struct BlockMeta {
    int32_t b, h, split, pos0, ntok, L, nsplit, flags, qb;
    int32_t pad[3];
};

struct Smem {
    using C = TcCfg;
    uint8_t q[C::kQBuf];                 // 1024-aligned (one unit's queries)
    uint8_t kbuf[C::kNK][kKVTile];       // 32 KB each
    uint8_t vbuf[C::kNV][kKVTile];
    uint64_t k_full[C::kNK], k_empty[C::kNK];
    uint64_t v_full[C::kNV], v_empty[C::kNV];
    uint64_t q_empty;
    uint64_t s_full[2];
    uint64_t p_full, p_empty;
    uint64_t o_full[2], o_empty[2];
    uint64_t stat_full, stat_empty;      // softmax -> epilogue hand-off of a finished unit
    BlockMeta meta[kNMeta];
    int32_t vid[kNMeta][kPagesPerBlock];  // page ids of a block, for its V copies
    float2 stat[kRows];                  // (reference maximum, running sum) per row
    int32_t ep_b, ep_h, ep_split, ep_nsplit, ep_end;
    uint32_t tmem_base;
    int32_t last;
};

// fits the 227 KB a CTA may opt into, with room to align the base to 1 KB
static_assert(sizeof(Smem) + 1024 <= 232448, "pva_tc_kernel shared memory");

__device__ __forceinline__ uint32_t par_of(int idx) { return (uint32_t)((idx >> 1) & 1); }

__global__ void __launch_bounds__(TcCfg::kThreads, 1)
    pva_tc_kernel(const __grid_constant__ CUtensorMap mkp, const __grid_constant__ CUtensorMap mvp,
                  const __grid_constant__ CUtensorMap mq0, const __grid_constant__ CUtensorMap mq1,
                  const __grid_constant__ AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    using C = TcCfg;
    constexpr int kNK = C::kNK, kNV = C::kNV, kQSlab = C::kQSlab, kQBuf = C::kQBuf;
    Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNK; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
        }
        for (int i = 0; i < kNV; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.o_full[i], 1);
            mbar_init(&sm.o_empty[i], C::kEpiWarps);
        }
        mbar_init(&sm.q_empty, 1);
        mbar_init(&sm.p_full, C::kSoftmaxWarps);
        mbar_init(&sm.p_empty, 1);
        mbar_init(&sm.stat_full, C::kSoftmaxWarps);
        mbar_init(&sm.stat_empty, C::kEpiWarps);
        fence_mbar_init();
    }
    // query rows past M are never written by the copies: keep them zero
    for (int x = threadIdx.x; x < kQBuf / 16; x += blockDim.x)
        reinterpret_cast<uint4 *>(&sm.q[0])[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ================================================= producer
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&mkp);
            prefetch_tensormap(&mvp);
            prefetch_tensormap(&mq0);
            prefetch_tensormap(&mq1);
        }
        int jk = 0, jv = 0, units = 0;      // K blocks issued, V blocks issued, units started (warp-uniform)
        bool ok = true;
        const uint32_t qbytes = (uint32_t)(a.M * 128 * 2);
        // the rings the copies land in: the MMA's tiles
        constexpr int PNK = kNK, PNV = kNV;
        constexpr uint32_t kBlockBytes = kKVTile;
        uint64_t *pk_full = sm.k_full, *pk_empty = sm.k_empty, *pv_full = sm.v_full, *pv_empty = sm.v_empty;
        // one copy per page: a 5-D box of a bf16 tile
        auto copy_page = [&](const CUtensorMap *map, uint8_t *ring_slot, int id, int hh, uint64_t *bar) {
            tma_load_5d(ring_slot + lane * 4096, map, 0, 0, 0, 0, id * a.Hkv + hh, bar, pol);
        };
        auto k_slot = [&](int s_) -> uint8_t * { return sm.kbuf[s_]; };
        auto v_slot = [&](int s_) -> uint8_t * { return sm.vbuf[s_]; };
        // V of the oldest block whose K is out, if its ring slot is free (a
        // non-blocking test): K runs ahead as far as its own ring allows and
        // V follows as PV frees slots, neither waiting for the other
        auto try_issue_v = [&]() -> bool {
            if (jv >= jk) return false;
            const int vs = jv % PNV;
            int ready = 1;
            if (lane == 0 && jv >= PNV) ready = mbar_test(&pv_empty[vs], (uint32_t)(((jv / PNV) & 1) ^ 1));
            if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
            if (lane == 0) mbar_arrive_expect_tx(&pv_full[vs], kBlockBytes);
            if (lane < kPagesPerBlock) {
                const int id = sm.vid[jv % kNMeta][lane], hh = sm.meta[jv % kNMeta].h;
                copy_page(&mvp, v_slot(vs), id, hh, &pv_full[vs]);
            }
            __syncwarp();
            ++jv;
            return true;
        };
        // bounded wait for phase `parity` of `bar`, issuing V copies meanwhile
        auto wait_issuing_v = [&](uint64_t *bar, uint32_t parity) -> bool {
            unsigned long long t0 = 0;
            while (true) {
                int done = 0;
                if (lane == 0) done = mbar_test(bar, parity);
                if (__shfl_sync(0xffffffffu, done, 0)) return true;
                if (try_issue_v()) {
                    t0 = 0;
                    continue;
                }
                // nothing to do yet: back off so the spin does not take issue
                // slots from the softmax warp sharing this scheduler
                __nanosleep(64);
                const unsigned long long now = global_ns();
                if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > kWaitLimitNs) {
                    if (lane == 0) raise_error(a.err, SVPA_DEVERR_TIMEOUT);
                    return false;
                }
            }
        };
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
            const int nblk = (n + kPagesPerBlock - 1) / kPagesPerBlock;
            const int32_t *bt = a.block_table + (size_t)b * a.max_blocks + page0;
            int blk_next = a.num_blocks;
            for (int i0 = 0; i0 < n && ok; i0 += 32) {
                int blk = a.num_blocks;  // out of range: zero-filled page
                if (i0 == 0) {
                    if (lane < n) blk = __ldg(bt + lane);
                } else {
                    blk = blk_next;
                }
                if (i0 + lane < n && (blk < 0 || blk >= a.num_blocks)) {
                    raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
                    blk = 0;
                }
                blk_next = a.num_blocks;
                if (i0 + 32 + lane < n) blk_next = __ldg(bt + i0 + 32 + lane);
                const int cnt = min(32, n - i0);
                for (int j0 = 0; j0 < cnt; j0 += kPagesPerBlock) {
                    // lanes 0..7 hold the ids of the block's 8 pages
                    int my_id = __shfl_sync(0xffffffffu, blk, (j0 + (lane & 7)) & 31);
                    if (j0 + (lane & 7) >= cnt) my_id = a.num_blocks;
                    const int bi = (i0 + j0) / kPagesPerBlock;  // block index in the unit
                    const int ks = jk % PNK;
                    if (jk >= PNK) ok = wait_issuing_v(&pk_empty[ks], (uint32_t)(((jk / PNK) & 1) ^ 1));
                    // the query tile is reloaded once the previous unit's last S is done
                    if (ok && bi == 0 && units >= 1) ok = wait_issuing_v(&sm.q_empty, (uint32_t)((units - 1) & 1));
                    if (!ok) break;
                    if (lane == 0) {
                        BlockMeta &m = sm.meta[jk % kNMeta];
                        m.b = b; m.h = h; m.split = split; m.L = L; m.nsplit = nsplit; m.qb = 0;
                        m.pos0 = (page0 + i0 + j0) * kBlockSize;
                        m.ntok = min(kPagesPerBlock, n - (i0 + j0)) * kBlockSize;
                        m.flags = (bi == 0 ? kFlagFirst : 0) | (bi == nblk - 1 ? kFlagLast : 0);
                        // the query tile rides on the unit's first K block
                        uint64_t *qbar = &pk_full[ks];
                        mbar_arrive_expect_tx(&pk_full[ks], kBlockBytes + (bi == 0 ? qbytes : 0u));
                        if (bi == 0) {
                            tma_load_4d(&sm.q[0], &mq0, 0, h * a.G, 0, b, qbar, pol);
                            tma_load_4d(&sm.q[kQSlab], &mq1, 0, h * a.G, 0, b, qbar, pol);
                        }
                    }
                    if (lane < kPagesPerBlock) {
                        sm.vid[jk % kNMeta][lane] = my_id;
                        copy_page(&mkp, k_slot(ks), my_id, h, &pk_full[ks]);
                    }
                    __syncwarp();
                    ++jk;
                    try_issue_v();
                }
            }
            ++units;
        }
        // the V copies still owed
        while (ok && jv < jk) {
            if (jv >= PNV) {
                int good = 1;
                if (lane == 0) good = mbar_wait(&pv_empty[jv % PNV], (uint32_t)(((jv / PNV) & 1) ^ 1), a.err);
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
            if (ok) try_issue_v();
        }
        if (lane == 0) {
            // end-of-work marker on the K ring
            const int ks = jk % PNK;
            if (ok && jk >= PNK) ok = mbar_wait(&pk_empty[ks], (uint32_t)(((jk / PNK) & 1) ^ 1), a.err);
            if (ok) {
                sm.meta[jk % kNMeta].flags = kFlagEnd;
                mbar_arrive_cnt(&pk_full[ks], 1u);
            }
            // wait (bounded) for the copies still in flight; a stage reused
            // by an end marker had completed before its empty barrier passed
            for (int i = jk >= PNK ? jk - PNK + 1 : 0; i < jk && ok; ++i)
                ok = mbar_wait(&pk_full[i % PNK], (uint32_t)((i / PNK) & 1), a.err);
            for (int i = jv >= PNV ? jv - PNV : 0; i < jv && ok; ++i)
                ok = mbar_wait(&pv_full[i % PNV], (uint32_t)((i / PNV) & 1), a.err);
            __threadfence();
            const int done = atomicAdd(&a.sched[1], 1);
            if (done == (int)gridDim.x - 1) {
                a.sched[0] = 0;
                a.sched[1] = 0;
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = umma_idesc_bf16(kRows, kNB, false);
            constexpr uint32_t idPV = umma_idesc_bf16(kRows, kD, true);
            const uint32_t qaddr = smem_u32(&sm.q[0]);
            // S_jj = Q K_jj^T once K_jj has landed (or forward the end marker)
            // buf_wait: wait for PV_{jj-2} (whose P shares S_jj's TMEM buffer);
            // callers pass false when they already know it has completed
            auto issue_s = [&](int jj, int &unit_jj, BlockMeta &m, bool buf_wait) -> bool {
                const int ks = jj % kNK;
                if (!mbar_wait(&sm.k_full[ks], (uint32_t)((jj / kNK) & 1), a.err)) return false;
                m = sm.meta[jj % kNMeta];
                // S buffer jj&1 holds P_{jj-2} until PV_{jj-2} has read it.  Only
                // waited while PV_{jj-1} cannot have completed yet, so the
                // barrier is never two phases ahead of the one tested.
                if (buf_wait && jj >= 2 && !mbar_wait(&sm.p_empty, (uint32_t)((jj - 2) & 1), a.err))
                    return false;
                if (m.flags & kFlagEnd) {
                    mbar_arrive(&sm.s_full[jj & 1]);
                    return true;
                }
                if (m.flags & kFlagFirst) ++unit_jj;
                tc_fence_after();
                const uint32_t qa = qaddr;
                const uint32_t ka = smem_u32(sm.kbuf[ks]);
                const uint32_t dS = tmem + kTmemS + (uint32_t)(jj & 1) * kNB;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t ad = umma_desc_sw128(qa + (kk >> 2) * kQSlab + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = umma_desc_sw128(ka + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048);
                    umma_bf16(dS, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.k_empty[ks]);
                umma_commit(&sm.s_full[jj & 1]);
                if (m.flags & kFlagLast) umma_commit(&sm.q_empty);
                return true;
            };
            BlockMeta cur, nxt;
            int j = 0, unit = -1;
            bool ok = issue_s(0, unit, cur, true);
            while (ok && !(cur.flags & kFlagEnd)) {
                int unit1 = unit;
                // S of block j+1 early when its K is already there; PV_j never
                // waits for the next block's data
                bool next_done = false;
                if (mbar_test(&sm.k_full[(j + 1) % kNK], (uint32_t)(((j + 1) / kNK) & 1))) {
                    ok = issue_s(j + 1, unit1, nxt, true);  // PV_j not issued yet
                    next_done = true;
                    if (!ok) break;
                }
                // O += P_j V_j once the softmax has written P_j and V_j has landed
                if (!mbar_wait(&sm.p_full, (uint32_t)(j & 1), a.err)) break;
                const int ob = unit & 1;
                if ((cur.flags & kFlagFirst) && unit >= 2 &&
                    !mbar_wait(&sm.o_empty[ob], par_of(unit) ^ 1u, a.err))
                    break;
                const int vs = j % kNV;
                if (!mbar_wait(&sm.v_full[vs], (uint32_t)((j / kNV) & 1), a.err)) break;
                // S_{j+1} will be issued after PV_j: settle its buffer now
                if (!next_done && j >= 1 && !mbar_wait(&sm.p_empty, (uint32_t)((j - 1) & 1), a.err)) break;
                tc_fence_after();
                const uint32_t pt = tmem + kTmemS + (uint32_t)(j & 1) * kNB;  // P_j (bf16 pairs)
                // V_j: page kt at kt * 4 KB as [row half][slab][8 rows][128 B]; one
                // MMA per page
                const uint32_t va = smem_u32(sm.vbuf[vs]);
                const uint32_t dO = tmem + kTmemO + (uint32_t)ob * kD;
#pragma unroll
                for (int kt = 0; kt < kNB / 16; ++kt) {
                    const uint64_t bd = umma_desc_sw128(va + kt * 4096, 1024, 2048);
                    umma_bf16_tmem_a(dO, pt + kt * 8, bd, idPV, ((cur.flags & kFlagFirst) && kt == 0) ? 0u : 1u);
                }
                umma_commit(&sm.v_empty[vs]);
                umma_commit(&sm.p_empty);
                if (cur.flags & kFlagLast) umma_commit(&sm.o_full[ob]);
                if (!next_done) {
                    ok = issue_s(j + 1, unit1, nxt, false);
                    if (!ok) break;
                }
                ++j;
                unit = unit1;
                cur = nxt;
            }
        }
        __syncwarp();
    } else if (warp >= C::kSoftmaxWarp0 && warp < C::kSoftmaxWarp0 + C::kSoftmaxWarps) {
        // ================================================= softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;          // query row == TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int G = a.G;
        const bool live = r < a.M;
        const int jq = live ? r / G : 0;
        const unsigned long long anc = live ? a.anc[jq] : 0ull;
        float m_ref = -CUDART_INF_F, l_run = 0.f;
        int j = 0, unit = -1;
        while (true) {
            if (!mbar_wait(&sm.s_full[j & 1], par_of(j), a.err)) break;
            const BlockMeta md = sm.meta[j % kNMeta];
            if (md.flags & kFlagEnd) {
                // tell the epilogue warps there is no further unit
                if (unit >= 0) mbar_wait(&sm.stat_empty, (uint32_t)(unit & 1), a.err);
                if (threadIdx.x == C::kSoftmaxWarp0 * 32) sm.ep_end = 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.stat_full);
                break;
            }
            if (md.flags & kFlagFirst) {
                ++unit;
                m_ref = -CUDART_INF_F;
                l_run = 0.f;
            }
            tc_fence_after();
            float s[kNB];
            {
                const uint32_t sa = tmem + kTmemS + (uint32_t)(j & 1) * kNB + lane_off;
#pragma unroll
                for (int c = 0; c < kNB / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(sa + c * 32, raw);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(raw[t]);
                }
            }

            const int L = md.L, T = L + a.n_q;
            // The hot path below is kept short on purpose (this code runs
            // once per 64-token block for every query row): max of the raw
            // scores, the scale folded into the exponent's FMA, and masking
            // only on the blocks that reach the speculative slots or a
            // partial block.
            if (md.pos0 + kNB > L || md.ntok < kNB) {
                // visibility of the block's tokens, 64 per bit mask word
                const int h0 = L - md.pos0;  // tokens of the block that are history
#pragma unroll
                for (int w = 0; w < kNB / 64; ++w) {
                    const int hw = min(max(h0 - 64 * w, 0), 64);
                    unsigned long long vis = hw == 64 ? ~0ull : ((1ull << hw) - 1ull);
                    const int sh = h0 - 64 * w;  // bit of speculative slot 0 in this word
                    if (sh >= 0) {
                        if (sh < 64) vis |= anc << sh;
                    } else if (-sh < 64) {
                        vis |= anc >> (-sh);
                    }
                    const int nw = min(max(md.ntok - 64 * w, 0), 64);
                    if (nw < 64) vis &= (1ull << nw) - 1ull;
#pragma unroll
                    for (int t = 0; t < 64; ++t)
                        if (!((vis >> t) & 1ull)) s[64 * w + t] = -CUDART_INF_F;
                }
            }
            // per-page maxima of the raw scores
            float pm[kPagesPerBlock];
#pragma unroll
            for (int x = 0; x < kPagesPerBlock; ++x) pm[x] = s[16 * x];
#pragma unroll
            for (int t = 0; t < kNB; ++t)
                if (t & 15) pm[t >> 4] = fmaxf(pm[t >> 4], s[t]);
            const float mraw = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                     fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
            const float mx = mraw == -CUDART_INF_F ? -CUDART_INF_F : mraw * a.scale_log2;
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_ref + kRescaleLog2 || (m_ref == -CUDART_INF_F && mx != -CUDART_INF_F)) {
                alpha = ex2_approx(m_ref - mx);  // 0 when m_ref is -inf
                m_ref = mx;
                rescale = !(md.flags & kFlagFirst) && l_run > 0.f;
                l_run *= alpha;
            }
            const float neg_m = m_ref == -CUDART_INF_F ? 0.f : -m_ref;
            const float sc = a.scale_log2;
            // P_j as bf16 pairs into the first half of S_j's TMEM columns
            const uint32_t pt = tmem + kTmemS + (uint32_t)(j & 1) * kNB + lane_off;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kNB / 64; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = live ? ex2_approx(fmaf(s[c * 64 + 2 * e], sc, neg_m)) : 0.f;
                    const float p1 = live ? ex2_approx(fmaf(s[c * 64 + 2 * e + 1], sc, neg_m)) : 0.f;
                    ls[e & 3] += p0 + p1;
                    w[e] = pack_bf16x2(p0, p1);
                }
                tmem_st32(pt + c * 32, w);
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // V rows past the sequence's last token may hold anything: zero
            // them once V_j has landed (PV_j is not issued before p_full)
            if (md.pos0 + md.ntok > T) {
                mbar_wait(&sm.v_full[j % kNV], (uint32_t)((j / kNV) & 1), a.err);
                const int t0 = T - md.pos0;
                const int nz = (md.ntok - t0) * 2 * 8;
                uint8_t *sv = sm.vbuf[j % kNV];
                for (int z = threadIdx.x - C::kSoftmaxWarp0 * 32; z < nz; z += C::kSoftmaxWarps * 32) {
                    const int row = t0 + z / 16, rem = z % 16;
                    *reinterpret_cast<uint4 *>(sv + (row >> 3) * 2048 + (rem >> 3) * 1024 + (row & 7) * 128 +
                                               ((rem & 7) << 4)) = make_uint4(0, 0, 0, 0);
                }
            }
            // TMEM loads and stores are warp-collective: the whole warp takes
            // the rescale path when any of its rows needs it (factor 1 elsewhere)
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? alpha : 1.f;
                // O (TMEM) holds P_{<j} V; PV_{j-1} must have landed first
                mbar_wait(&sm.p_empty, (uint32_t)((j - 1) & 1), a.err);
                tc_fence_after();
                const uint32_t oa = tmem + kTmemO + (uint32_t)(unit & 1) * kD + lane_off;
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(oa + c * 32, raw);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) raw[t] = __float_as_uint(__uint_as_float(raw[t]) * f);
                    tmem_st32(oa + c * 32, raw);
                }
                tmem_st_wait();
            }
            tmem_st_wait();
            // P_j is published only once PV_{j-1} has completed (PV_j cannot
            // have started), which keeps the MMA issuer's p_full and p_empty
            // waits unambiguous
            if (j >= 1) mbar_wait(&sm.p_empty, (uint32_t)((j - 1) & 1), a.err);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full);

            if (md.flags & kFlagLast) {
                // hand the unit's row statistics to the epilogue warps (one
                // slot: the previous unit's must have been taken)
                if (unit >= 1) mbar_wait(&sm.stat_empty, (uint32_t)((unit - 1) & 1), a.err);
                sm.stat[r] = make_float2(m_ref, l_run);
                if (threadIdx.x == C::kSoftmaxWarp0 * 32) {
                    sm.ep_b = md.b;
                    sm.ep_h = md.h;
                    sm.ep_split = md.split;
                    sm.ep_nsplit = md.nsplit;
                    sm.ep_end = 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.stat_full);
            }
            ++j;
        }
    } else if (warp >= C::kEpiWarp0 && warp < C::kEpiWarp0 + C::kEpiWarps) {
        // ================================================= epilogue
        // One thread per query row (TMEM lane) streams a finished unit's O
        // out of TMEM while the softmax warps already work on the next unit
        // (O is double-buffered in TMEM).
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int G = a.G;
        const bool live = r < a.M;
        const int jq = live ? r / G : 0;
        const int gi = r - jq * G;
        const int ew = warp - C::kEpiWarp0;
        constexpr int NE = C::kEpiWarps;
        for (int unit = 0;; ++unit) {
            if (!mbar_wait(&sm.stat_full, (uint32_t)(unit & 1), a.err)) break;
            if (sm.ep_end) break;
            const int b = sm.ep_b, h = sm.ep_h, split = sm.ep_split, nsplit = sm.ep_nsplit;
            const float2 st = sm.stat[r];
            const float m_ref = st.x, l_run = st.y;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.stat_empty);
            const int ob = unit & 1;
            if (!mbar_wait(&sm.o_full[ob], par_of(unit), a.err)) break;
            tc_fence_after();
            const uint32_t oa = tmem + kTmemO + (uint32_t)ob * kD + lane_off;
            const int u2 = b * a.Hkv + h;
            const size_t od = (((size_t)b * a.n_q + jq) * a.Hq + (size_t)h * G + gi);
            const size_t pr_own = ((size_t)u2 * a.max_splits + split) * a.M + r;
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            // O row streamed out of TMEM 32 columns at a time: final output
            // when the unit is the whole sequence, else a split partial
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t raw[32];
                tmem_ld32(oa + c * 32, raw);
                tmem_ld_wait();
                if (live) {
                    if (nsplit == 1) {
                        uint4 *orow = reinterpret_cast<uint4 *>(a.out + od * kD + c * 32);
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(raw[c8 * 8 + 0]) * inv, __uint_as_float(raw[c8 * 8 + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(raw[c8 * 8 + 2]) * inv, __uint_as_float(raw[c8 * 8 + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(raw[c8 * 8 + 4]) * inv, __uint_as_float(raw[c8 * 8 + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(raw[c8 * 8 + 6]) * inv, __uint_as_float(raw[c8 * 8 + 7]) * inv);
                            orow[c8] = v;
                        }
                    } else {
                        uint4 *prow4 = reinterpret_cast<uint4 *>(a.part_acc + pr_own * kD + c * 32);
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4)
                            prow4[c4] = make_uint4(raw[c4 * 4], raw[c4 * 4 + 1], raw[c4 * 4 + 2], raw[c4 * 4 + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_empty[ob]);
            if (nsplit == 1) {
                if (live && a.lse) a.lse[od] = (m_ref + __log2f(l_run)) * 0.69314718055994530942f;
                continue;
            }
            if (live) {
                a.part_ml[pr_own * 2] = m_ref;
                a.part_ml[pr_own * 2 + 1] = l_run;
            }
            __threadfence();
            named_barrier_sync(kBarEpi, NE * 32);
            if (ew == 0 && lane == 0) {
                const int t = atomicAdd(&a.tickets[u2], 1);
                sm.last = (t == nsplit - 1);
                if (sm.last) a.tickets[u2] = 0;
            }
            named_barrier_sync(kBarEpi, NE * 32);
            const int last = sm.last;
            named_barrier_sync(kBarEpi, NE * 32);
            if (!last) continue;
            // the last split's CTA merges every split's partial rows with
            // log-sum-exp weights (an online merge: running maximum, rescaled
            // sum): one warp per row, 4 columns per lane, four rows and two
            // splits per pass so that their loads are in flight together
            __threadfence();
            const size_t base = (size_t)u2 * a.max_splits * a.M;
            for (int r0 = ew; r0 < a.M; r0 += 4 * NE) {
                float mrow[4], lrow[4];
                float4 o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    mrow[i] = -CUDART_INF_F;
                    lrow[i] = 0.f;
                    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                for (int s0 = 0; s0 < nsplit; s0 += 2) {
                    float2 ml[4][2];
                    float4 v[4][2];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int rr = r0 + NE * i;
                            if (rr < a.M && s0 + k < nsplit) {
                                const size_t pr = base + (size_t)(s0 + k) * a.M + rr;
                                ml[i][k] = __ldcg(reinterpret_cast<const float2 *>(a.part_ml + pr * 2));
                                v[i][k] = __ldcg(reinterpret_cast<const float4 *>(a.part_acc + pr * kD) + lane);
                            } else {
                                ml[i][k] = make_float2(-CUDART_INF_F, 0.f);
                                v[i][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const float mk = ml[i][k].x;
                            if (mk == -CUDART_INF_F) continue;  // an empty split (or none)
                            const float mn = fmaxf(mrow[i], mk);
                            const float f_old = ex2_approx(mrow[i] - mn);  // 0 when mrow is -inf
                            const float f_new = ex2_approx(mk - mn);
                            lrow[i] = lrow[i] * f_old + ml[i][k].y * f_new;
                            o[i].x = o[i].x * f_old + v[i][k].x * f_new;
                            o[i].y = o[i].y * f_old + v[i][k].y * f_new;
                            o[i].z = o[i].z * f_old + v[i][k].z * f_new;
                            o[i].w = o[i].w * f_old + v[i][k].w * f_new;
                            mrow[i] = mn;
                        }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = r0 + NE * i;
                    if (rr >= a.M) break;
                    const float inv2 = lrow[i] > 0.f ? 1.f / lrow[i] : 0.f;
                    const int jq2 = rr / G, gi2 = rr - jq2 * G;
                    const size_t od2 = (((size_t)b * a.n_q + jq2) * a.Hq + (size_t)h * G + gi2);
                    uint2 v2;
                    v2.x = pack_bf16x2(o[i].x * inv2, o[i].y * inv2);
                    v2.y = pack_bf16x2(o[i].z * inv2, o[i].w * inv2);
                    reinterpret_cast<uint2 *>(a.out + od2 * kD)[lane] = v2;
                    if (lane == 0 && a.lse) a.lse[od2] = (mrow[i] + __log2f(lrow[i])) * 0.69314718055994530942f;
                }
            }
        }
    }
    // every TMEM user is done (the MMA issuer's last operations were waited
    // on by the softmax warps through o_full) before the owner frees it
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {
cudaError_t launch_tc(const CUtensorMap &mk, const CUtensorMap &mv, const AttnMaps &m, const AttnArgs &a, int grid,
                      cudaStream_t st) {
    const size_t smem = sizeof(Smem) + 1024;
    static DeviceMemo<int> attr_set;  // the shared-memory opt-in, once per device
    int done = 0;
    cudaError_t e = attr_set.get(&done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(pva_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    pva_tc_kernel<<<grid, TcCfg::kThreads, smem, st>>>(mk, mv, m.q[0], m.q[1], a);
    return cudaGetLastError();
}
}  // namespace

// bf16 pages: the 5-D page maps (FP8 pages take paged_verify_attn_f8.cu's kernel)
cudaError_t launch_paged_verify_attn_tc(const AttnMaps &m, const AttnArgs &a, int grid, cudaStream_t st) {
    return launch_tc(m.kpage, m.vpage, m, a, grid, st);
}

}  // namespace svpa
