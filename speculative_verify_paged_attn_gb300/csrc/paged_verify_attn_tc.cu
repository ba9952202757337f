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
constexpr int kPage8 = 16 * 128;                // one FP8 (page, kv head) tile
constexpr int kTile8 = kPagesPerBlock * kPage8;  // FP8 K (or V) block: 16 KB
constexpr float kMaxScale8 = 146.f;             // 448 * scale stays below the f16 maximum
constexpr int kTileScales = 16 * (128 / 64);    // tile scales of one (page, kv head): 16 rows x 2

// Two layouts of the same kernel.
//  bf16 pages: warps 0 producer, 1 MMA, 2-5 softmax, 6-9 epilogue; 3-deep K
//    and V rings of bf16 blocks that the MMA reads directly.
//  FP8 pages (at most 64 query rows, so two TMEM lane quadrants): warps 0
//    producer, 1 MMA, 4-5 softmax, 8-9 epilogue, 2/3/10 K converters, 6/7/11
//    V converters; the producer streams E4M3 pages (and, by cp.async, their
//    scales) into 2-deep staging rings, the converters turn each block into
//    f16 (exactly; the K page scale then enters the softmax's exponent and the
//    V page scale multiplies P) in 2-deep K and V tile rings, and the MMAs
//    run kind::f16 with f16 queries (converted in place) and f16 P.  With one
//    scale per 64-element tile of a row (the TILES instantiation) the
//    converters multiply each row-half by its own scale instead.  The
//    query buffer holds 64 rows; the MMA still reads 128, rows 64..127 being
//    whatever follows and feeding only TMEM lanes no thread reads.
template <bool FP8>
struct TcCfg {
    static constexpr int kThreads = FP8 ? 384 : 320;
    static constexpr int kNK = FP8 ? 2 : 3;     // tiles the MMA reads (K freed once S_j is done)
    static constexpr int kNV = FP8 ? 2 : 3;     // (V freed once PV_j is done)
    static constexpr int kNK8 = FP8 ? 2 : 1;    // FP8 staging rings
    static constexpr int kNV8 = FP8 ? 2 : 1;
    static constexpr int kQSlab = (FP8 ? 64 : 128) * 128;  // one 64-column slab of the query buffer
    static constexpr int kQBuf = 2 * kQSlab;
    // arrivals that complete a staging slot: the producer's expect_tx, and on
    // a K slot one cp.async per page for each of its two page scales (K's and
    // V's: the softmax takes both with block j's scores, so it never waits
    // for V's conversion)
    static constexpr uint32_t kStageArrivalsK = 1 + 2 * kPagesPerBlock;
    static constexpr uint32_t kStageArrivalsV = 1;
    static constexpr int kSoftmaxWarp0 = FP8 ? 4 : 2;
    static constexpr int kSoftmaxWarps = FP8 ? 2 : 4;
    static constexpr int kEpiWarp0 = FP8 ? 8 : 6;
    static constexpr int kEpiWarps = FP8 ? 2 : 4;
    static constexpr int kConvWarps = 3;        // per operand (FP8 only)
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

// one scale per 64-element tile of each row of a staged FP8 block (the
// tile-scale instantiation only), one slot per staging slot
struct alignas(16) TileScaleRing {
    float k[TcCfg<true>::kNK8][kPagesPerBlock][kTileScales];
    float v[TcCfg<true>::kNV8][kPagesPerBlock][kTileScales];
};
struct NoTileScales {};

template <bool FP8>
struct Stage8 {  // FP8 staging rings
    uint8_t k8[TcCfg<FP8>::kNK8][kTile8];
    uint8_t v8[TcCfg<FP8>::kNV8][kTile8];
    float ksc[kNMeta][kPagesPerBlock];  // page scales of the blocks in flight
    float vsc[kNMeta][kPagesPerBlock];
    uint64_t k8_full[TcCfg<FP8>::kNK8], k8_empty[TcCfg<FP8>::kNK8];
    uint64_t v8_full[TcCfg<FP8>::kNV8], v8_empty[TcCfg<FP8>::kNV8];
    uint64_t q_full;
};
struct NoStage8 {};

template <bool FP8, bool TILES>
struct Smem {
    using C = TcCfg<FP8>;
    uint8_t q[C::kQBuf];                 // 1024-aligned (one unit's queries)
    uint8_t kbuf[C::kNK][kKVTile];       // 32 KB each
    uint8_t vbuf[C::kNV][kKVTile];
    typename std::conditional<FP8, Stage8<FP8>, NoStage8>::type st8;
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
    // last, so that the other members keep their offsets without tile scales
    typename std::conditional<TILES, TileScaleRing, NoTileScales>::type t64;
};

// fits the 227 KB a CTA may opt into, with room to align the base to 1 KB
static_assert(sizeof(Smem<false, false>) + 1024 <= 232448, "pva_tc_kernel shared memory");
static_assert(sizeof(Smem<true, false>) + 1024 <= 232448, "pva_tc_kernel shared memory");
static_assert(sizeof(Smem<true, true>) + 1024 <= 232448, "pva_tc_kernel shared memory");
using SmemFp8Tiles = Smem<true, true>;
static_assert(offsetof(SmemFp8Tiles, t64) % 16 == 0, "bulk copies land on 16-byte boundaries");

// f16 MMA instruction descriptor (FP8 pages): as umma_idesc_bf16 with both
// operand formats F16.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool b_mn_major) {
    return umma_idesc_bf16(M, N, b_mn_major) & ~((1u << 7) | (1u << 10));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// bf16 pair -> f16 pair (round to nearest)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ uint32_t par_of(int idx) { return (uint32_t)((idx >> 1) & 1); }

// TILES (FP8 only): one scale per 64-element tile of a row, applied by the
// converters, instead of one per (page, kv head) applied in the softmax
template <bool FP8, bool TILES>
__global__ void __launch_bounds__(TcCfg<FP8>::kThreads, 1)
    pva_tc_kernel(const __grid_constant__ CUtensorMap mkp, const __grid_constant__ CUtensorMap mvp,
                  const __grid_constant__ CUtensorMap mq0, const __grid_constant__ CUtensorMap mq1,
                  const __grid_constant__ AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    using C = TcCfg<FP8>;
    constexpr int kNK = C::kNK, kNV = C::kNV, kQSlab = C::kQSlab, kQBuf = C::kQBuf;
    Smem<FP8, TILES> &sm =
        *reinterpret_cast<Smem<FP8, TILES> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        // FP8: the K and V tiles are published by the converter warps
        const uint32_t tile_arrivals = FP8 ? C::kConvWarps : 1;
        for (int i = 0; i < kNK; ++i) {
            mbar_init(&sm.k_full[i], tile_arrivals);
            mbar_init(&sm.k_empty[i], 1);
        }
        for (int i = 0; i < kNV; ++i) {
            mbar_init(&sm.v_full[i], tile_arrivals);
            mbar_init(&sm.v_empty[i], 1);
        }
        if constexpr (FP8) {
            for (int i = 0; i < C::kNK8; ++i) {
                mbar_init(&sm.st8.k8_full[i], C::kStageArrivalsK);
                mbar_init(&sm.st8.k8_empty[i], C::kConvWarps);
            }
            for (int i = 0; i < C::kNV8; ++i) {
                mbar_init(&sm.st8.v8_full[i], C::kStageArrivalsV);
                mbar_init(&sm.st8.v8_empty[i], C::kConvWarps);
            }
            mbar_init(&sm.st8.q_full, 1);
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
        // the rings the copies land in: the MMA's tiles (bf16) or the FP8
        // staging rings in front of the converters
        constexpr int PNK = FP8 ? C::kNK8 : kNK, PNV = FP8 ? C::kNV8 : kNV;
        constexpr uint32_t kBlockBytes = FP8 ? kTile8 : kKVTile;
        uint64_t *pk_full, *pk_empty, *pv_full, *pv_empty;
        if constexpr (FP8) {
            pk_full = sm.st8.k8_full;
            pk_empty = sm.st8.k8_empty;
            pv_full = sm.st8.v8_full;
            pv_empty = sm.st8.v8_empty;
        } else {
            pk_full = sm.k_full;
            pk_empty = sm.k_empty;
            pv_full = sm.v_full;
            pv_empty = sm.v_empty;
        }
        // one copy per page: a 5-D box of a bf16 tile, or a 2 KB FP8 tile
        auto copy_page = [&](const CUtensorMap *map, uint8_t *ring_slot, int id, int hh, uint64_t *bar) {
            if constexpr (FP8)
                tma_load_4d(ring_slot + lane * kPage8, map, 0, 0, hh, id, bar, pol);
            else
                tma_load_5d(ring_slot + lane * 4096, map, 0, 0, 0, 0, id * a.Hkv + hh, bar, pol);
        };
        // FP8: the page's scale by cp.async, counted on the same staging
        // barrier (a missing page takes the block's first page's scale: its
        // bytes are zero)
        auto copy_scale = [&](const float *scales, int id, int hh, float *dst, uint64_t *bar) {
            const int id0 = __shfl_sync(0x000000ffu, id, 0);
            const int sid = (id >= 0 && id < a.num_blocks) ? id : id0;
            cp_async_4(dst, scales + (size_t)sid * a.Hkv + hh);
            cp_async_mbar_arrive_noinc(bar);
        };
        // tile scales: the page's 32 tile scales (128 bytes) by a bulk copy,
        // counted in the staging barrier's bytes, into staging slot `slot`
        auto copy_tile_scales = [&](const float *scales, int id, int hh, float *dst, uint64_t *bar) {
            const int id0 = __shfl_sync(0x000000ffu, id, 0);
            const int sid = (id >= 0 && id < a.num_blocks) ? id : id0;
            bulk_copy_g2s(dst, scales + ((size_t)sid * a.Hkv + hh) * kTileScales, kTileScales * 4, bar);
        };
        constexpr uint32_t tile_bytes = TILES ? kPagesPerBlock * kTileScales * 4 : 0u;
        auto k_slot = [&](int s_) -> uint8_t * {
            if constexpr (FP8) return sm.st8.k8[s_]; else return sm.kbuf[s_];
        };
        auto v_slot = [&](int s_) -> uint8_t * {
            if constexpr (FP8) return sm.st8.v8[s_]; else return sm.vbuf[s_];
        };
        // V of the oldest block whose K is out, if its ring slot is free (a
        // non-blocking test): K runs ahead as far as its own ring allows and
        // V follows as PV frees slots, neither waiting for the other
        auto try_issue_v = [&]() -> bool {
            if (jv >= jk) return false;
            const int vs = jv % PNV;
            int ready = 1;
            if (lane == 0 && jv >= PNV) ready = mbar_test(&pv_empty[vs], (uint32_t)(((jv / PNV) & 1) ^ 1));
            if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
            if (lane == 0) mbar_arrive_expect_tx(&pv_full[vs], kBlockBytes + tile_bytes);
            if (lane < kPagesPerBlock) {
                const int id = sm.vid[jv % kNMeta][lane], hh = sm.meta[jv % kNMeta].h;
                copy_page(&mvp, v_slot(vs), id, hh, &pv_full[vs]);
                if constexpr (TILES) copy_tile_scales(a.v_scale, id, hh, sm.t64.v[vs][lane], &pv_full[vs]);
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
                        // bf16: the query tile rides on the unit's first K block;
                        // FP8: it has a barrier of its own (the converters
                        // turn it into f16 before the first K tile)
                        uint64_t *qbar = &pk_full[ks];
                        if constexpr (FP8) qbar = &sm.st8.q_full;
                        if (FP8 && bi == 0) mbar_arrive_expect_tx(qbar, qbytes);
                        mbar_arrive_expect_tx(&pk_full[ks], kBlockBytes + tile_bytes + (!FP8 && bi == 0 ? qbytes : 0u));
                        if (bi == 0) {
                            tma_load_4d(&sm.q[0], &mq0, 0, h * a.G, 0, b, qbar, pol);
                            tma_load_4d(&sm.q[kQSlab], &mq1, 0, h * a.G, 0, b, qbar, pol);
                        }
                    }
                    if (lane < kPagesPerBlock) {
                        sm.vid[jk % kNMeta][lane] = my_id;
                        copy_page(&mkp, k_slot(ks), my_id, h, &pk_full[ks]);
                        if constexpr (FP8) {
                            copy_scale(a.k_scale, my_id, h, &sm.st8.ksc[jk % kNMeta][lane], &pk_full[ks]);
                            copy_scale(a.v_scale, my_id, h, &sm.st8.vsc[jk % kNMeta][lane], &pk_full[ks]);
                        }
                        if constexpr (TILES)
                            copy_tile_scales(a.k_scale, my_id, h, sm.t64.k[ks][lane], &pk_full[ks]);
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
            // end-of-work marker on the K ring (and, FP8, on the V staging
            // ring for the V converters)
            const int ks = jk % PNK;
            if (ok && jk >= PNK) ok = mbar_wait(&pk_empty[ks], (uint32_t)(((jk / PNK) & 1) ^ 1), a.err);
            if (ok) {
                sm.meta[jk % kNMeta].flags = kFlagEnd;
                mbar_arrive_cnt(&pk_full[ks], FP8 ? C::kStageArrivalsK : 1u);
            }
            const int vs = jv % PNV;
            if constexpr (FP8) {
                if (ok && jv >= PNV) ok = mbar_wait(&pv_empty[vs], (uint32_t)(((jv / PNV) & 1) ^ 1), a.err);
                if (ok) mbar_arrive_cnt(&pv_full[vs], C::kStageArrivalsV);
            }
            // wait (bounded) for the copies still in flight; a stage reused
            // by an end marker had completed before its empty barrier passed
            for (int i = jk >= PNK ? jk - PNK + 1 : 0; i < jk && ok; ++i)
                ok = mbar_wait(&pk_full[i % PNK], (uint32_t)((i / PNK) & 1), a.err);
            for (int i = jv >= PNV ? jv - PNV + (FP8 ? 1 : 0) : 0; i < jv && ok; ++i)
                ok = mbar_wait(&pv_full[i % PNV], (uint32_t)((i / PNV) & 1), a.err);
            if constexpr (FP8)
                if (ok && units >= 1) ok = mbar_wait(&sm.st8.q_full, (uint32_t)((units - 1) & 1), a.err);
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
            constexpr uint32_t idS = FP8 ? umma_idesc_f16(kRows, kNB, false) : umma_idesc_bf16(kRows, kNB, false);
            constexpr uint32_t idPV = FP8 ? umma_idesc_f16(kRows, kD, true) : umma_idesc_bf16(kRows, kD, true);
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
                if constexpr (FP8) {
                    // the block's four 32-column loads issued back to back, one
                    // wait (the FP8 softmax is the critical path)
                    uint32_t raw[kNB / 32][32];
#pragma unroll
                    for (int c = 0; c < kNB / 32; ++c) tmem_ld32(sa + c * 32, raw[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < kNB / 32; ++c)
#pragma unroll
                        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(raw[c][t]);
                } else {
#pragma unroll
                    for (int c = 0; c < kNB / 32; ++c) {
                        uint32_t raw[32];
                        tmem_ld32(sa + c * 32, raw);
                        tmem_ld_wait();
#pragma unroll
                        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(raw[t]);
                    }
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
            // per-page maxima of the raw scores (FP8: a page's K scale
            // multiplies its scores; scales are >= 0, so the maximum of the
            // scaled scores is the largest scaled page maximum)
            float pm[kPagesPerBlock];
#pragma unroll
            for (int x = 0; x < kPagesPerBlock; ++x) pm[x] = s[16 * x];
#pragma unroll
            for (int t = 0; t < kNB; ++t)
                if (t & 15) pm[t >> 4] = fmaxf(pm[t >> 4], s[t]);
            float ksc[kPagesPerBlock], vsc[kPagesPerBlock];
            if constexpr (FP8) {
#pragma unroll
                for (int x = 0; x < kPagesPerBlock; ++x) {
                    // (tile scales are already in the converted tiles)
                    ksc[x] = TILES ? 1.f : sm.st8.ksc[j % kNMeta][x];
                    vsc[x] = TILES ? 1.f : sm.st8.vsc[j % kNMeta][x];
                    if (pm[x] != -CUDART_INF_F) pm[x] *= ksc[x];
                }
            }
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
            // (FP8: V_j's page scales, which multiply P, came with K_j's
            // staging, which S_j's completion follows)
            // P_j as bf16 pairs into the first half of S_j's TMEM columns
            const uint32_t pt = tmem + kTmemS + (uint32_t)(j & 1) * kNB + lane_off;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (FP8) {
                // FP8 pages: P is f16, so each pair of exponents is evaluated by
                // one ex2.f16x2 on the fp32 arguments rounded to f16 (an argument
                // is at most 8 under the lazy maximum, where f16 keeps P within
                // ~0.14%); the row sum adds those f16 values, in f16 within a
                // page (16 values) and in fp32 across pages; P times the V page
                // scale is formed in f16.  A page whose K scale is 0 has scores
                // 0: its multiplier stays positive so masked columns stay -inf.
#pragma unroll
                for (int c = 0; c < kNB / 64; ++c) {
                    uint32_t w[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int pg = c * 4 + q;  // the page of these 16 columns
                        const float scp = fmaxf(sc * ksc[pg], 1e-30f);
                        const uint32_t v2 = pack_f16x2(vsc[pg], vsc[pg]);
                        uint32_t acc = 0u;  // f16 pair (+0, +0)
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) {
                            const int e = q * 8 + e8;
                            const float x0 = live ? fmaf(s[c * 64 + 2 * e], scp, neg_m) : -CUDART_INF_F;
                            const float x1 = live ? fmaf(s[c * 64 + 2 * e + 1], scp, neg_m) : -CUDART_INF_F;
                            const uint32_t p2 = ex2_f16x2(pack_f16x2(x0, x1));
                            acc = add_f16x2(acc, p2);
                            w[e] = mul_f16x2(p2, v2);
                        }
                        const float2 f = f16x2_to_float2(acc);
                        ls[q] += f.x + f.y;
                    }
                    tmem_st32(pt + c * 32, w);
                }
            } else {
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
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // V rows past the sequence's last token may hold anything: zero
            // them once V_j has landed (PV_j is not issued before p_full)
            if (!FP8 && md.pos0 + md.ntok > T) {  // (FP8: the V converters zero them)
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
    if constexpr (FP8) {
        const bool kconv = warp == 2 || warp == 3 || warp == 10;
        const bool vconv = warp == 6 || warp == 7 || warp == 11;
        if (kconv || vconv) {
            // ================================================= FP8 converters
            // Block j's E4M3 pages -> one f16 tile in the MMA's layout (page p
            // at p * 4 KB as [row half][slab][8 rows][128 B], 128-byte
            // swizzle), each value times its page's scale; the V converters
            // also zero the rows past the sequence's last token.  The K
            // converters first turn each unit's bf16 query tile into f16.
            const int ci = kconv ? (warp == 10 ? 2 : warp - 2) : (warp == 11 ? 2 : warp - 6);
            const int ct = ci * 32 + lane;  // 0..95
            constexpr int NCT = C::kConvWarps * 32;
            const int ring = kconv ? C::kNK8 : C::kNV8;
            const int tiles = kconv ? kNK : kNV;
            uint64_t *full8 = kconv ? sm.st8.k8_full : sm.st8.v8_full;
            uint64_t *empty8 = kconv ? sm.st8.k8_empty : sm.st8.v8_empty;
            int units_seen = 0;
            for (int j = 0;; ++j) {
                const int s8 = j % ring, tb = j % tiles;
                if (!mbar_wait(&full8[s8], (uint32_t)((j / ring) & 1), a.err)) break;
                const BlockMeta md = sm.meta[j % kNMeta];
                uint64_t *tile_full = kconv ? &sm.k_full[tb] : &sm.v_full[tb];
                uint64_t *tile_empty = kconv ? &sm.k_empty[tb] : &sm.v_empty[tb];
                // the tile is free once S (K) or PV (V) of block j - tiles is done
                if (j >= tiles && !mbar_wait(tile_empty, (uint32_t)(((j / tiles) & 1) ^ 1), a.err)) break;
                if (md.flags & kFlagEnd) {
                    // forward the end marker to the MMA issuer
                    __syncwarp();
                    if (kconv && lane == 0) mbar_arrive(tile_full);
                    break;
                }
                const uint8_t *src = kconv ? sm.st8.k8[s8] : sm.st8.v8[s8];
                uint8_t *tile = kconv ? sm.kbuf[tb] : sm.vbuf[tb];
                // both page scales of the block came with its K staging slot
                if (kconv && lane < kPagesPerBlock) {
                    const float ks = sm.st8.ksc[j % kNMeta][lane], vs = sm.st8.vsc[j % kNMeta][lane];
                    if (!(ks >= 0.f && ks <= kMaxScale8) || !(vs >= 0.f && vs <= kMaxScale8))
                        raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                }
                if (kconv && (md.flags & kFlagFirst)) {
                    // the unit's queries, bf16 -> f16 in place (rows < M)
                    if (!mbar_wait(&sm.st8.q_full, (uint32_t)(units_seen & 1), a.err)) break;
                    ++units_seen;
                    for (int i = ct; i < a.M * 16; i += NCT) {
                        const int row = i >> 4, c = i & 15;
                        uint4 *qp = reinterpret_cast<uint4 *>(&sm.q[(c >> 3) * kQSlab + row * 128 + ((c & 7) << 4)]);
                        uint4 v = *qp;
                        v.x = bf16x2_to_f16x2(v.x);
                        v.y = bf16x2_to_f16x2(v.y);
                        v.z = bf16x2_to_f16x2(v.z);
                        v.w = bf16x2_to_f16x2(v.w);
                        *qp = v;
                    }
                }
                const int t_end = kconv ? kNB : md.L + a.n_q - md.pos0;  // V rows from t_end on are zeroed
                // item i: row i / 8, 16 columns 16 (i % 8) ..; four items in flight per thread
                constexpr int kItems = kNB * 8, kPer = (kItems + NCT - 1) / NCT;
#pragma unroll 1
                for (int t0 = 0; t0 < kPer; t0 += 4) {
                    uint4 e[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = ct + NCT * (t0 + u), row = i >> 3, g = i & 7;
                        e[u] = make_uint4(0, 0, 0, 0);
                        if (t0 + u < kPer && i < kItems && row < t_end)
                            e[u] = *reinterpret_cast<const uint4 *>(src + row * 128 + ((g ^ (row & 7)) << 4));
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = ct + NCT * (t0 + u), row = i >> 3, g = i & 7;
                        if (t0 + u >= kPer || i >= kItems) continue;
                        uint4 lo, hi;
                        lo.x = e4m3x2_to_f16x2(e[u].x & 0xffffu);
                        lo.y = e4m3x2_to_f16x2(e[u].x >> 16);
                        lo.z = e4m3x2_to_f16x2(e[u].y & 0xffffu);
                        lo.w = e4m3x2_to_f16x2(e[u].y >> 16);
                        hi.x = e4m3x2_to_f16x2(e[u].z & 0xffffu);
                        hi.y = e4m3x2_to_f16x2(e[u].z >> 16);
                        hi.z = e4m3x2_to_f16x2(e[u].w & 0xffffu);
                        hi.w = e4m3x2_to_f16x2(e[u].w >> 16);
                        if constexpr (TILES) {
                          if (row < md.L + a.n_q - md.pos0) {
                            // this group's 64-element tile: (page, slot, half) of the block;
                            // rows past the last token keep unscaled bytes (their scales
                            // need not be set: K columns there are masked, V rows zeroed)
                            const float tsc = (kconv ? sm.t64.k[s8] : sm.t64.v[s8])[row >> 4][(row & 15) * 2 + (g >> 2)];
                            if (!(tsc >= 0.f && tsc <= kMaxScale8)) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                            const uint32_t t2 = pack_f16x2(tsc, tsc);
                            lo.x = mul_f16x2(lo.x, t2);
                            lo.y = mul_f16x2(lo.y, t2);
                            lo.z = mul_f16x2(lo.z, t2);
                            lo.w = mul_f16x2(lo.w, t2);
                            hi.x = mul_f16x2(hi.x, t2);
                            hi.y = mul_f16x2(hi.y, t2);
                            hi.z = mul_f16x2(hi.z, t2);
                            hi.w = mul_f16x2(hi.w, t2);
                          }
                        }
                        const int r8 = row & 7, c0 = (g & 3) * 2;
                        uint8_t *dst = tile + (row >> 3) * 2048 + (g >> 2) * 1024 + r8 * 128;
                        *reinterpret_cast<uint4 *>(dst + ((c0 ^ r8) << 4)) = lo;
                        *reinterpret_cast<uint4 *>(dst + (((c0 + 1) ^ r8) << 4)) = hi;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(tile_full);
                    mbar_arrive(&empty8[s8]);
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

size_t attn_tc_smem_bytes() {
    return std::max(sizeof(Smem<false, false>), std::max(sizeof(Smem<true, false>), sizeof(Smem<true, true>))) + 1024;
}

namespace {
template <bool FP8, bool TILES>
cudaError_t launch_tc(const CUtensorMap &mk, const CUtensorMap &mv, const AttnMaps &m, const AttnArgs &a, int grid,
                      cudaStream_t st) {
    const size_t smem = sizeof(Smem<FP8, TILES>) + 1024;
    static DeviceMemo<int> attr_set;  // the shared-memory opt-in, once per device
    int done = 0;
    cudaError_t e = attr_set.get(&done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(pva_tc_kernel<FP8, TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    pva_tc_kernel<FP8, TILES><<<grid, TcCfg<FP8>::kThreads, smem, st>>>(mk, mv, m.q[0], m.q[1], a);
    return cudaGetLastError();
}
}  // namespace

// FP8 pages: the E4M3 page maps (one 2 KB box per page); bf16: the 5-D page maps
cudaError_t launch_paged_verify_attn_tc(const AttnMaps &m, const AttnArgs &a, int grid, bool fp8, cudaStream_t st) {
    if (!fp8) return launch_tc<false, false>(m.kpage, m.vpage, m, a, grid, st);
    // (FP8 pages with one scale per page take paged_verify_attn_f8.cu's kernel)
    if (!a.scale_tile) return cudaErrorInvalidValue;
    return launch_tc<true, true>(m.k[0], m.v[0], m, a, grid, st);
}

}  // namespace svpa
