// paged_verify_attn_f8.cu -- paged verification attention over FP8-E4M3
// pages with one scale per (page, kv head), on the 5th-generation tensor
// cores (tcgen05 + TMEM) for sm_103a, for up to 64 query rows per kv head
// (grouped-query models: G * n_q <= 64).
//
// Same computation as paged_verify_attn.cu ("The Sub-Millisecond Speculative
// Decoding Meltdown", section "Speculative Decoding Mechanics & The K-Token
// Penalty": A = softmax(Q K^T * scale + M_tree) V over a paged K/V history;
// "Custom FP8 Quantized Memory Block Layout": E4M3 pages with per-block
// scales; "Triton CUDA Fused Speculative Tree-Verification Kernel": per-page
// block lookup, K/V cache [blocks, heads, 16, dim], K/V scales [blocks,
// heads], running max / sum).
//
// Scores: S = Q K^T by tcgen05.mma kind::f8f6f4 straight on the staged E4M3
// K pages (no conversion of K).  Each query row is split into two E4M3 terms
// at a power-of-two scale of its own, q * 2^e = hi + lo (hi = the row rounded
// to E4M3, lo = the remainder rounded to E4M3), and both terms accumulate
// into one fp32 TMEM tile: the scores carry ~8 significant bits of each
// query value, as many as its bf16 input.  The softmax multiplies a row's
// scores by 2^-e, the page's K scale and sm_scale * log2(e) in one factor.
// P V: kind::f16, with V converted exactly to f16 by converter warps and P
// in f16 (P times the page's V scale), accumulating into fp32 TMEM.
//
// Work: the 128-token blocks of all (sequence, kv head) pairs, in that order,
// split evenly over one persistent CTA per SM (a per-sequence block prefix,
// computed by a small kernel just before, locates a CTA's share); a pair cut
// by a share boundary is processed in pieces whose partial results the last
// piece's CTA merges with log-sum-exp weights.
// 16 warps; a warp reads the TMEM lanes of quadrant warp % 4 only, and the
// query rows live in quadrants 0 and 1, so the row-owning warps sit on SM
// sub-partitions 0 and 1 and everything else on 2 and 3:
//   warps 0,1 / 4,5 / 8,9 / 12,13
//                   softmax and epilogue: warp w owns the rows of lane
//                   quadrant w % 4 and the block's tokens 32 (w / 4) .. + 31;
//                   the four warps of a quadrant exchange their block maxima
//                   through shared memory (a bounded mbarrier wait), so that
//                   all keep one lazy reference maximum per row, and at a
//                   unit's end their partial row sums, then write their 32
//                   columns of O (the output, or a piece's partial; the last
//                   piece of a (sequence, kv head) merges the pieces);
//   warp 2          producer: walks the CTA's share; each piece's bf16
//                   query tile into one of two query slots; per 128-token
//                   block, 8 E4M3 K page tiles (TMA, 128-byte swizzle) and
//                   both page scales (cp.async) into a 4-deep K ring that the
//                   MMA reads directly, and the V page tiles into a 3-deep
//                   staging ring;
//   warp 3          P V issuer (one thread) and TMEM owner: O += P_j V_j with
//                   P_j read from TMEM, once P_j is published and V_j converted;
//   warp 14         score issuer (one thread): S_j into one of two TMEM S
//                   buffers as soon as K_j, the unit's split queries and the
//                   buffer are ready (two issuing threads, so that neither
//                   chain of waits and issues holds up the other);
//   warps 6,7,10,11 V converters: E4M3 -> f16 (exact) in the MMA's tile
//                   layout, rows past the sequence's end zeroed;
//   warp 15         query split: each thread turns two landed bf16 query
//                   rows into their two E4M3 terms in place and records
//                   their scales.
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
constexpr int kPB = 8;                      // pages per block
constexpr int kNB = kPB * 16;               // tokens per block
constexpr int kRows = 128;                  // MMA M
constexpr int kPage8 = 16 * 128;            // one E4M3 (page, kv head) tile
constexpr int kTile8 = kPB * kPage8;        // E4M3 block: 16 KB
constexpr int kTile16 = kNB * kD * 2;       // f16 V block: 32 KB
constexpr int kNV8 = 3;                     // V staging ring
constexpr int kNV = 2;                      // f16 V tiles (tile j & 1; freed by P V_j's p_free signal)
constexpr int kNMeta = 8;                   // block descriptors in flight
constexpr int kQSlab = 64 * 128;            // one 128-byte column slab of 64 query rows
constexpr int kQSlot = 2 * kQSlab;          // one unit's queries (bf16, then the two E4M3 terms)
constexpr int kNQScale = 4;                 // query-scale records in flight
constexpr int kThreads = 512;
constexpr int kProducerWarp = 2;
constexpr int kMmaWarp = 3;                 // P V issuer, TMEM owner
constexpr int kSWarp = 14;                  // score MMA issuer
constexpr int kSoftWarps = 8;               // 0, 1, 4, 5, 8, 9, 12, 13 (warp % 4 = quadrant, warp / 4 = column slot)
constexpr int kConvWarps = 4;               // 6, 7, 10, 11
constexpr int kPrepWarp = 15;               // query split
// P (at most 2^8 under the lazy maximum) times a V scale stays below the f16
// maximum 65504
constexpr float kMaxVScale8 = 255.f;
// V tile scales times 448 stay below the f16 maximum (V is converted to f16
// with its tile scales)
constexpr float kMaxTileScale8 = 146.f;
constexpr int kTileScales = 16 * 2;         // tile scales of one (page, kv head): 16 rows x 2 halves
constexpr float kRescaleLog2 = 8.f;         // rescale O when a maximum grows by > 2^8
// TMEM columns: O 0..127 (one buffer: the epilogue drains a unit's O before
// the next unit's first P V), S[0] 128..255, S[1] 256..383, P[0] 384..447,
// P[1] 448..511 (P of block j as f16 pairs in P[j & 1], apart from S so that
// a softmax warp may read its S columns again while others write P)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS = 128, kTmemP = 384;
constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagEnd = 4;

struct BlockMeta {
    int32_t b, h, split, pos0, ntok, L, nsplit, flags;
    int32_t slot;  // the piece's partial-result slot (2 * CTA + 0 for its first piece, + 1 for its last)
    int32_t pad[3];
};

// TILES: one scale per 64-element tile of a row (K and V) instead of one per
// (page, kv head)
template <bool TILES>
struct F8Cfg {
    static constexpr int kNK8 = TILES ? 3 : 4;  // K ring (read by the MMA)
    // arrivals that complete a K ring slot: the producer's expect_tx and, with
    // per-page scales, one cp.async arrival per page for each of its two page
    // scales (tile scales come by bulk copies counted in the slot's bytes)
    static constexpr uint32_t kStageArrivalsK = TILES ? 1 : 1 + 2 * kPB;
};

// tile scales of the blocks in flight: K's by block (the softmax applies them
// to the scores), V's by staging slot (the converters apply them)
struct alignas(16) TileScalesF8 {
    float k[kNMeta][kPB][kTileScales];
    float v[kNV8][kPB][kTileScales];
};
struct NoTileScalesF8 {};

template <bool TILES>
struct SmemF8 {
    using C = F8Cfg<TILES>;
    uint8_t q[2][kQSlot];                    // 1024-aligned query slots
    uint8_t k8[C::kNK8][kTile8];
    uint8_t v8[kNV8][kTile8];
    uint8_t vbuf[kNV][kTile16];
    float ksc[kNMeta][kPB];                   // page scales of the blocks in flight
    float vsc[kNMeta][kPB];
    float qscale[kNQScale][64];               // 2^-e of each query row, per unit in flight
    float xmax[2][2][4][32];                  // [quadrant][block parity][column slot][lane]
    float lsum[2][4][32];                     // [quadrant][column slot][lane]: partial row sums at a unit's end
    uint64_t k8_full[C::kNK8], k8_empty[C::kNK8];
    uint64_t v8_full[kNV8], v8_empty[kNV8];
    uint64_t v_full[kNV];
    uint64_t q_full[2], q_ready[2], q_empty[2];
    uint64_t s_full[2];
    uint64_t p_full[2];                       // P_j published (p_full[j & 1])
    // P V_j done (its commit arrives on p_free[j & 1]): P[j & 1], the f16 V
    // tile j & 1 and O's P V_j contribution are then free / complete
    uint64_t p_free[2];
    uint64_t o_full, o_empty;
    uint64_t lbar[2];                         // the quadrant's partial row sums exchanged
    uint64_t gbar;                            // the eight softmax warps (split pieces' ticket)
    uint64_t xbar[2][2];                      // [quadrant][block parity]
    uint64_t s_read;                          // TILES: the softmax has read S (one S buffer)
    BlockMeta meta[kNMeta];
    int32_t vid[kNMeta][kPB];                 // page ids of a block, for its V copies
    int32_t q_is_end[2];                      // the producer's end marker on a query slot
    uint32_t tmem_base;
    int32_t last;
    typename std::conditional<TILES, TileScalesF8, NoTileScalesF8>::type t64;
};

static_assert(sizeof(SmemF8<false>) + 1024 <= 232448, "pva_f8_kernel shared memory");
static_assert(sizeof(SmemF8<true>) + 1024 <= 232448, "pva_f8_kernel shared memory");
static_assert(offsetof(SmemF8<false>, k8) % 1024 == 0 && offsetof(SmemF8<false>, v8) % 1024 == 0 &&
                  offsetof(SmemF8<false>, vbuf) % 1024 == 0 && offsetof(SmemF8<true>, v8) % 1024 == 0 &&
                  offsetof(SmemF8<true>, vbuf) % 1024 == 0,
              "swizzled tiles start on 1024-byte boundaries");
static_assert(offsetof(SmemF8<true>, t64) % 16 == 0, "bulk copies land on 16-byte boundaries");

// Instruction descriptors: fp32 D; kind::f8f6f4 with A and B E4M3, both
// K-major; kind::f16 with A and B f16, B MN-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_f16_bmn(int M, int N) {
    return umma_idesc_bf16(M, N, true) & ~((1u << 7) | (1u << 10));
}

__device__ __forceinline__ void umma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ uint32_t par_of(int idx) { return (uint32_t)((idx >> 1) & 1); }

// Bounded wait for phase `parity` of `bar` in which the waiting thread stays
// suspended (up to kSuspendNs per probe) until the phase completes, instead
// of probing in a loop: the waiting warps leave their scheduler's issue slots
// to the warps that work.  Returns false (and raises SVPA_DEVERR_TIMEOUT)
// after kWaitLimitNs of wall time.
constexpr uint32_t kSuspendNs = 100000;
__device__ __forceinline__ bool try_wait_suspend(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, int32_t *err) {
    if (try_wait_suspend(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (try_wait_suspend(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            raise_error(err, SVPA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// two fp32 values -> two E4M3 codes (round to nearest, saturating), lo in the low byte
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}

// The producer's V copies: V of the oldest block whose K is out, if its
// staging slot is free (a non-blocking test); warp-collective.
template <bool TILES>
__device__ __forceinline__ bool producer_try_issue_v(SmemF8<TILES> &sm, const CUtensorMap *mvp, const float *v_scale,
                                                     int num_blocks, int Hkv, uint64_t pol, int &jv, int jk) {
    const int lane = threadIdx.x & 31;
    if (jv >= jk) return false;
    const int vs = jv % kNV8;
    int ready = 1;
    if (lane == 0 && jv >= kNV8) ready = mbar_test(&sm.v8_empty[vs], (uint32_t)(((jv / kNV8) & 1) ^ 1));
    if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
    if (lane == 0) mbar_arrive_expect_tx(&sm.v8_full[vs], kTile8 + (TILES ? kPB * kTileScales * 4 : 0u));
    if (lane < kPB) {
        const int id = sm.vid[jv % kNMeta][lane], hh = sm.meta[jv % kNMeta].h;
        tma_load_4d(sm.v8[vs] + lane * kPage8, mvp, 0, 0, hh, id, &sm.v8_full[vs], pol);
        if constexpr (TILES) {
            // the page's 32 tile scales (a missing page takes the block's
            // first page's: its bytes are zero)
            const int id0 = __shfl_sync(0x000000ffu, id, 0);
            const int sid = (id >= 0 && id < num_blocks) ? id : id0;
            bulk_copy_g2s(sm.t64.v[vs][lane], v_scale + ((size_t)sid * Hkv + hh) * kTileScales, kTileScales * 4,
                          &sm.v8_full[vs]);
        }
    }
    __syncwarp();
    ++jv;
    return true;
}

// Bounded wait (warp-collective) for phase `parity` of `bar`, issuing V
// copies meanwhile.
template <bool TILES>
__device__ __forceinline__ bool producer_wait_issuing_v(SmemF8<TILES> &sm, const CUtensorMap *mvp,
                                                        const float *v_scale, int num_blocks, int Hkv, uint64_t pol,
                                                        int &jv, int jk, uint64_t *bar, uint32_t parity,
                                                        int32_t *err) {
    const int lane = threadIdx.x & 31;
    unsigned long long t0 = 0;
    while (true) {
        int done = 0;
        if (lane == 0) done = mbar_test(bar, parity);
        if (__shfl_sync(0xffffffffu, done, 0)) return true;
        if (producer_try_issue_v<TILES>(sm, mvp, v_scale, num_blocks, Hkv, pol, jv, jk)) {
            t0 = 0;
            continue;
        }
        // nothing to do yet: back off, leaving the issue slots to the
        // converter warps that share this scheduler
        __nanosleep(64);
        const unsigned long long now = global_ns();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > kWaitLimitNs) {
            if (lane == 0) raise_error(err, SVPA_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// The score issuer's S_jj = (Q_hi + Q_lo) K_jj^T once K_jj has landed, its
// TMEM buffer is free and, on a unit's first block, its queries are split (or
// the end marker forwarded).  Per-page scales: S_jj's buffer held S_{jj-2},
// which the softmax has read once it published P_{jj-2} (p_full[jj & 1]; P_jj
// cannot be published before S_jj, so the parity is unambiguous).  Tile
// scales: the one buffer, read for S_{jj-1} (s_read).  The buffer is waited
// for before the end marker too, so that the softmax never sees s_full two
// phases ahead.
template <bool TILES>
__device__ __forceinline__ bool mma_issue_s(SmemF8<TILES> &sm, int32_t *err, uint32_t tmem, int jj, int &unit_jj,
                                         BlockMeta &m) {
    constexpr uint32_t idS = idesc_e4m3(kRows, kNB);
    constexpr int NK8 = F8Cfg<TILES>::kNK8;
    const int ks = jj % NK8;
    if (!wait_phase(&sm.k8_full[ks], (uint32_t)((jj / NK8) & 1), err)) return false;
    m = sm.meta[jj % kNMeta];
    if (TILES && jj >= 1 && !wait_phase(&sm.s_read, (uint32_t)((jj - 1) & 1), err)) return false;
    if (!TILES && jj >= 2 && !wait_phase(&sm.p_full[jj & 1], par_of(jj - 2), err)) return false;
    if (m.flags & kFlagEnd) {
        mbar_arrive(&sm.s_full[jj & 1]);
        return true;
    }
    if (m.flags & kFlagFirst) {
        ++unit_jj;
        if (!wait_phase(&sm.q_ready[unit_jj & 1], par_of(unit_jj), err)) return false;
    }
    tc_fence_after();
    const uint32_t dS = tmem + kTmemS + (TILES ? 0u : (uint32_t)(jj & 1) * kNB);
    // two query terms x four 32-byte K steps, one accumulation; TILES: the
    // head dimensions 0-63 (K steps 0, 1) into S0 and 64-127 into S1, the
    // tile scales of a token's two halves being applied by the softmax
    const uint32_t qa = smem_u32(sm.q[unit_jj & 1]);
    const uint32_t ka = smem_u32(sm.k8[ks]);
#pragma unroll
    for (int step = 0; step < 8; ++step) {
        const int term = step >> 2, kk = step & 3;
        const uint64_t ad = umma_desc_sw128(qa + term * kQSlab + kk * 32, 16, 1024);
        const uint64_t bd = umma_desc_sw128(ka + kk * 32, 16, 1024);
        if constexpr (TILES)
            umma_e4m3(dS + (uint32_t)(kk >> 1) * kNB, ad, bd, idS, (term | (kk & 1)) ? 1u : 0u);
        else
            umma_e4m3(dS, ad, bd, idS, step > 0 ? 1u : 0u);
    }
    umma_commit(&sm.k8_empty[ks]);
    umma_commit(&sm.s_full[jj & 1]);
    if (m.flags & kFlagLast) umma_commit(&sm.q_empty[unit_jj & 1]);
    return true;
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// A barrier of the eight softmax warps on an mbarrier: every one of them
// calls it at the same points in the same order; `phase` (a per-thread
// counter) numbers those points.  Bounded: false (and SVPA_DEVERR_TIMEOUT)
// when the wait runs out, after which the caller leaves its loop.
__device__ __forceinline__ bool soft_sync(uint64_t *bar, uint32_t &phase, int32_t *err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = wait_phase(bar, phase & 1u, err);
    ++phase;
    return ok;
}

// The softmax, and the epilogue, of one (lane quadrant, column slot): the
// rows of quadrant `quarter` (TMEM lanes), the 32 columns 32 sl .. of every
// block (pages 2 sl, 2 sl + 1).  The eight warps share this one body and its
// code is kept small (one 32-column chunk per block, nothing unrolled twice):
// every role's hot loop must stay in its SM sub-partition's instruction cache.
template <bool TILES>
__device__ __noinline__ void softmax_role(SmemF8<TILES> &sm, const AttnArgs &a, uint32_t tmem, int quarter, int sl) {
    const int lane = threadIdx.x & 31;
    const int r = quarter * 32 + lane;  // query row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int G = a.G;
    const bool live = r < a.M;
    const int jq = live ? r / G : 0;
    const int gi = r - jq * G;
    const unsigned long long anc = live ? a.anc[jq] : 0ull;
    const int pg0 = 2 * sl, tok0 = 32 * sl;
    float m_ref = -CUDART_INF_F, l_run = 0.f, rowmul = 0.f;
    uint32_t gph = 0;  // soft_sync phases passed
    int j = 0, unit = -1;
    while (true) {
        if (!wait_phase(&sm.s_full[j & 1], par_of(j), a.err)) break;
        const BlockMeta md = sm.meta[j % kNMeta];
        if (md.flags & kFlagEnd) {
            // the end marker, forwarded to the P V issuer on p_full[j & 1] once
            // P V_{j-2} is done (so that p_full is never two phases ahead of it)
            if (j >= 2) wait_phase(&sm.p_free[j & 1], par_of(j - 2), a.err);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[j & 1]);
            break;
        }
        const bool first = (md.flags & kFlagFirst) != 0;
        if (first) {
            ++unit;
            m_ref = -CUDART_INF_F;
            l_run = 0.f;
            rowmul = a.scale_log2 * sm.qscale[unit % kNQScale][r];
        }
        tc_fence_after();
        const uint32_t sa = tmem + kTmemS + (TILES ? 0u : (uint32_t)(j & 1) * kNB) + lane_off + (uint32_t)tok0;
        // the page scales of this slot's pages came with K_j's staging, which
        // S_j's completion follows (with tile scales the V scales are in the
        // converted V and the K scales multiply the two halves' scores below)
        float ka = 1.f, kb = 1.f, va = 1.f, vb = 1.f;
        if constexpr (!TILES) {
            ka = sm.ksc[j % kNMeta][pg0];
            kb = sm.ksc[j % kNMeta][pg0 + 1];
            va = sm.vsc[j % kNMeta][pg0];
            vb = sm.vsc[j % kNMeta][pg0 + 1];
            if (quarter == 0 && lane == 0 &&
                (!(ka >= 0.f && ka <= 3.0e38f) || !(kb >= 0.f && kb <= 3.0e38f) ||
                 !(va >= 0.f && va <= kMaxVScale8) || !(vb >= 0.f && vb <= kMaxVScale8)))
                raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        }
        uint32_t sc[32];
        tmem_ld32(sa, sc);
        if constexpr (TILES) {
            // the scores of head dimensions 64-127 (S1) too; once both are in
            // registers the MMA may write the next block's S
            uint32_t s1[32];
            tmem_ld32(sa + kNB, s1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_read);
            // token t of the slot (page pg0 + t / 16, row t % 16): S0 times the
            // tile scale of its dimensions 0-63 plus S1 times that of 64-127.
            // Quadrant 0's warps check the scales they use: a finite scale >= 0
            // is, as an unsigned word, at most 0x7f7fffff (sign bit clear,
            // exponent below 255).
            uint32_t worst = 0u;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const float4 *ts = reinterpret_cast<const float4 *>(sm.t64.k[j % kNMeta][pg0 + x]);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 v = ts[q4];  // rows 2 q4, 2 q4 + 1: (half 0, half 1) each
                    const int t = 16 * x + 2 * q4;
                    sc[t] = __float_as_uint(fmaf(__uint_as_float(s1[t]), v.y, __uint_as_float(sc[t]) * v.x));
                    sc[t + 1] = __float_as_uint(fmaf(__uint_as_float(s1[t + 1]), v.w, __uint_as_float(sc[t + 1]) * v.z));
                    if (quarter == 0)
                        worst = max(max(worst, max(__float_as_uint(v.x), __float_as_uint(v.y))),
                                    max(__float_as_uint(v.z), __float_as_uint(v.w)));
                }
            }
            if (quarter == 0 && lane == 0 && worst > 0x7f7fffffu) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        } else {
            tmem_ld_wait();
        }
        if (md.pos0 + kNB > md.L || md.ntok < kNB) {
            // only on the blocks that reach the speculative slots or a partial
            // block: invisible tokens' scores -> -inf.  Visibility of this
            // slot's tokens: the 64-token mask word of the block that holds
            // them, shifted down to token tok0.
            const int wv = tok0 >> 6;
            const int h0 = md.L - md.pos0 - 64 * wv;  // history tokens from the word's first
            const int hw = min(max(h0, 0), 64);
            unsigned long long vis = hw == 64 ? ~0ull : ((1ull << hw) - 1ull);
            if (h0 >= 0) {
                if (h0 < 64) vis |= anc << h0;
            } else if (-h0 < 64) {
                vis |= anc >> (-h0);
            }
            const int nw = min(max(md.ntok - 64 * wv, 0), 64);
            if (nw < 64) vis &= (1ull << nw) - 1ull;
            const uint32_t v0 = (uint32_t)(vis >> (tok0 & 63));
#pragma unroll
            for (int t = 0; t < 32; ++t)
                if (!((v0 >> t) & 1u)) sc[t] = __float_as_uint(-CUDART_INF_F);
        }
        // the largest scaled score of the slot: a page's K scale multiplies
        // its scores, so it is the largest scaled page maximum (scales >= 0)
        float pa = -CUDART_INF_F, pb = -CUDART_INF_F;
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            pa = fmaxf(pa, __uint_as_float(sc[t]));
            pb = fmaxf(pb, __uint_as_float(sc[16 + t]));
        }
        float lm = -CUDART_INF_F;
        if (pa != -CUDART_INF_F) lm = pa * ka;
        if (pb != -CUDART_INF_F) lm = fmaxf(lm, pb * kb);
        // the quadrant's four warps exchange their maxima
        sm.xmax[quarter][j & 1][sl][lane] = lm == -CUDART_INF_F ? -CUDART_INF_F : lm * rowmul;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.xbar[quarter][j & 1]);
        if (!wait_phase(&sm.xbar[quarter][j & 1], par_of(j), a.err)) break;
        const float mx = fmaxf(fmaxf(sm.xmax[quarter][j & 1][0][lane], sm.xmax[quarter][j & 1][1][lane]),
                               fmaxf(sm.xmax[quarter][j & 1][2][lane], sm.xmax[quarter][j & 1][3][lane]));
        // the same decision in the four warps of a quadrant: they see the
        // same maxima and keep the same reference
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_ref + kRescaleLog2 || (m_ref == -CUDART_INF_F && mx != -CUDART_INF_F)) {
            alpha = ex2_approx(m_ref - mx);  // 0 when m_ref is -inf
            rescale = !first && m_ref != -CUDART_INF_F;
            m_ref = mx;
            l_run *= alpha;
        }
        // (a row past M gets -inf arguments: its P is never read)
        const float neg_m = !live ? -CUDART_INF_F : (m_ref == -CUDART_INF_F ? 0.f : -m_ref);
        // P as f16 pairs into P[j & 1], token t in column t / 2: each pair of
        // exponents by one ex2.f16x2 on the fp32 arguments rounded to f16 (an
        // argument is at most 8 under the lazy maximum, where f16 keeps P
        // within ~0.14%); the row sum adds those f16 values, in f16 within a
        // page (16 values) and in fp32 across pages; P times the page's V
        // scale is formed in f16.  A page whose K scale is 0 has scores 0:
        // its multiplier stays positive so masked columns stay -inf.
        uint32_t w[16];
        float ls = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float scp = fmaxf(rowmul * (h ? kb : ka), 1e-30f);
            const float vs = h ? vb : va;
            const uint32_t v2 = pack_f16x2(vs, vs);
            uint32_t acc = 0u;  // f16 pair (+0, +0)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 16 * h + 2 * e;
                const uint32_t p2 = ex2_f16x2(pack_f16x2(fmaf(__uint_as_float(sc[t]), scp, neg_m),
                                                         fmaf(__uint_as_float(sc[t + 1]), scp, neg_m)));
                acc = add_f16x2(acc, p2);
                w[8 * h + e] = mul_f16x2(p2, v2);
            }
            const float2 f = f16x2_to_float2(acc);
            ls += f.x + f.y;
        }
        // P[j & 1] held P_{j-2}: its P V must have read it (at block j no later
        // P V on that buffer can have completed, so the parity is unambiguous)
        if (j >= 2) wait_phase(&sm.p_free[j & 1], par_of(j - 2), a.err);
        tc_fence_after();
        tmem_st16(tmem + kTmemP + (uint32_t)(j & 1) * (kNB / 2) + lane_off + (uint32_t)(tok0 / 2), w);
        l_run += ls;
        // TMEM loads and stores are warp-collective: the whole warp takes the
        // rescale path when any of its rows needs it (factor 1 elsewhere); each
        // warp rescales the O columns of its own slot
        if (__any_sync(0xffffffffu, rescale)) {
            const float f = rescale ? alpha : 1.f;
            // O (TMEM) holds P_{<j} V; PV_{j-1} must have landed first (PV_{j-2}
            // has: P[j & 1] was free above, so the parity is unambiguous)
            wait_phase(&sm.p_free[(j - 1) & 1], par_of(j - 1), a.err);
            tc_fence_after();
            const uint32_t oa = tmem + kTmemO + lane_off + (uint32_t)tok0;
            uint32_t raw[32];
            tmem_ld32(oa, raw);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t) raw[t] = __float_as_uint(__uint_as_float(raw[t]) * f);
            tmem_st32(oa, raw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[j & 1]);
        ++j;
        if (!(md.flags & kFlagLast)) continue;

        // ------------------------------------------- the unit's epilogue
        // the row sum: the quadrant's four partial sums
        sm.lsum[quarter][sl][lane] = l_run;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.lbar[quarter]);
        if (!wait_phase(&sm.lbar[quarter], (uint32_t)(unit & 1), a.err)) break;
        const float l_tot = (sm.lsum[quarter][0][lane] + sm.lsum[quarter][1][lane]) +
                            (sm.lsum[quarter][2][lane] + sm.lsum[quarter][3][lane]);
        // this slot's 32 columns of O, once the unit's last P V has landed:
        // the final output when the unit is a whole (sequence, kv head), else
        // an fp32 partial in the piece's slot
        if (!wait_phase(&sm.o_full, (uint32_t)(unit & 1), a.err)) break;
        tc_fence_after();
        const int b = md.b, h = md.h, nsplit = md.nsplit;
        const size_t od = (((size_t)b * a.n_q + jq) * a.Hq + (size_t)h * G + gi);
        const size_t pr_own = (size_t)md.slot * a.M + r;
        {
            uint32_t raw[32];
            tmem_ld32(tmem + kTmemO + lane_off + (uint32_t)tok0, raw);
            tmem_ld_wait();
            if (live) {
                if (nsplit == 1) {
                    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
                    uint4 *orow = reinterpret_cast<uint4 *>(a.out + od * kD + tok0);
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
                    uint4 *prow4 = reinterpret_cast<uint4 *>(a.sk_acc + pr_own * kD + tok0);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4)
                        prow4[c4] = make_uint4(raw[c4 * 4], raw[c4 * 4 + 1], raw[c4 * 4 + 2], raw[c4 * 4 + 3]);
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_empty);
        if (nsplit == 1) {
            if (sl == 0 && live && a.lse) a.lse[od] = (m_ref + __log2f(l_tot)) * 0.69314718055994530942f;
            continue;
        }
        if (sl == 0 && live) {
            a.sk_ml[pr_own * 2] = m_ref;
            a.sk_ml[pr_own * 2 + 1] = l_tot;
        }
        __threadfence();
        // every softmax warp's part of the piece is written: take a ticket;
        // the last piece of the (sequence, kv head) merges all of them
        if (!soft_sync(&sm.gbar, gph, a.err)) break;
        const int u2 = b * a.Hkv + h;
        if (quarter == 0 && sl == 0 && lane == 0) {
            const int t = atomicAdd(&a.tickets[u2], 1);
            sm.last = (t == nsplit - 1);
            if (sm.last) a.tickets[u2] = 0;
        }
        if (!soft_sync(&sm.gbar, gph, a.err)) break;
        if (!sm.last) continue;
        // the merge: an online log-sum-exp merge over the pieces (running
        // maximum, rescaled sum), one warp per row, 4 columns per lane, four
        // rows and two pieces per pass so that their loads are in flight
        // together; the pieces of (b, h) are the CTAs c_first .. c_first +
        // nsplit - 1, each in its first-piece slot except possibly the first
        __threadfence();
        const long long W = a.sk_prefix[a.B];
        const int nsh = (int)min((long long)gridDim.x, W);  // shares of the work
        const long long p0 = a.sk_prefix[b];
        const long long pbh = p0 + (long long)h * ((a.sk_prefix[b + 1] - p0) / a.Hkv);
        const int c_first = (int)(((pbh + 1) * nsh - 1) / W);
        const int k_first = ((long long)c_first * W / nsh == pbh) ? 0 : 1;
        auto slot_of = [&](int i) -> size_t { return (size_t)(2 * (c_first + i) + (i == 0 ? k_first : 0)); };
        const int ew = sl * 2 + quarter;  // 0..7
        constexpr int NE = kSoftWarps;
#pragma unroll 1
        for (int r0 = ew; r0 < a.M; r0 += 4 * NE) {
            float mrow[4], lrow[4];
            float4 o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mrow[i] = -CUDART_INF_F;
                lrow[i] = 0.f;
                o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll 1
            for (int s0 = 0; s0 < nsplit; s0 += 2) {
                float2 ml[4][2];
                float4 v[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int rr = r0 + NE * i;
                        if (rr < a.M && s0 + k < nsplit) {
                            const size_t pr = slot_of(s0 + k) * a.M + rr;
                            ml[i][k] = __ldcg(reinterpret_cast<const float2 *>(a.sk_ml + pr * 2));
                            v[i][k] = __ldcg(reinterpret_cast<const float4 *>(a.sk_acc + pr * kD) + lane);
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
                        if (mk == -CUDART_INF_F) continue;  // an empty piece (or none)
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

template <bool TILES>
__global__ void __launch_bounds__(kThreads, 1)
    pva_f8_kernel(const __grid_constant__ CUtensorMap mkp, const __grid_constant__ CUtensorMap mvp,
                  const __grid_constant__ CUtensorMap mq0, const __grid_constant__ CUtensorMap mq1,
                  const __grid_constant__ AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SmemF8<TILES> &sm =
        *reinterpret_cast<SmemF8<TILES> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kNK8 = F8Cfg<TILES>::kNK8;
    constexpr uint32_t kStageArrivalsK = F8Cfg<TILES>::kStageArrivalsK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNK8; ++i) {
            mbar_init(&sm.k8_full[i], kStageArrivalsK);
            mbar_init(&sm.k8_empty[i], 1);
        }
        for (int i = 0; i < kNV8; ++i) {
            mbar_init(&sm.v8_full[i], 1);
            mbar_init(&sm.v8_empty[i], kConvWarps);
        }
        for (int i = 0; i < kNV; ++i) {
            mbar_init(&sm.v_full[i], kConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_ready[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.xbar[i][0], 4);
            mbar_init(&sm.xbar[i][1], 4);
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_empty, kSoftWarps);
        mbar_init(&sm.lbar[0], 4);
        mbar_init(&sm.lbar[1], 4);
        mbar_init(&sm.gbar, kSoftWarps);
        mbar_init(&sm.p_full[0], kSoftWarps);
        mbar_init(&sm.p_full[1], kSoftWarps);
        mbar_init(&sm.p_free[0], 1);
        mbar_init(&sm.p_free[1], 1);
        mbar_init(&sm.s_read, kSoftWarps);
        fence_mbar_init();
    }
    // query rows past M are never written by the copies: keep them zero
    for (int x = threadIdx.x; x < 2 * kQSlot / 16; x += blockDim.x)
        reinterpret_cast<uint4 *>(&sm.q[0][0])[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kProducerWarp) {
        // ================================================= producer
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&mkp);
            prefetch_tensormap(&mvp);
            prefetch_tensormap(&mq0);
            prefetch_tensormap(&mq1);
        }
        int jk = 0, jv = 0, units = 0;  // K blocks issued, V blocks issued, units started (warp-uniform)
        bool ok = true;
        const uint32_t qbytes = (uint32_t)(a.M * 128 * 2);
        // the page's scale by cp.async, counted on the K slot's barrier (a
        // missing page takes the block's first page's scale: its bytes are zero)
        auto copy_scale = [&](const float *scales, int id, int hh, float *dst, uint64_t *bar) {
            const int id0 = __shfl_sync(0x000000ffu, id, 0);
            const int sid = (id >= 0 && id < a.num_blocks) ? id : id0;
            cp_async_4(dst, scales + (size_t)sid * a.Hkv + hh);
            cp_async_mbar_arrive_noinc(bar);
        };
        auto try_issue_v = [&]() -> bool {
            return producer_try_issue_v<TILES>(sm, &mvp, a.v_scale, a.num_blocks, a.Hkv, pol, jv, jk);
        };
        auto wait_issuing_v = [&](uint64_t *bar, uint32_t parity) -> bool {
            return producer_wait_issuing_v<TILES>(sm, &mvp, a.v_scale, a.num_blocks, a.Hkv, pol, jv, jk, bar, parity,
                                                  a.err);
        };
        // This CTA's share of the work: blocks [xs, xe) of the flat order
        // (sequence, kv head, block), W blocks in all split evenly over the
        // grid; a (sequence, kv head) cut by a share boundary is a piece of
        // each CTA it meets, and the CTAs' pieces are merged like splits
        // (min(grid, W) shares, so that every share holds at least one
        // block; CTAs past them have none)
        const long long W = a.sk_prefix[a.B];
        const int nsh = (int)min((long long)gridDim.x, W);  // shares of the work
        const long long xs = (int)blockIdx.x < nsh ? (long long)blockIdx.x * W / nsh : W;
        const long long xe = (int)blockIdx.x < nsh ? (long long)(blockIdx.x + 1) * W / nsh : W;
        auto cta_of = [&](long long x) -> int { return (int)(((x + 1) * nsh - 1) / W); };
        long long x = xs;
        int b = 0;
        if (x < xe) {  // the sequence whose blocks hold x: prefix[b] <= x < prefix[b + 1]
            int lo = 0, hi = a.B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.sk_prefix[mid] <= x) lo = mid; else hi = mid - 1;
            }
            b = lo;
        }
        while (ok && x < xe) {
            while (a.sk_prefix[b + 1] <= x) ++b;
            const long long p0 = a.sk_prefix[b];
            const int nbh = (int)((a.sk_prefix[b + 1] - p0) / a.Hkv);  // blocks of each kv head
            const int h = (int)((x - p0) / nbh), f = (int)((x - p0) % nbh);
            const long long pbh = p0 + (long long)h * nbh;
            const int nblk = (int)min((long long)(nbh - f), xe - x);  // blocks of this piece
            const int c_first = cta_of(pbh);
            const int nsplit = cta_of(pbh + nbh - 1) - c_first + 1, split = (int)blockIdx.x - c_first;
            const int slot = 2 * (int)blockIdx.x + (x == xs ? 0 : 1);
            x += nblk;
            const int L = __ldg(a.context_lens + b);
            const int npages = (L + a.n_q + kBlockSize - 1) / kBlockSize;
            const int page0 = f * kPB;
            const int n = min(nblk * kPB, npages - page0);  // pages of this piece
            const int32_t *bt = a.block_table + (size_t)b * a.max_blocks + page0;
            // the piece's queries into slot units & 1, once the piece two back
            // (the slot's previous user) has issued its last S
            const int qs = units & 1;
            if (units >= 2) ok = wait_issuing_v(&sm.q_empty[qs], (uint32_t)(((units >> 1) & 1) ^ 1));
            if (!ok) break;
            if (lane == 0) {
                sm.q_is_end[qs] = 0;
                mbar_arrive_expect_tx(&sm.q_full[qs], qbytes);
                tma_load_4d(&sm.q[qs][0], &mq0, 0, h * a.G, 0, b, &sm.q_full[qs], pol);
                tma_load_4d(&sm.q[qs][kQSlab], &mq1, 0, h * a.G, 0, b, &sm.q_full[qs], pol);
            }
            __syncwarp();
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
                for (int j0 = 0; j0 < cnt; j0 += kPB) {
                    // lanes 0..7 hold the ids of the block's 8 pages
                    int my_id = __shfl_sync(0xffffffffu, blk, (j0 + (lane & 7)) & 31);
                    if (j0 + (lane & 7) >= cnt) my_id = a.num_blocks;
                    const int bi = (i0 + j0) / kPB;  // block index in the unit
                    const int ks = jk % kNK8;
                    if (jk >= kNK8) ok = wait_issuing_v(&sm.k8_empty[ks], (uint32_t)(((jk / kNK8) & 1) ^ 1));
                    if (!ok) break;
                    if (lane == 0) {
                        BlockMeta &m = sm.meta[jk % kNMeta];
                        m.b = b; m.h = h; m.split = split; m.L = L; m.nsplit = nsplit; m.slot = slot;
                        m.pos0 = (page0 + i0 + j0) * kBlockSize;
                        m.ntok = min(kPB, n - (i0 + j0)) * kBlockSize;
                        m.flags = (bi == 0 ? kFlagFirst : 0) | (bi == nblk - 1 ? kFlagLast : 0);
                        mbar_arrive_expect_tx(&sm.k8_full[ks], kTile8 + (TILES ? kPB * kTileScales * 4 : 0u));
                    }
                    if (lane < kPB) {
                        sm.vid[jk % kNMeta][lane] = my_id;
                        tma_load_4d(sm.k8[ks] + lane * kPage8, &mkp, 0, 0, h, my_id, &sm.k8_full[ks], pol);
                        if constexpr (TILES) {
                            // the page's 32 K tile scales by a bulk copy counted in the
                            // slot's bytes (a missing page takes the block's first page's)
                            const int id0 = __shfl_sync(0x000000ffu, my_id, 0);
                            const int sid = (my_id >= 0 && my_id < a.num_blocks) ? my_id : id0;
                            bulk_copy_g2s(sm.t64.k[jk % kNMeta][lane],
                                          a.k_scale + ((size_t)sid * a.Hkv + h) * kTileScales, kTileScales * 4,
                                          &sm.k8_full[ks]);
                        } else {
                            copy_scale(a.k_scale, my_id, h, &sm.ksc[jk % kNMeta][lane], &sm.k8_full[ks]);
                            copy_scale(a.v_scale, my_id, h, &sm.vsc[jk % kNMeta][lane], &sm.k8_full[ks]);
                        }
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
            if (jv >= kNV8) {
                int good = 1;
                if (lane == 0) good = wait_phase(&sm.v8_empty[jv % kNV8], (uint32_t)(((jv / kNV8) & 1) ^ 1), a.err);
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
            }
            if (ok) try_issue_v();
        }
        if (lane == 0) {
            // end-of-work markers: on the K ring (for the score issuer and,
            // through S, the softmax, which forwards it to the P V issuer), the
            // V staging ring (converters) and the next query slot (query split)
            const int ks = jk % kNK8;
            if (ok && jk >= kNK8) ok = wait_phase(&sm.k8_empty[ks], (uint32_t)(((jk / kNK8) & 1) ^ 1), a.err);
            if (ok) {
                sm.meta[jk % kNMeta].flags = kFlagEnd;
                mbar_arrive_cnt(&sm.k8_full[ks], kStageArrivalsK);
            }
            const int vs = jv % kNV8;
            if (ok && jv >= kNV8) ok = wait_phase(&sm.v8_empty[vs], (uint32_t)(((jv / kNV8) & 1) ^ 1), a.err);
            if (ok) mbar_arrive(&sm.v8_full[vs]);
            const int qs = units & 1;
            if (ok && units >= 2) ok = wait_phase(&sm.q_empty[qs], (uint32_t)(((units >> 1) & 1) ^ 1), a.err);
            if (ok) {
                sm.q_is_end[qs] = 1;
                mbar_arrive(&sm.q_full[qs]);
            }
            // wait (bounded) for the copies still in flight; a slot reused by
            // an end marker had completed before its empty barrier passed
            for (int i = jk >= kNK8 ? jk - kNK8 + 1 : 0; i < jk && ok; ++i)
                ok = wait_phase(&sm.k8_full[i % kNK8], (uint32_t)((i / kNK8) & 1), a.err);
            for (int i = jv >= kNV8 ? jv - kNV8 + 1 : 0; i < jv && ok; ++i)
                ok = wait_phase(&sm.v8_full[i % kNV8], (uint32_t)((i / kNV8) & 1), a.err);
            if (ok && units >= 1) ok = wait_phase(&sm.q_full[(units - 1) & 1], (uint32_t)(((units - 1) >> 1) & 1), a.err);
            __threadfence();
            const int done = atomicAdd(&a.sched[1], 1);
            if (done == (int)gridDim.x - 1) {
                a.sched[0] = 0;
                a.sched[1] = 0;
            }
        }
    } else if (warp == kMmaWarp) {
        // ================================================= P V issuer
        // O += P_j V_j once the softmax has published P_j (or forwarded the end
        // marker) and V_j is converted; a unit's first P V overwrites O, whose
        // previous unit must have been drained
        if (lane == 0) {
            constexpr uint32_t idPV = idesc_f16_bmn(kRows, kD);
            int unit = -1;
            for (int j = 0;; ++j) {
                if (!wait_phase(&sm.p_full[j & 1], par_of(j), a.err)) break;
                // (block j's descriptor stays until P V_j is done: the producer
                // reuses its slot only after S_{j+4}, which follows P_{j+2},
                // which waits for P V_j)
                const int flags = sm.meta[j % kNMeta].flags;
                if (flags & kFlagEnd) break;
                if (flags & kFlagFirst) {
                    ++unit;
                    if (unit >= 1 && !wait_phase(&sm.o_empty, (uint32_t)((unit - 1) & 1), a.err)) break;
                }
                const int vs = j % kNV;
                if (!wait_phase(&sm.v_full[vs], (uint32_t)((j / kNV) & 1), a.err)) break;
                tc_fence_after();
                const uint32_t pt = tmem + kTmemP + (uint32_t)(j & 1) * (kNB / 2);  // P_j (f16 pairs)
                // V_j: page kt at kt * 4 KB as [row half][slab][8 rows][128 B]; one
                // MMA per page
                const uint32_t va = smem_u32(sm.vbuf[vs]);
                const uint32_t dO = tmem + kTmemO;
#pragma unroll
                for (int kt = 0; kt < kNB / 16; ++kt) {
                    const uint64_t bd = umma_desc_sw128(va + kt * 4096, 1024, 2048);
                    umma_bf16_tmem_a(dO, pt + kt * 8, bd, idPV, ((flags & kFlagFirst) && kt == 0) ? 0u : 1u);
                }
                umma_commit(&sm.p_free[j & 1]);
                if (flags & kFlagLast) umma_commit(&sm.o_full);
            }
        }
        __syncwarp();
    } else if (warp == kSWarp) {
        // ================================================= score issuer
        if (lane == 0) {
            int unit = -1;
            for (int jj = 0;; ++jj) {
                BlockMeta m;
                if (!mma_issue_s<TILES>(sm, a.err, tmem, jj, unit, m)) break;
                if (m.flags & kFlagEnd) break;
            }
        }
        __syncwarp();
    } else if (warp == kPrepWarp) {
        // ================================================= query split
        // Thread l takes query rows l and l + 32 of a landed slot in turn (bf16,
        // two 128-byte column slabs), turning row r into q * 2^e = hi + lo: hi
        // the row rounded to E4M3,
        // lo the remainder rounded to E4M3, with 2^e the power of two that
        // puts the row's largest magnitude in [128, 256) (below the E4M3
        // maximum 448).  hi overwrites slab 0 and lo slab 1 of the same row,
        // each as 128 E4M3 bytes in the 128-byte-swizzled K-major layout the
        // MMA reads; 2^-e goes to the softmax with the unit.
        for (int nu = 0;; ++nu) {
            const int qs = nu & 1;
            if (!wait_phase(&sm.q_full[qs], par_of(nu), a.err)) break;
            if (sm.q_is_end[qs]) break;
#pragma unroll 1
            for (int rr = 0; rr < 2; ++rr) {
            const int r = rr * 32 + lane;
            float inv_scale = 1.f;
            if (r < a.M) {
                uint8_t *row0 = &sm.q[qs][r * 128];
                uint8_t *row1 = &sm.q[qs][kQSlab + r * 128];
                // chunk c of the row (dims 8c .. 8c + 7): slab c / 8, swizzled position
                auto chunk = [&](int c) -> uint4 {
                    const uint8_t *row = c < 8 ? row0 : row1;
                    return *reinterpret_cast<const uint4 *>(row + (((c & 7) ^ (r & 7)) << 4));
                };
                float amax = 0.f;
#pragma unroll 4
                for (int c = 0; c < 16; ++c) {
                    const uint4 vc = chunk(c);
                    const uint32_t ww[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        amax = fmaxf(amax, fabsf(__uint_as_float(ww[e] << 16)));
                        amax = fmaxf(amax, fabsf(__uint_as_float(ww[e] & 0xffff0000u)));
                    }
                }
                float scale = 1.f;
                if (!(amax <= 3.0e38f)) {  // inf or NaN in the row
                    raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                } else if (amax > 0.f) {
                    // amax in [2^(E-127), 2^(E-126)): 2^(134-E) puts it in [128, 256)
                    // (clamped so that both powers of two are normal floats)
                    const int E = (int)((__float_as_uint(amax) >> 23) & 0xff);
                    const int e2 = min(max(134 - E, -126), 126);
                    scale = __uint_as_float((uint32_t)(e2 + 127) << 23);
                    inv_scale = __uint_as_float((uint32_t)(127 - e2) << 23);
                }
                // 16 dims -> one 16-byte chunk of each term, written in place:
                // the whole row is read again (into registers) before the
                // first term overwrites it
                uint4 vin[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) vin[c] = chunk(c);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 src = vin[2 * g + (k >> 1)];
                        const uint32_t wa = (k & 1) ? src.z : src.x, wb = (k & 1) ? src.w : src.y;
                        const float x0 = __uint_as_float(wa << 16) * scale;
                        const float x1 = __uint_as_float(wa & 0xffff0000u) * scale;
                        const float x2 = __uint_as_float(wb << 16) * scale;
                        const float x3 = __uint_as_float(wb & 0xffff0000u) * scale;
                        const uint32_t h01 = e4m3x2_of(x0, x1), h23 = e4m3x2_of(x2, x3);
                        const float2 d01 = f16x2_to_float2(e4m3x2_to_f16x2(h01));
                        const float2 d23 = f16x2_to_float2(e4m3x2_to_f16x2(h23));
                        hw[k] = h01 | (h23 << 16);
                        lw[k] = e4m3x2_of(x0 - d01.x, x1 - d01.y) | (e4m3x2_of(x2 - d23.x, x3 - d23.y) << 16);
                    }
                    const int off = ((g ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(row0 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(row1 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            sm.qscale[nu % kNQScale][r] = inv_scale;
            }
            fence_proxy_async_smem();  // the MMA reads the terms through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.q_ready[qs]);
        }
    } else if ((warp & 3) < 2) {
        // ================================================= softmax
        // column slot warp / 4: pages 2 slot, 2 slot + 1 of each block
        softmax_role<TILES>(sm, a, tmem, warp & 3, warp >> 2);
    } else {
        // ================================================= V converters
        // Block j's E4M3 V pages -> one f16 tile in the MMA's layout (page p
        // at p * 4 KB as [row half][slab][8 rows][128 B], 128-byte swizzle),
        // exactly (the page's V scale multiplies P); rows past the sequence's
        // last token are zeroed.
        const int ci = ((warp >> 2) - 1) * 2 + (warp & 1);  // 6, 7, 10, 11 -> 0..3
        const int ct = ci * 32 + lane;
        constexpr int NCT = kConvWarps * 32;
        for (int j = 0;; ++j) {
            const int s8 = j % kNV8, tb = j % kNV;
            if (!wait_phase(&sm.v8_full[s8], (uint32_t)((j / kNV8) & 1), a.err)) break;
            // the tile is free once PV of block j - 2 is done
            if (j >= kNV && !wait_phase(&sm.p_free[tb], par_of(j - 2), a.err)) break;
            const BlockMeta md = sm.meta[j % kNMeta];
            if (md.flags & kFlagEnd) break;
            const uint8_t *src = sm.v8[s8];
            uint8_t *tile = sm.vbuf[tb];
            const int t_end = md.L + a.n_q - md.pos0;  // rows from t_end on are zeroed
            // item i: row i / 8, 16 columns 16 (i % 8) ..; four items in flight per thread
            constexpr int kItems = kNB * 8, kPer = kItems / NCT;
            static_assert(kItems % NCT == 0 && kPer % 4 == 0, "converter items");
#pragma unroll 1
            for (int t0 = 0; t0 < kPer; t0 += 4) {
                uint4 e[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = ct + NCT * (t0 + u), row = i >> 3, g = i & 7;
                    e[u] = make_uint4(0, 0, 0, 0);
                    if (row < t_end) e[u] = *reinterpret_cast<const uint4 *>(src + row * 128 + ((g ^ (row & 7)) << 4));
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = ct + NCT * (t0 + u), row = i >> 3, g = i & 7;
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
                        if (row < t_end) {
                            // this group's 64-element tile: (page, row, half) of the
                            // block (rows past the last token keep their zeros)
                            const float tsc = sm.t64.v[s8][row >> 4][(row & 15) * 2 + (g >> 2)];
                            if (!(tsc >= 0.f && tsc <= kMaxTileScale8)) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
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
                mbar_arrive(&sm.v_full[tb]);
                mbar_arrive(&sm.v8_empty[s8]);
            }
        }
    }
    // every TMEM user is done (the issuers' last operations were waited on
    // by the softmax and epilogue warps) before the owner frees it
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Per-sequence block prefix for the even split of the work: prefix[b] =
// Hkv * (number of 128-token blocks of sequences 0 .. b-1), prefix[B] = W.  A
// sequence whose length is negative or needs more than max_blocks pages
// counts no blocks (its rows are not written) and raises
// SVPA_DEVERR_BAD_VALUE.  One CTA, 1024 threads, sequences 1024 at a time.
__global__ void __launch_bounds__(1024) streamk_prefix_kernel(const int32_t *context_lens, int B, int n_q,
                                                              int Hkv, int max_blocks, long long *prefix,
                                                              int32_t *err) {
    __shared__ long long warp_tot[32];
    __shared__ long long carry;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += 1024) {
        const int b = base + (int)threadIdx.x;
        long long v = 0;
        if (b < B) {
            const int L = context_lens[b];
            const int npages = (L + n_q + kBlockSize - 1) / kBlockSize;
            if (L < 0 || npages > max_blocks)
                raise_error(err, SVPA_DEVERR_BAD_VALUE);
            else
                v = (long long)((npages + kPB - 1) / kPB) * Hkv;
        }
        // inclusive scan within the warp, then over the warp totals
        long long incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += t;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            long long wt = warp_tot[lane], wi = wt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const long long t = __shfl_up_sync(0xffffffffu, wi, d);
                if (lane >= d) wi += t;
            }
            warp_tot[lane] = wi - wt;  // exclusive prefix of the warp totals
        }
        __syncthreads();
        const long long excl = carry + warp_tot[warp] + incl - v;
        if (b < B) prefix[b] = excl;
        __syncthreads();
        if (threadIdx.x == 1023) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) prefix[B] = carry;
}

}  // namespace

namespace {
template <bool TILES>
cudaError_t launch_f8(const AttnMaps &m, const AttnArgs &a, int grid, cudaStream_t st) {
    const size_t smem = sizeof(SmemF8<TILES>) + 1024;
    static DeviceMemo<int> attr_set;  // the shared-memory opt-in, once per device
    int done = 0;
    cudaError_t e = attr_set.get(&done, [&](int *v) {
        *v = 1;
        return cudaFuncSetAttribute(pva_f8_kernel<TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    pva_f8_kernel<TILES><<<grid, kThreads, smem, st>>>(m.k[0], m.v[0], m.q[0], m.q[1], a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_streamk_prefix(const int32_t *context_lens, int B, int n_q, int Hkv, int max_blocks,
                                  long long *prefix, int32_t *err, cudaStream_t st) {
    streamk_prefix_kernel<<<1, 1024, 0, st>>>(context_lens, B, n_q, Hkv, max_blocks, prefix, err);
    return cudaGetLastError();
}

// FP8 pages, head_dim 128, G * n_q <= 64: one scale per (page, kv head), or
// (scale_tile 64) one per 64-element tile of a row
cudaError_t launch_paged_verify_attn_f8(const AttnMaps &m, const AttnArgs &a, int grid, cudaStream_t st) {
    return a.scale_tile ? launch_f8<true>(m, a, grid, st) : launch_f8<false>(m, a, grid, st);
}

}  // namespace svpa
