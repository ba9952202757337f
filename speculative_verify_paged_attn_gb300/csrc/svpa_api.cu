// svpa_api.cu -- the C ABI of libsvpa.so for the attention call: host-side
// validation, workspace layout, split-size choice, tensor-map encoding and
// kernel launches; plus the status strings and the error-word check.  The
// other entry points of the step are in svpa_step_api.cu and
// svpa_logits_api.cu.  No function here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/svpa.h"
#include "svpa_internal.h"

using namespace svpa;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int sm_count() {
    static DeviceMemo<int> memo;
    int n = 0;
    const cudaError_t e = memo.get(&n, [](int *v) {
        int dev = 0;
        cudaError_t r = cudaGetDevice(&dev);
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
        return r == cudaSuccess && *v <= 0 ? cudaErrorInvalidValue : r;
    });
    return e == cudaSuccess ? n : 148;
}

struct AttnPlan {
    int M, split_pages, max_splits;
    bool use_tc;
    int grid_slots;      // resident CTAs of the chosen kernel
    bool ordered;        // units handed out longest sequence first
    bool streamk;        // blocks split evenly over the grid (FP8 tcgen05 kernel)
    size_t off_order, off_prefix, off_ml, off_acc, bytes;
};

svpa_status plan_attn(const svpa_attn_params *p, AttnPlan *pl) {
    if (!p) return SVPA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->n_q < 1 || p->n_q > kMaxNq || p->num_q_heads < 1 || p->num_kv_heads < 1 ||
        p->num_q_heads % p->num_kv_heads != 0 || p->block_size != kBlockSize || p->max_blocks_per_seq < 1 ||
        p->num_blocks < 1 || !(p->sm_scale > 0.f) || !std::isfinite(p->sm_scale) || p->split_pages < 0)
        return SVPA_ERR_INVALID_ARG;
    if (p->kv_dtype != SVPA_KV_BF16 && p->kv_dtype != SVPA_KV_FP8_E4M3) return SVPA_ERR_INVALID_ARG;
    if (p->variant < 0 || p->variant > 2) return SVPA_ERR_INVALID_ARG;
    if (p->variant == 2 && p->head_dim != 128) return SVPA_ERR_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return SVPA_ERR_UNSUPPORTED;
    if (p->kv_dtype == SVPA_KV_FP8_E4M3 && p->head_dim != 128) return SVPA_ERR_UNSUPPORTED;
    if (p->scale_tile != 0 && p->scale_tile != 64) return SVPA_ERR_INVALID_ARG;
    // tile scales are applied by the tcgen05 kernel's converter warps only
    if (p->scale_tile == 64 && (p->kv_dtype != SVPA_KV_FP8_E4M3 || p->variant == 1)) return SVPA_ERR_UNSUPPORTED;
    const int G = p->num_q_heads / p->num_kv_heads;
    const long long M = (long long)G * p->n_q;
    if (M > kMaxRows) return SVPA_ERR_UNSUPPORTED;
    pl->M = (int)M;
    const int D = p->head_dim;
    const int eb = p->kv_dtype == SVPA_KV_FP8_E4M3 ? 1 : 2;
    // kernel variant and its resident grid (the persistent CTAs); the
    // tcgen05 kernel takes FP8 pages for up to 64 query rows per kv head
    if ((p->variant == 2 || p->scale_tile == 64) && eb == 1 && M > 64) return SVPA_ERR_UNSUPPORTED;
    pl->use_tc = p->variant == 2 || p->scale_tile == 64 ||
                 (p->variant == 0 && D == 128 && M > 16 && (eb == 2 || M <= 64));
    pl->grid_slots = sm_count();
    if (!pl->use_tc) {
        AttnLaunch lp;
        pl->grid_slots *= attn_plan_launch(D, eb == 1, (int)M, &lp) == cudaSuccess ? lp.ctas_per_sm : 4;
    }
    int sp = p->split_pages;
    if (sp == 0) {
        // about 16 units of work per resident CTA slot (sequences taken at
        // their maximum length): enough for the dynamic scheduler to balance
        // the load without multiplying split partials
        const double units = (double)std::max(1, p->batch) * p->num_kv_heads;
        const double per = units * p->max_blocks_per_seq / (16.0 * pl->grid_slots);
        int pw = 16;
        while (pw * 2 <= per && pw < 1024) pw *= 2;
        // keep a split's partial rows (written, then read back by the merge)
        // near 1% of its K/V bytes: with many rows per kv head the partials
        // and their merge cost more than the balance finer splits buy (draft
        // tree, 116 rows: 128-page splits 607 us, unsplit 476 us on GB300)
        const double page_bytes = 2.0 * kBlockSize * D * eb;
        const double partial_bytes = (double)M * (D + 2) * 4;
        int min_pages = (int)std::ceil(100.0 * partial_bytes / page_bytes);
        min_pages = (min_pages + 15) / 16 * 16;
        sp = std::max(pw, min_pages);
    }
    sp = std::min(sp, 4096);
    pl->split_pages = sp;
    pl->max_splits = (p->max_blocks_per_seq + sp - 1) / sp;
    const size_t units = (size_t)p->batch * p->num_kv_heads;
    // [scheduler counters][tickets][split (max, sum)][split accumulators]
    size_t off = kAlign + align_up(units * sizeof(int32_t));
    // unsplit units vary most in length: hand out the longest first (a
    // greedy longest-first order; the draft-tree workload's 1024 unsplit
    // units on 152 SMs: about 12% above the ideal finish in index order,
    // about 2% longest first, by a list-scheduling estimate)
    // (only when there are more units than resident CTAs: otherwise every
    // unit starts at once and the extra launch buys nothing)
    pl->ordered = pl->max_splits == 1 && p->batch > 1 && p->batch <= kMaxOrderedSeqs &&
                  units > (size_t)pl->grid_slots;
    // FP8 pages on the tcgen05 kernel: the blocks of all
    // (sequence, kv head) pairs are split evenly over the grid (no split
    // size, no ordering): [per-sequence block prefix, int64][pieces' (max,
    // sum)][pieces' accumulators], two piece slots per CTA
    pl->streamk = pl->use_tc && eb == 1;
    if (pl->streamk) {
        pl->ordered = false;
        pl->split_pages = 0;
        pl->max_splits = 1;
        pl->off_order = off;
        pl->off_prefix = off;
        off += align_up(((size_t)p->batch + 1) * sizeof(long long));
        pl->off_ml = off;
        off += align_up((size_t)2 * pl->grid_slots * M * 2 * sizeof(float));
        pl->off_acc = off;
        off += align_up((size_t)2 * pl->grid_slots * M * D * sizeof(float));
        pl->bytes = off;
        return SVPA_OK;
    }
    pl->off_prefix = 0;
    pl->off_order = off;
    if (pl->ordered) off += align_up((size_t)p->batch * sizeof(int32_t));
    pl->off_ml = off;
    if (pl->max_splits > 1) {
        off += align_up(units * pl->max_splits * M * 2 * sizeof(float));
        pl->off_acc = off;
        off += align_up(units * pl->max_splits * M * D * sizeof(float));
    } else {
        pl->off_acc = off;
    }
    pl->bytes = std::max<size_t>(off, kAlign);
    return SVPA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

svpa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SVPA_OK : SVPA_ERR_CUDA; }

}  // namespace

namespace svpa {

svpa_status check_attn_call(const svpa_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                            const float *k_scale, const float *v_scale, const int32_t *block_table,
                            const int32_t *context_lens, const uint64_t *ancestor_mask, const void *out,
                            const int32_t *error_flag) {
    if (p->batch > 65535) return SVPA_ERR_UNSUPPORTED;
    const bool fp8 = p->kv_dtype == SVPA_KV_FP8_E4M3;
    if (!q || !k_pool || !v_pool || !block_table || !context_lens || !out || !error_flag)
        return SVPA_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return SVPA_ERR_INVALID_ARG;
    if (p->scale_tile == 64 && (!aligned16(k_scale) || !aligned16(v_scale))) return SVPA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q) || !aligned16(out)) return SVPA_ERR_INVALID_ARG;
    if (ancestor_mask) {
        for (int j = 0; j < p->n_q; ++j) {
            // a query always sees itself, never a later slot
            if (!((ancestor_mask[j] >> j) & 1ull)) return SVPA_ERR_INVALID_ARG;
            if (j + 1 < 64 && (ancestor_mask[j] >> (j + 1)) != 0ull) return SVPA_ERR_INVALID_ARG;
        }
    }
    return SVPA_OK;
}

}  // namespace svpa

extern "C" {

const char *svpa_status_string(svpa_status s) {
    switch (s) {
        case SVPA_OK: return "ok";
        case SVPA_ERR_INVALID_ARG: return "invalid argument";
        case SVPA_ERR_UNSUPPORTED: return "unsupported configuration";
        case SVPA_ERR_CUDA: return "CUDA error";
        case SVPA_ERR_OUT_OF_BLOCKS: return "free block stack overflow";
        case SVPA_ERR_BAD_BLOCK: return "block id outside the pool";
        case SVPA_ERR_WORKSPACE: return "workspace missing or too small";
        case SVPA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int32_t svpa_version(void) { return 100; }

svpa_status svpa_attn_kernel(const svpa_attn_params *p, int32_t *kernel) {
    if (!kernel) return SVPA_ERR_INVALID_ARG;
    AttnPlan pl;
    const svpa_status s = plan_attn(p, &pl);
    if (s != SVPA_OK) return s;
    *kernel = pl.use_tc ? 2 : 1;
    return SVPA_OK;
}

svpa_status svpa_attn_launches(const svpa_attn_params *p, int32_t *launches) {
    if (!launches) return SVPA_ERR_INVALID_ARG;
    AttnPlan pl;
    const svpa_status s = plan_attn(p, &pl);
    if (s != SVPA_OK) return s;
    *launches = p->batch == 0 ? 0 : (pl.ordered || pl.streamk ? 2 : 1);
    return SVPA_OK;
}

svpa_status svpa_attn_workspace_size(const svpa_attn_params *p, size_t *bytes) {
    if (!bytes) return SVPA_ERR_INVALID_ARG;
    AttnPlan pl;
    const svpa_status s = plan_attn(p, &pl);
    if (s != SVPA_OK) return s;
    *bytes = pl.bytes;
    return SVPA_OK;
}

svpa_status svpa_paged_verify_attn(const svpa_attn_params *p, const void *q, const void *k_pool,
                                   const void *v_pool, const float *k_scale, const float *v_scale,
                                   const int32_t *block_table, const int32_t *context_lens,
                                   const uint64_t *ancestor_mask, void *out, float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_paged_verify_attn");
    AttnPlan pl;
    svpa_status s = plan_attn(p, &pl);
    if (s != SVPA_OK) return s;
    if (p->batch == 0) return SVPA_OK;
    s = svpa::check_attn_call(p, q, k_pool, v_pool, k_scale, v_scale, block_table, context_lens, ancestor_mask,
                              out, error_flag);
    if (s != SVPA_OK) return s;
    const bool fp8 = p->kv_dtype == SVPA_KV_FP8_E4M3;
    if (!workspace || workspace_bytes < pl.bytes || !aligned16(workspace)) return SVPA_ERR_WORKSPACE;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return SVPA_ERR_CUDA;

    const int D = p->head_dim;
    const int eb = fp8 ? 1 : 2;
    AttnMaps maps;
    memset(&maps, 0, sizeof maps);
    const cuuint64_t dims[4] = {(cuuint64_t)(fp8 ? 128 : 64), 16, (cuuint64_t)p->num_kv_heads,
                                (cuuint64_t)p->num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)D * eb, (cuuint64_t)16 * D * eb,
                                   (cuuint64_t)p->num_kv_heads * 16 * D * eb};
    const cuuint32_t box[4] = {(cuuint32_t)(fp8 ? 128 : 64), 16, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int slabs = (D * eb) / 128;
    for (int sl = 0; sl < 2; ++sl) {
        const int use = sl < slabs ? sl : 0;
        char *kb = (char *)const_cast<void *>(k_pool) + use * 128;
        char *vb = (char *)const_cast<void *>(v_pool) + use * 128;
        if (enc(&maps.k[sl], dt, 4, kb, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
        if (enc(&maps.v[sl], dt, 4, vb, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
    }

    if (pl.use_tc && !fp8) {
        // one (page, kv head) tile per copy: dims (64 columns, 8 rows, 2 column
        // slabs, 2 row halves, kv head x block), landing as
        // [row half][slab][8 rows][128 B] -- 1 KB swizzle atoms with a uniform
        // 2 KB stride between 8-row groups across the pages of a block
        const cuuint64_t pd[5] = {64, 8, 2, 2, (cuuint64_t)p->num_kv_heads * p->num_blocks};
        const cuuint64_t ps[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)8 * D * 2, (cuuint64_t)16 * D * 2};
        const cuuint32_t pbox[5] = {64, 8, 2, 2, 1};
        const cuuint32_t es5[5] = {1, 1, 1, 1, 1};
        if (enc(&maps.kpage, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(k_pool), pd, ps, pbox, es5,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
        if (enc(&maps.vpage, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(v_pool), pd, ps, pbox, es5,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
    }
    if (!pl.use_tc && !fp8 && D == 128) {
        // warp-MMA kernel: one (page, kv head) tile per copy, landing as
        // [slab][16 rows][128 B] (dims 64 columns, 16 rows, 2 slabs, kv heads, blocks)
        const cuuint64_t sd[5] = {64, 16, 2, (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->num_blocks};
        const cuuint64_t ss[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)16 * D * 2,
                                  (cuuint64_t)p->num_kv_heads * 16 * D * 2};
        const cuuint32_t sbox[5] = {64, 16, 2, 1, 1};
        const cuuint32_t es5[5] = {1, 1, 1, 1, 1};
        if (enc(&maps.kslabs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(k_pool), sd, ss, sbox, es5,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
        if (enc(&maps.vslabs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(v_pool), sd, ss, sbox, es5,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SVPA_ERR_CUDA;
    }
    {
        // queries [B, n_q, Hq, D] bf16: box = (64 columns, G heads, n_q queries, 1)
        const int G = p->num_q_heads / p->num_kv_heads;
        const cuuint64_t qd[4] = {64, (cuuint64_t)p->num_q_heads, (cuuint64_t)p->n_q, (cuuint64_t)p->batch};
        const cuuint64_t qs[3] = {(cuuint64_t)D * 2, (cuuint64_t)p->num_q_heads * D * 2,
                                  (cuuint64_t)p->n_q * p->num_q_heads * D * 2};
        const cuuint32_t qbox[4] = {64, (cuuint32_t)G, (cuuint32_t)p->n_q, 1};
        const int qslabs = D * 2 / 128;
        for (int sl = 0; sl < 2; ++sl) {
            char *qb = (char *)const_cast<void *>(q) + (sl < qslabs ? sl : 0) * 128;
            if (enc(&maps.q[sl], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, qb, qd, qs, qbox, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return SVPA_ERR_CUDA;
        }
    }

    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.sched = reinterpret_cast<int32_t *>(ws);
    a.tickets = reinterpret_cast<int32_t *>(ws + kAlign);
    a.order = pl.ordered ? reinterpret_cast<const int32_t *>(ws + pl.off_order) : nullptr;
    a.part_ml = reinterpret_cast<float *>(ws + pl.off_ml);
    a.part_acc = reinterpret_cast<float *>(ws + pl.off_acc);
    a.err = error_flag;
    a.B = p->batch;
    a.n_q = p->n_q;
    a.Hq = p->num_q_heads;
    a.Hkv = p->num_kv_heads;
    a.G = p->num_q_heads / p->num_kv_heads;
    a.M = pl.M;
    a.max_blocks = p->max_blocks_per_seq;
    a.num_blocks = p->num_blocks;
    a.split_pages = pl.split_pages;
    a.max_splits = pl.max_splits;
    a.scale_log2 = p->sm_scale * 1.4426950408889634f;
    a.scale_tile = p->scale_tile;
    for (int j = 0; j < p->n_q; ++j)
        a.anc[j] = ancestor_mask ? ancestor_mask[j] : ((j == 63) ? ~0ull : ((1ull << (j + 1)) - 1ull));
    a.total_units = p->batch * p->num_kv_heads * pl.max_splits;
    if (pl.ordered) {
        cudaError_t e = launch_seq_order(context_lens, p->batch, reinterpret_cast<int32_t *>(ws + pl.off_order),
                                         static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (pl.streamk) {
        a.sk_prefix = reinterpret_cast<const long long *>(ws + pl.off_prefix);
        a.sk_ml = reinterpret_cast<float *>(ws + pl.off_ml);
        a.sk_acc = reinterpret_cast<float *>(ws + pl.off_acc);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = launch_streamk_prefix(context_lens, p->batch, p->n_q, p->num_kv_heads,
                                              p->max_blocks_per_seq, reinterpret_cast<long long *>(ws + pl.off_prefix),
                                              error_flag, st);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(launch_paged_verify_attn_f8(maps, a, pl.grid_slots, st));
    }
    if (pl.use_tc) {
        const int grid = std::max(1, std::min(pl.grid_slots, a.total_units));
        return from_cuda(launch_paged_verify_attn_tc(maps, a, grid, static_cast<cudaStream_t>(stream)));
    }
    AttnLaunch lp;
    if (attn_plan_launch(D, fp8, pl.M, &lp) != cudaSuccess) return SVPA_ERR_CUDA;
    a.n_stages = lp.n_stages;
    const int grid = std::max(1, std::min(lp.ctas_per_sm * sm_count(), a.total_units));
    return from_cuda(launch_paged_verify_attn(maps, a, D, fp8, grid, lp.smem, static_cast<cudaStream_t>(stream)));
}

svpa_status svpa_check_error(const int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_check_error");
    if (!error_flag) return SVPA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SVPA_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, error_flag, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SVPA_ERR_CUDA;
    if (v == 0) return SVPA_OK;
    if (v & SVPA_DEVERR_BAD_BLOCK) return SVPA_ERR_BAD_BLOCK;
    if (v & SVPA_DEVERR_FREE_OVERFLOW) return SVPA_ERR_OUT_OF_BLOCKS;
    if (v & SVPA_DEVERR_TIMEOUT) return SVPA_ERR_TIMEOUT;
    return SVPA_ERR_INVALID_ARG;
}

}  // extern "C"
