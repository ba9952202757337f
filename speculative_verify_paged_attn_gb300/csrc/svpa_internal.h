// svpa_internal.h -- host/device argument structs and launch entry points
// shared between the C-ABI layer (svpa_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>
#include <mutex>

#include "../../include/svpa.h"

namespace svpa {

// An NVTX range around one C-ABI call, named after the entry point, so that a
// profiler's timeline shows which library call enqueued which kernels.  With
// no tool attached the NVTX calls return at once.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// Host-side launch facts (function attributes, occupancy, SM count) are
// computed once per device and remembered: a serving loop calls with the same
// shapes every step, and each runtime query costs microseconds of host time.
constexpr int kMaxDevices = 64;
template <typename T>
struct DeviceMemo {
    std::mutex mu;
    T value[kMaxDevices];
    bool have[kMaxDevices] = {};
    // f(T*) -> cudaError_t computes the value on a miss; errors are not remembered
    template <typename F>
    cudaError_t get(T *out, F f) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return f(out);
        std::lock_guard<std::mutex> g(mu);
        if (!have[dev]) {
            e = f(&value[dev]);
            if (e != cudaSuccess) return e;
            have[dev] = true;
        }
        *out = value[dev];
        return cudaSuccess;
    }
};

constexpr int kBlockSize = 16;   // tokens per page
constexpr int kMaxNq = 64;       // queries per sequence (one 64-bit mask row each)
constexpr int kMaxRows = 128;    // GQA group size x queries handled by one CTA

// Arguments of the paged verification attention kernel (passed by value).
struct AttnArgs {
    const __nv_bfloat16 *q;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_table;
    const int32_t *context_lens;
    __nv_bfloat16 *out;
    float *lse;
    float *part_acc;      // [B*Hkv, max_splits, M, D]
    float *part_ml;       // [B*Hkv, max_splits, M, 2]  (running max in log2 units, sum)
    int32_t *tickets;     // [B*Hkv]
    const int32_t *order; // [B] sequences, longest first, in the order units are handed out; or null
    int32_t *sched;       // [2]: next work unit, CTAs finished (both back to 0 after a call)
    int32_t *err;
    int32_t B, n_q, Hq, Hkv, G, M;
    int32_t max_blocks, num_blocks, split_pages, max_splits, n_stages, total_units;
    int32_t scale_tile;   // FP8 scales: 0 per (page, kv head), 64 per 64-element tile
    float scale_log2;     // sm_scale * log2(e)
    unsigned long long anc[kMaxNq];  // visibility of speculative slots per query
    // even split of the blocks over the grid (FP8 tcgen05 kernel): the
    // per-sequence block prefix [B + 1], and the pieces' partial rows, two
    // slots per CTA: (max, sum) [2 * grid, M, 2] and accumulators [2 * grid, M, D]
    const long long *sk_prefix;
    float *sk_ml;
    float *sk_acc;
};

struct AttnMaps {
    CUtensorMap k[2];     // 128-byte column slabs of the K pages
    CUtensorMap v[2];
    CUtensorMap q[2];     // 128-byte column slabs of the queries of one (sequence, kv head)
    CUtensorMap kpage;    // a whole bf16 (page, kv head) tile in one box (tcgen05 kernel)
    CUtensorMap vpage;
    CUtensorMap kslabs;   // a whole bf16 D-128 (page, kv head) tile in one box, as [slab][16 rows]
    CUtensorMap vslabs;
};

struct AttnLaunch {
    int n_stages;
    int ctas_per_sm;
    size_t smem;
};

// The attention call's pointer, alignment, batch and ancestor-mask checks
// (everything but the shape, which plan checks, and the workspace): both
// attention entry points run them before enqueueing anything.
svpa_status check_attn_call(const svpa_attn_params *p, const void *q, const void *k_pool, const void *v_pool,
                            const float *k_scale, const float *v_scale, const int32_t *block_table,
                            const int32_t *context_lens, const uint64_t *ancestor_mask, const void *out,
                            const int32_t *error_flag);

// Launch the attention kernel matching (head_dim, fp8, row tiles).
cudaError_t launch_paged_verify_attn(const AttnMaps &maps, const AttnArgs &a, int head_dim,
                                     bool fp8, int grid, size_t smem, cudaStream_t stream);
// Stage count, resident CTAs per SM and dynamic shared memory for a shape.
cudaError_t attn_plan_launch(int head_dim, bool fp8, int M, AttnLaunch *out);
// Sequence ids sorted by decreasing context length (ties by index) into
// order[0..B): the persistent kernels hand out long units first.
constexpr int kMaxOrderedSeqs = 4096;
cudaError_t launch_seq_order(const int32_t *context_lens, int B, int32_t *order, cudaStream_t stream);
// tcgen05 / TMEM variant (bf16 pages, head_dim 128, one CTA per SM).
cudaError_t launch_paged_verify_attn_tc(const AttnMaps &maps, const AttnArgs &a, int grid, cudaStream_t stream);
// tcgen05 / TMEM variant for FP8 pages with one scale per (page, kv head):
// E4M3 scores MMA on the staged K pages, G * n_q <= 64, one CTA per SM.
cudaError_t launch_paged_verify_attn_f8(const AttnMaps &maps, const AttnArgs &a, int grid, cudaStream_t stream);
// The per-sequence block prefix the FP8 tcgen05 kernel splits its work by.
cudaError_t launch_streamk_prefix(const int32_t *context_lens, int B, int n_q, int Hkv, int max_blocks,
                                  long long *prefix, int32_t *err, cudaStream_t stream);

// Rejection sampler.
struct AcceptArgs {
    const float *p;
    const float *q;
    const int32_t *tokens;
    const float *u_acc;
    const float *u_s;
    int32_t *accepted_len;
    int32_t *out_tokens;
    uint8_t *near;
    int32_t *err;
    int32_t B, gamma, V;
};
cudaError_t launch_spec_accept(const AcceptArgs &a, cudaStream_t stream);

// Rejection sampler fed by logits (P and Q formed in the kernel).
struct LogitsArgs {
    const float *lp;  // target logits [B, gamma+1, V]
    const float *lq;  // draft logits [B, gamma, V]
    const int32_t *tokens;
    const float *u_acc;
    const float *u_s;
    int32_t *accepted_len;
    int32_t *out_tokens;
    uint8_t *near;
    int32_t *err;
    int32_t B, gamma, V;
    float c_target, c_draft;  // log2(e) / temperature, > 0
    float2 *stats;            // workspace: (max, sum) per 8192-token slab [B, 2 gamma + 1, n_slabs]
    int32_t n_slabs;          // set by the launch
};
size_t spec_accept_logits_stats_bytes(int B, int gamma, int V);
cudaError_t launch_spec_accept_logits(const LogitsArgs &a, cudaStream_t stream);
int spec_accept_tree_max_vocab();

struct TreeArgs {
    const float *p;
    const float *q;
    const int32_t *tokens;
    const float *u_acc;
    const float *u_s;
    int32_t *accepted_len;
    int32_t *path_nodes;
    int32_t *out_tokens;
    uint8_t *near;
    int32_t *err;
    int32_t B, n_nodes, V, width, n_internal;
    float c_target, c_draft;  // fed by logits (p, q are logits): log2(e) / temperature
    int8_t parent[kMaxNq];
    int8_t qrow[kMaxNq];
};
// parent[] validated (parent[0] = -1, 0 <= parent[i] < i, n_nodes 1..64) into
// a.parent, a.qrow, a.n_nodes, a.n_internal and a.width; false when invalid.
bool fill_tree_shape(const int32_t *parent, int n_nodes, TreeArgs &a);
cudaError_t launch_spec_accept_tree(const TreeArgs &a, cudaStream_t stream);
cudaError_t launch_spec_accept_tree_logits(const TreeArgs &a, cudaStream_t stream);

struct CommitArgs {
    int32_t *block_table;
    int32_t *context_lens;
    const int32_t *accepted_len;
    int32_t *refcount;
    int32_t *free_stack;
    int32_t *free_top;
    const int32_t *path_nodes;
    uint8_t *k_pool;
    uint8_t *v_pool;
    int32_t *err;
    int32_t B, n_q, max_blocks, num_blocks, path_width, Hkv, row_bytes;
};
cudaError_t launch_block_table_commit(const CommitArgs &a, cudaStream_t stream);

// Paged K/V append (allocation, copy-on-write, FP8 quantise-on-write).
constexpr int kMaxAppendRows = 4096;                           // n_new limit
constexpr int kMaxAppendPages = kMaxAppendRows / kBlockSize + 1;  // pages one sequence touches
struct AppendArgs {
    const uint16_t *new_k;  // bf16 bits [B, n_new, Hkv, D]
    const uint16_t *new_v;
    int32_t *block_table;
    const int32_t *context_lens;
    int32_t *refcount;
    int32_t *free_stack;
    int32_t *free_top;
    uint8_t *k_pool;
    uint8_t *v_pool;
    float *k_scale;
    float *v_scale;
    int32_t *err;
    size_t page_bytes;      // one block, all kv heads
    int32_t scales_per_block;  // FP8: Hkv (per page) or Hkv * 16 * D / 64 (per 64-element tile)
    int32_t B, n_new, Hkv, D, max_blocks, num_blocks, fp8, scale_tile;
};
cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream);

// Acceptance telemetry and the adaptive draft length.
struct GammaArgs {
    const int32_t *accepted_len;
    float *seq_state;         // [B][2] (A, N) or null
    int32_t *seq_gamma_next;  // [B] or null
    float *batch_state;       // [2]
    int32_t *batch_gamma_next;
    float *telemetry;         // [4]
    int32_t *err;
    int32_t B, gamma;
    float decay, r;
};
cudaError_t launch_gamma_update(const GammaArgs &a, cudaStream_t stream);

}  // namespace svpa
