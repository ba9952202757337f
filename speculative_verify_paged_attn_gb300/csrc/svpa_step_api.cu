// svpa_step_api.cu -- the C ABI of the step's calls after the attention: the
// samplers on probabilities (linear and draft tree), the block-table commit,
// the K/V append and the draft-length update.  Host-side validation and the
// launches; no function here allocates device memory.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "../../include/svpa.h"
#include "svpa_internal.h"

using namespace svpa;

namespace {

constexpr size_t kAlign = 256;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

svpa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SVPA_OK : SVPA_ERR_CUDA; }

}  // namespace

namespace svpa {

bool fill_tree_shape(const int32_t *parent, int n_nodes, TreeArgs &a) {
    if (!parent || n_nodes < 1 || n_nodes > kMaxNq || parent[0] != -1) return false;
    for (int i = 1; i < n_nodes; ++i)
        if (parent[i] < 0 || parent[i] >= i) return false;
    int depth_max = 0, n_internal = 0;
    for (int i = 0; i < n_nodes; ++i) {
        int d = 0;
        for (int x = i; x > 0; x = parent[x]) ++d;
        depth_max = std::max(depth_max, d);
        bool has_child = false;
        for (int c = i + 1; c < n_nodes; ++c) has_child |= parent[c] == i;
        a.qrow[i] = has_child ? (int8_t)n_internal++ : (int8_t)-1;
        a.parent[i] = (int8_t)parent[i];
    }
    a.n_nodes = n_nodes;
    a.n_internal = n_internal;
    a.width = depth_max + 1;
    return true;
}

}  // namespace svpa

extern "C" {

svpa_status svpa_spec_accept_workspace_size(int32_t batch, int32_t vocab, size_t *bytes) {
    if (!bytes || batch < 0 || vocab < 1) return SVPA_ERR_INVALID_ARG;
    // reserved: the samplers keep no state between CTAs
    *bytes = kAlign;
    return SVPA_OK;
}

svpa_status svpa_spec_accept(int32_t batch, int32_t gamma, int32_t vocab, const float *p_probs,
                             const float *q_probs, const int32_t *draft_tokens, const float *u_accept,
                             const float *u_sample, int32_t *accepted_len, int32_t *out_tokens,
                             uint8_t *near_boundary, void *workspace, size_t workspace_bytes,
                             int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_spec_accept");
    if (batch < 0 || gamma < 1 || gamma > 32 || vocab < 1) return SVPA_ERR_INVALID_ARG;
    if (batch == 0) return SVPA_OK;
    if (!p_probs || !q_probs || !draft_tokens || !u_accept || !u_sample || !accepted_len || !out_tokens ||
        !error_flag)
        return SVPA_ERR_INVALID_ARG;
    size_t need;
    svpa_spec_accept_workspace_size(batch, vocab, &need);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SVPA_ERR_WORKSPACE;
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.p = p_probs;
    a.q = q_probs;
    a.tokens = draft_tokens;
    a.u_acc = u_accept;
    a.u_s = u_sample;
    a.accepted_len = accepted_len;
    a.out_tokens = out_tokens;
    a.near = near_boundary;
    a.err = error_flag;
    a.B = batch;
    a.gamma = gamma;
    a.V = vocab;
    return from_cuda(launch_spec_accept(a, static_cast<cudaStream_t>(stream)));
}

svpa_status svpa_spec_accept_tree(int32_t batch, int32_t n_nodes, int32_t vocab, const int32_t *parent,
                                  const float *p_probs, const float *q_probs, const int32_t *node_tokens,
                                  const float *u_accept, const float *u_sample, int32_t *accepted_len,
                                  int32_t *path_nodes, int32_t *out_tokens, uint8_t *near_boundary,
                                  void *workspace, size_t workspace_bytes, int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_spec_accept_tree");
    (void)workspace;
    (void)workspace_bytes;
    TreeArgs a;
    memset(&a, 0, sizeof a);
    if (batch < 0 || vocab < 1 || !fill_tree_shape(parent, n_nodes, a)) return SVPA_ERR_INVALID_ARG;
    if (vocab > spec_accept_tree_max_vocab()) return SVPA_ERR_UNSUPPORTED;  // residual slices in shared memory
    if (batch == 0) return SVPA_OK;
    if (!p_probs || !q_probs || !node_tokens || !u_accept || !u_sample || !accepted_len || !path_nodes ||
        !out_tokens || !error_flag)
        return SVPA_ERR_INVALID_ARG;
    a.p = p_probs;
    a.q = q_probs;
    a.tokens = node_tokens;
    a.u_acc = u_accept;
    a.u_s = u_sample;
    a.accepted_len = accepted_len;
    a.path_nodes = path_nodes;
    a.out_tokens = out_tokens;
    a.near = near_boundary;
    a.err = error_flag;
    a.B = batch;
    a.V = vocab;
    return from_cuda(launch_spec_accept_tree(a, static_cast<cudaStream_t>(stream)));
}

svpa_status svpa_block_table_commit(int32_t batch, int32_t n_q, int32_t block_size, int32_t max_blocks_per_seq,
                                    int32_t num_blocks, int32_t *block_table, int32_t *context_lens,
                                    const int32_t *accepted_len, int32_t *refcount, int32_t *free_stack,
                                    int32_t *free_top, const int32_t *path_nodes, int32_t path_width,
                                    void *k_pool, void *v_pool, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t kv_dtype, int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_block_table_commit");
    if (batch < 0 || n_q < 1 || n_q > kMaxNq || block_size != kBlockSize || max_blocks_per_seq < 1 ||
        num_blocks < 1)
        return SVPA_ERR_INVALID_ARG;
    if (batch == 0) return SVPA_OK;
    if (!block_table || !context_lens || !accepted_len || !refcount || !free_stack || !free_top || !error_flag)
        return SVPA_ERR_INVALID_ARG;
    CommitArgs a;
    memset(&a, 0, sizeof a);
    if (path_nodes) {
        if (kv_dtype != SVPA_KV_BF16) return SVPA_ERR_UNSUPPORTED;  // per-page FP8 scales differ
        if (!k_pool || !v_pool || path_width < 1 || num_kv_heads < 1 || (head_dim != 64 && head_dim != 128))
            return SVPA_ERR_INVALID_ARG;
        if (!aligned16(k_pool) || !aligned16(v_pool)) return SVPA_ERR_INVALID_ARG;
        a.row_bytes = head_dim * 2;
    }
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.accepted_len = accepted_len;
    a.refcount = refcount;
    a.free_stack = free_stack;
    a.free_top = free_top;
    a.path_nodes = path_nodes;
    a.k_pool = static_cast<uint8_t *>(k_pool);
    a.v_pool = static_cast<uint8_t *>(v_pool);
    a.err = error_flag;
    a.B = batch;
    a.n_q = n_q;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.path_width = path_width;
    a.Hkv = num_kv_heads;
    return from_cuda(launch_block_table_commit(a, static_cast<cudaStream_t>(stream)));
}

svpa_status svpa_kv_append(int32_t batch, int32_t n_new, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t max_blocks_per_seq, int32_t num_blocks, int32_t kv_dtype,
                           int32_t scale_tile, const void *new_k, const void *new_v, int32_t *block_table,
                           const int32_t *context_lens, int32_t *refcount, int32_t *free_stack,
                           int32_t *free_top, void *k_pool, void *v_pool, float *k_scale, float *v_scale,
                           int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_kv_append");
    if (batch < 0 || n_new < 1 || n_new > kMaxAppendRows || num_kv_heads < 1 || num_kv_heads > 4096 ||
        head_dim < 8 || head_dim % 8 != 0 || block_size != kBlockSize || max_blocks_per_seq < 1 ||
        num_blocks < 1 || (kv_dtype != SVPA_KV_BF16 && kv_dtype != SVPA_KV_FP8_E4M3))
        return SVPA_ERR_INVALID_ARG;
    const bool fp8 = kv_dtype == SVPA_KV_FP8_E4M3;
    if (fp8 ? (head_dim % 16 != 0 || head_dim > 256) : head_dim > 1024) return SVPA_ERR_INVALID_ARG;
    if (scale_tile != 0 && (scale_tile != 64 || !fp8 || head_dim % 64 != 0)) return SVPA_ERR_INVALID_ARG;
    if (batch == 0) return SVPA_OK;
    if (!new_k || !new_v || !block_table || !context_lens || !refcount || !free_stack || !free_top || !k_pool ||
        !v_pool || !error_flag || (fp8 && (!k_scale || !v_scale)))
        return SVPA_ERR_INVALID_ARG;
    if (!aligned16(new_k) || !aligned16(new_v) || !aligned16(k_pool) || !aligned16(v_pool))
        return SVPA_ERR_INVALID_ARG;
    AppendArgs a;
    memset(&a, 0, sizeof a);
    a.new_k = static_cast<const uint16_t *>(new_k);
    a.new_v = static_cast<const uint16_t *>(new_v);
    a.block_table = block_table;
    a.context_lens = context_lens;
    a.refcount = refcount;
    a.free_stack = free_stack;
    a.free_top = free_top;
    a.k_pool = static_cast<uint8_t *>(k_pool);
    a.v_pool = static_cast<uint8_t *>(v_pool);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.err = error_flag;
    a.page_bytes = (size_t)num_kv_heads * kBlockSize * head_dim * (fp8 ? 1 : 2);
    a.scales_per_block = scale_tile ? num_kv_heads * kBlockSize * (head_dim / 64) : num_kv_heads;
    a.scale_tile = scale_tile;
    a.B = batch;
    a.n_new = n_new;
    a.Hkv = num_kv_heads;
    a.D = head_dim;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.fp8 = fp8;
    return from_cuda(launch_kv_append(a, static_cast<cudaStream_t>(stream)));
}

svpa_status svpa_gamma_update(int32_t batch, int32_t gamma, const int32_t *accepted_len, float *seq_state,
                              int32_t *seq_gamma_next, float *batch_state, int32_t *batch_gamma_next,
                              float *telemetry, float decay, float draft_cost_ratio, int32_t *error_flag,
                              void *stream) {
    svpa::NvtxRange nvtx_range("svpa_gamma_update");
    if (batch < 1 || gamma < 1 || gamma > kMaxNq - 1 || !(decay >= 0.f && decay <= 1.f) ||
        !(draft_cost_ratio >= 0.f) || !accepted_len || !batch_state || !batch_gamma_next || !telemetry ||
        !error_flag || (seq_gamma_next && !seq_state))
        return SVPA_ERR_INVALID_ARG;
    GammaArgs a;
    a.accepted_len = accepted_len;
    a.seq_state = seq_state;
    a.seq_gamma_next = seq_gamma_next;
    a.batch_state = batch_state;
    a.batch_gamma_next = batch_gamma_next;
    a.telemetry = telemetry;
    a.err = error_flag;
    a.B = batch;
    a.gamma = gamma;
    a.decay = decay;
    a.r = draft_cost_ratio;
    return from_cuda(launch_gamma_update(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
