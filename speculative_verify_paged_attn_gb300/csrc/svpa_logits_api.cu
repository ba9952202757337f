// svpa_logits_api.cu -- the C ABI of the samplers' logits front-ends (linear
// and draft tree): host-side validation and the launches.  No function here allocates device memory.
#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>
#include <string.h>

#include <cmath>

#include "../../include/svpa.h"
#include "svpa_internal.h"

using namespace svpa;

namespace {

// log2(e) / T rounded once to fp32, for a finite T > 0 whose scale is finite
// in fp32 (a temperature so small that it overflows is refused).
bool scale_of_temperature(float T, float *c) {
    if (!std::isfinite(T) || !(T > 0.f)) return false;
    const double v = 1.4426950408889634 / (double)T;
    if (!(v <= (double)FLT_MAX)) return false;
    *c = (float)v;
    return true;
}

}  // namespace

extern "C" {

svpa_status svpa_spec_accept_logits_workspace_size(int32_t batch, int32_t gamma, int32_t vocab, size_t *bytes) {
    if (!bytes || batch < 0 || gamma < 1 || gamma > 32 || vocab < 1) return SVPA_ERR_INVALID_ARG;
    if (vocab > spec_accept_tree_max_vocab()) return SVPA_ERR_UNSUPPORTED;
    // the (max, sum) pair of every 8192-token slab of every row
    const size_t need = spec_accept_logits_stats_bytes(batch, gamma, vocab);
    *bytes = need < 256 ? 256 : (need + 255) / 256 * 256;
    return SVPA_OK;
}

svpa_status svpa_spec_accept_logits(int32_t batch, int32_t gamma, int32_t vocab, float temperature,
                                    float draft_temperature, const float *target_logits,
                                    const float *draft_logits, const int32_t *draft_tokens,
                                    const float *u_accept, const float *u_sample, int32_t *accepted_len,
                                    int32_t *out_tokens, uint8_t *near_boundary, void *workspace,
                                    size_t workspace_bytes, int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_spec_accept_logits");
    if (batch < 0 || gamma < 1 || gamma > 32 || vocab < 1) return SVPA_ERR_INVALID_ARG;
    float ct = 0.f, cd = 0.f;
    if (!scale_of_temperature(temperature, &ct) || !scale_of_temperature(draft_temperature, &cd))
        return SVPA_ERR_INVALID_ARG;
    if (vocab > spec_accept_tree_max_vocab()) return SVPA_ERR_UNSUPPORTED;  // one cluster per row
    if (batch > 0x7fffffff / 8) return SVPA_ERR_UNSUPPORTED;
    if ((long long)batch * (2 * gamma + 1) * ((vocab + 8191) / 8192) > 0x7fffffffLL) return SVPA_ERR_UNSUPPORTED;
    if (batch == 0) return SVPA_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample || !accepted_len ||
        !out_tokens || !error_flag)
        return SVPA_ERR_INVALID_ARG;
    size_t need = 0;
    svpa_spec_accept_logits_workspace_size(batch, gamma, vocab, &need);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15) != 0)
        return SVPA_ERR_WORKSPACE;
    LogitsArgs a;
    memset(&a, 0, sizeof a);
    a.lp = target_logits;
    a.lq = draft_logits;
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
    a.c_target = ct;
    a.c_draft = cd;
    a.stats = static_cast<float2 *>(workspace);
    const cudaError_t e = launch_spec_accept_logits(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVPA_OK : SVPA_ERR_CUDA;
}

svpa_status svpa_spec_accept_tree_logits(int32_t batch, int32_t n_nodes, int32_t vocab, const int32_t *parent,
                                         float temperature, float draft_temperature, const float *target_logits,
                                         const float *draft_logits, const int32_t *node_tokens,
                                         const float *u_accept, const float *u_sample, int32_t *accepted_len,
                                         int32_t *path_nodes, int32_t *out_tokens, uint8_t *near_boundary,
                                         int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_spec_accept_tree_logits");
    TreeArgs a;
    memset(&a, 0, sizeof a);
    if (batch < 0 || vocab < 1 || !fill_tree_shape(parent, n_nodes, a)) return SVPA_ERR_INVALID_ARG;
    float ct = 0.f, cd = 0.f;
    if (!scale_of_temperature(temperature, &ct) || !scale_of_temperature(draft_temperature, &cd))
        return SVPA_ERR_INVALID_ARG;
    if (vocab > spec_accept_tree_max_vocab()) return SVPA_ERR_UNSUPPORTED;  // one cluster per row
    if (batch > 0x7fffffff / 8) return SVPA_ERR_UNSUPPORTED;
    if (batch == 0) return SVPA_OK;
    if (!target_logits || !draft_logits || !node_tokens || !u_accept || !u_sample || !accepted_len ||
        !path_nodes || !out_tokens || !error_flag)
        return SVPA_ERR_INVALID_ARG;
    a.p = target_logits;
    a.q = draft_logits;
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
    a.c_target = ct;
    a.c_draft = cd;
    const cudaError_t e = launch_spec_accept_tree_logits(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SVPA_OK : SVPA_ERR_CUDA;
}

}  // extern "C"
