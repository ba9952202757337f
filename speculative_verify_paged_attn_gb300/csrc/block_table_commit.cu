// block_table_commit.cu -- commit accepted tokens / roll back rejected ones.
//
// Semantics ("LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING",
// architecture diagram: commit accepted tokens to the KV-cache block table,
// discard the KV blocks of rejected tokens; "Speculative Decoding &
// KV-Cache PagedAttention in Enterprise LLM Serving", PagedKVCacheManager:
// per-block reference counts, a block returns to the free pool when its
// count reaches zero, shared prefix blocks carry one count per holder):
//   new length = L + k + 1; logical pages from ceil(new/16) up to the last
//   page the step wrote are dropped from the table, their counts decremented
//   and the blocks whose count reaches zero pushed on the free stack.
// For a draft tree the accepted path's K/V rows are first moved to the
// linear slots L+1 .. L+k so that the committed history stays contiguous.
//
// One CTA per sequence.  Device-side checks raise error bits instead of
// trapping: a bad length or draft-tree path leaves that sequence untouched; a
// bad block id among the dropped pages is skipped.
#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

__global__ void __launch_bounds__(128) commit_kernel(const __grid_constant__ CommitArgs a) {
    const int b = blockIdx.x;
    __shared__ int s_L, s_k, s_ok;
    int32_t *table = a.block_table + (size_t)b * a.max_blocks;
    if (threadIdx.x == 0) {
        const int L = a.context_lens[b];
        const int k = a.accepted_len[b];
        const int had = (L + a.n_q + kBlockSize - 1) / kBlockSize;
        int ok = !(L < 0 || k < 0 || k >= a.n_q || had > a.max_blocks);
        if (!ok) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        if (ok && a.path_nodes) {
            // the whole path is checked before any row moves, so that a bad
            // path leaves the sequence (rows, table, counts, length) untouched
            const int32_t *path = a.path_nodes + (size_t)b * a.path_width;
            ok = k < a.path_width;
            for (int d = 1; ok && d <= k; ++d) {
                const int pd = path[d];
                ok = pd >= d && pd < a.n_q;
                if (ok) {
                    const int sb = table[(L + pd) / kBlockSize], db = table[(L + d) / kBlockSize];
                    ok = sb >= 0 && sb < a.num_blocks && db >= 0 && db < a.num_blocks;
                }
            }
            if (!ok) raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
        }
        s_ok = ok;
        s_L = L;
        s_k = k;
    }
    __syncthreads();
    if (!s_ok) return;
    const int L = s_L, k = s_k;

    if (a.path_nodes) {
        // move slot L + path[d] to slot L + d for d = 1..k, in increasing d
        // (a node's BFS index is at least its depth, so a source is never a
        // slot already written by an earlier step)
        const int32_t *path = a.path_nodes + (size_t)b * a.path_width;
        const int words = a.row_bytes / 16;  // 16-byte words per row
        for (int d = 1; d <= k; ++d) {
            const int src = L + path[d], dst = L + d;
            const int sb = table[src / kBlockSize], db = table[dst / kBlockSize];
            const int total = 2 * a.Hkv * words;
            for (int w = threadIdx.x; w < total; w += blockDim.x) {
                const int which = w / (a.Hkv * words);
                const int rem = w - which * a.Hkv * words;
                const int g = rem / words, x = rem - g * words;
                uint8_t *pool = which ? a.v_pool : a.k_pool;
                const size_t so = (((size_t)sb * a.Hkv + g) * kBlockSize + src % kBlockSize) * a.row_bytes;
                const size_t dof = (((size_t)db * a.Hkv + g) * kBlockSize + dst % kBlockSize) * a.row_bytes;
                reinterpret_cast<uint4 *>(pool + dof)[x] = reinterpret_cast<const uint4 *>(pool + so)[x];
            }
            __syncthreads();
        }
    }

    const int new_len = L + k + 1;
    const int keep = (new_len + kBlockSize - 1) / kBlockSize;
    const int had = (L + a.n_q + kBlockSize - 1) / kBlockSize;
    for (int i = keep + threadIdx.x; i < had; i += blockDim.x) {
        const int blk = table[i];
        if (blk < 0 || blk >= a.num_blocks) {
            raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
            continue;
        }
        table[i] = -1;
        const int old = atomicSub(&a.refcount[blk], 1);
        if (old == 1) {
            const int pos = atomicAdd(a.free_top, 1);
            if (pos < a.num_blocks) a.free_stack[pos] = blk;
            else raise_error(a.err, SVPA_DEVERR_FREE_OVERFLOW);
        } else if (old < 1) {
            raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        }
    }
    if (threadIdx.x == 0) a.context_lens[b] = new_len;
}

}  // namespace

cudaError_t launch_block_table_commit(const CommitArgs &a, cudaStream_t stream) {
    commit_kernel<<<a.B, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace svpa
