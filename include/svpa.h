/*
 * svpa.h -- C ABI of libsvpa.so: the target-model verification step of
 * speculative decoding over a paged KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The operations of one verification step, in call order:
 *
 *   svpa_kv_append           write the n_q new K/V rows of every sequence into
 *                            its pages (block allocation, copy-on-write of a
 *                            shared page, FP8 requantisation).
 *   svpa_paged_verify_attn   the n_q verification queries of every sequence
 *                            (the last committed token plus the gamma drafts,
 *                            or the nodes of a draft tree) attend over the
 *                            sequence's K/V history, fetched page by page
 *                            through its block table.
 *   svpa_spec_accept         draft/target rejection sampling over the gamma
 *   svpa_spec_accept_tree    drafts (or along a draft tree): accepted count,
 *                            accepted tokens and the correction/bonus token.
 *   svpa_spec_accept_logits  the same from logits (the softmax rows formed
 *   svpa_spec_accept_tree_logits  in the kernel, at sampling temperatures).
 *   svpa_block_table_commit  commit the accepted tokens and roll back the
 *                            rest: new lengths, dropped pages returned to the
 *                            free stack when their reference count reaches 0.
 *   svpa_gamma_update        acceptance moving averages and the draft length
 *                            of the next step (with E[K] / speed-up telemetry).
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer unless its comment says HOST.
 *    The caller owns and allocates all memory; no entry point calls an
 *    allocator (the one fixed array the library holds, the scratch of
 *    svpa_paged_verify_attn_noalloc, is reserved when its module loads).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).  Arguments are validated on the
 *    host before anything is enqueued; a non-OK status means nothing ran.
 *  - Faults found on the device (a block id outside the pool, a free-stack
 *    overflow, a wait that ran out of time) are OR-ed into the caller's
 *    `error_flag` word (int32, device, zero before the call) as SVPA_DEVERR_*
 *    bits; kernels never trap.  svpa_check_error() synchronises the stream,
 *    reads the word and maps it to a status.
 *  - Calls that share buffers are not thread safe; order them on one stream.
 *  - Output of an operation whose error_flag came back non-zero is undefined.
 */
#ifndef SVPA_H
#define SVPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum svpa_status {
    SVPA_OK = 0,
    SVPA_ERR_INVALID_ARG = 1,   /* null pointer, bad size or shape            */
    SVPA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim)  */
    SVPA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed          */
    SVPA_ERR_OUT_OF_BLOCKS = 4, /* the free stack overflowed or ran empty
                                   (device)                                   */
    SVPA_ERR_BAD_BLOCK = 5,     /* a block id outside [0, num_blocks) (device)*/
    SVPA_ERR_WORKSPACE = 6,     /* workspace missing or too small             */
    SVPA_ERR_TIMEOUT = 7        /* a device-side wait gave up (device)        */
} svpa_status;

/* bits of the device error word */
#define SVPA_DEVERR_BAD_BLOCK 1
#define SVPA_DEVERR_TIMEOUT 2
#define SVPA_DEVERR_FREE_OVERFLOW 4 /* free stack overflowed (commit) or empty (append) */
#define SVPA_DEVERR_BAD_VALUE 8 /* an out-of-range length, count or token id */

/* K/V page element types */
#define SVPA_KV_BF16 0
#define SVPA_KV_FP8_E4M3 1

/*
 * Geometry of one paged-attention call.
 *
 * Source: "The Sub-Millisecond Speculative Decoding Meltdown", section
 * "Triton CUDA Fused Speculative Tree-Verification Kernel" (argument list:
 * query [B, H, K, D], K/V cache [blocks, heads, block_size, dim], K/V scales
 * [blocks, heads], block tables [B, pages per sequence], sm_scale); the
 * query/output layout here is [B, n_q, Hq, D] and kv heads are grouped
 * (query head h reads kv head h / (Hq / Hkv)).
 */
typedef struct svpa_attn_params {
    int32_t batch;              /* B >= 0                                     */
    int32_t n_q;                /* queries per sequence, 1..64 (gamma + 1, or
                                   the number of draft-tree nodes incl. root)  */
    int32_t num_q_heads;        /* Hq                                         */
    int32_t num_kv_heads;       /* Hkv, Hq % Hkv == 0, Hq / Hkv * n_q <= 128  */
    int32_t head_dim;           /* D: 64 or 128                               */
    int32_t block_size;         /* tokens per page: 16                        */
    int32_t max_blocks_per_seq; /* row stride of block_table                  */
    int32_t num_blocks;         /* physical pages in the pool                 */
    int32_t kv_dtype;           /* SVPA_KV_BF16 or SVPA_KV_FP8_E4M3           */
    float sm_scale;             /* softmax scale, normally 1/sqrt(D)          */
    int32_t split_pages;        /* pages per KV split; 0 = chosen by library
                                   (not used by the tcgen05 kernel for FP8
                                   pages)                                      */
    int32_t variant;            /* 0 = chosen by library; 1 = warp-level MMA
                                   kernel; 2 = tcgen05/TMEM kernel (head_dim
                                   128; FP8 pages with Hq / Hkv * n_q <= 64)   */
    int32_t scale_tile;         /* FP8 scale granularity: 0 = one scale per
                                   (page, kv head); 64 = one scale per 64
                                   consecutive elements of a token's row
                                   ("The Sub-Millisecond Speculative Decoding
                                   Meltdown", implementation checklist:
                                   block scales per 64-element tile), on the
                                   tcgen05 kernel only (head_dim 128,
                                   Hq / Hkv * n_q <= 64), else
                                   SVPA_ERR_UNSUPPORTED                        */
} svpa_attn_params;

/* The attention kernel svpa_paged_verify_attn runs for `p`: 1 = warp-level
 * MMA kernel, 2 = tcgen05/TMEM kernel (p->variant, or the library's choice
 * when p->variant is 0).  Same validation as svpa_attn_workspace_size. */
svpa_status svpa_attn_kernel(const svpa_attn_params *p, int32_t *kernel);

/* Kernel launches one svpa_paged_verify_attn call makes for `p`: 1, or 2
 * when the unsplit work units are first ranked longest sequence first.  Same
 * validation as svpa_attn_workspace_size. */
svpa_status svpa_attn_launches(const svpa_attn_params *p, int32_t *launches);

/* Bytes of workspace svpa_paged_verify_attn needs for `p` (split-KV partial
 * results, per-(sequence, kv head) tickets and, for unsplit work, the order
 * in which sequences are handed out: longest first).  The workspace must be
 * zero-filled once before its first use; every completed call leaves its
 * ticket words at zero again. */
svpa_status svpa_attn_workspace_size(const svpa_attn_params *p, size_t *bytes);

/*
 * Paged verification attention.
 *
 * Computes, for sequence b, query j and query head h,
 *   out[b][j][h] = softmax_p( q[b][j][h] . K[p] * sm_scale  over visible p ) . V
 * where the sequence's committed history has context_lens[b] = L_b tokens,
 * the n_q queries occupy positions L_b .. L_b + n_q - 1 (their K/V are
 * already written to the pool), position p lives in physical page
 * block_table[b][p / 16] at slot p % 16, and query j sees every p < L_b plus
 * the speculative slot L_b + i when bit i of ancestor_mask[j] is set
 * (causal when ancestor_mask is NULL: i <= j).
 *
 * Sources: "The Sub-Millisecond Speculative Decoding Meltdown", section
 * "Speculative Decoding Mechanics & The K-Token Penalty" (A = Softmax((Q K^T +
 * M_tree)/sqrt(d_k)) V with a tree mask) and section "Custom FP8 Quantized
 * Memory Block Layout" (e4m3 pages with per-block K and V scales);
 * "Speculative Decoding and KV-Cache Compression", section 2.3 (the bundle's
 * K/V are present before any acceptance decision).
 *
 *  q            bf16 [B, n_q, Hq, D]
 *  k_pool,
 *  v_pool       [num_blocks, Hkv, 16, D], bf16 or FP8-E4M3 (OCP "fn"
 *               encoding); 16-byte aligned
 *  k_scale,
 *  v_scale      fp32 [num_blocks, Hkv] (FP8 only; NULL for bf16): the real
 *               value of a stored byte x is e4m3(x) * scale[block][kv head];
 *               with scale_tile 64: fp32 [num_blocks, Hkv, 16, D / 64],
 *               16-byte aligned, the byte at (block, head, slot, d) scaled by
 *               scale[block][head][slot][d / 64]
 *  block_table  int32 [B, max_blocks_per_seq]; entries past a sequence's last
 *               page are ignored
 *  context_lens int32 [B], committed history L_b >= 0 with
 *               ceil((L_b + n_q) / 16) <= max_blocks_per_seq
 *  ancestor_mask HOST uint64 [n_q] or NULL (causal)
 *  out          bf16 [B, n_q, Hq, D] (written)
 *  lse          fp32 [B, n_q, Hq] natural-log sum of exp(scores), or NULL
 *  workspace    device scratch of at least svpa_attn_workspace_size() bytes
 * Accumulation is fp32; the contraction runs on the tensor cores.  FP8
 * pages on the tcgen05 kernel: the scores are an E4M3 MMA on the stored K
 * bytes against each query row split into two E4M3 terms at a power-of-two
 * scale of its own (any finite |q|); K scales multiply the scores in fp32
 * (any finite scale >= 0; with tile scales, each 64-dimension half of a
 * token's scores by its own scale); V is converted exactly to f16 and P
 * (at most 2^8 under the kernel's lazy maximum) is f16:
 *  - one scale per page (scale_tile 0): P times the V scale is formed in
 *    f16, so a V scale above 255 raises SVPA_DEVERR_BAD_VALUE;
 *  - one scale per 64-element tile (scale_tile 64): V is converted with its
 *    tile scales, so a V tile scale above 146 (448 * scale would pass the
 *    f16 maximum) raises SVPA_DEVERR_BAD_VALUE;
 * a negative or NaN scale raises it too.  split_pages is not used there:
 * the blocks of all (sequence, kv head) pairs are split evenly over the
 * GPU's SMs.  The warp-level kernel (variant 1) applies the scales in fp32
 * and has none of these limits.  The kernels cannot see the scales before they run,
 * so this is the caller's contract: with FP8 pages whose scales may pass
 * those limits, set variant = 1.
 */
svpa_status svpa_paged_verify_attn(const svpa_attn_params *p, const void *q,
                                   const void *k_pool, const void *v_pool,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_table,
                                   const int32_t *context_lens,
                                   const uint64_t *ancestor_mask, void *out,
                                   float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t *error_flag,
                                   void *stream);

/* Bytes of workspace the samplers take for `batch` rows of `vocab` tokens.
 * Reserved: the samplers keep no state in it (the size is 256 bytes); pass a
 * 16-byte aligned device buffer of at least that size. */
svpa_status svpa_spec_accept_workspace_size(int32_t batch, int32_t vocab,
                                            size_t *bytes);

/*
 * Linear draft/target rejection sampler, one row per sequence.
 *
 * For i = 0 .. gamma-1 draft x_i is accepted iff u_accept[i] * Q_i(x_i) <=
 * P_i(x_i), the product rounded once to fp32 (no fused multiply-add) -- the
 * realisation of alpha_i = min(1, P(x_i)/Q(x_i)); k = the first rejected
 * index, or gamma.  If k < gamma the emitted token is drawn from the residual
 * r = max(0, P_k - Q_k) (from P_k if r is all zero), else a bonus token is
 * drawn from P_gamma: the token is the first t whose running sum of r exceeds
 * u_sample * sum(r).
 *
 * Sources: "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING", section
 * "Verification Acceptance Probabilities and Speedup Math" (alpha_i) and its
 * architecture diagram ("Rejection Recovery (Resample)"); "Speculative
 * Decoding & KV-Cache PagedAttention in Enterprise LLM Serving", the
 * draft-verify pipeline figure (k accepted drafts plus one sampled correction
 * token); the residual distribution is the one that makes the output follow P
 * exactly ("Speculative Decoding and KV-Cache Compression", section 2.1).
 *
 *  p_probs      fp32 [B, gamma+1, V] target distributions (rows sum to ~1)
 *  q_probs      fp32 [B, gamma, V]   draft distributions
 *  draft_tokens int32 [B, gamma], each in [0, V)
 *  u_accept     fp32 [B, gamma] uniforms in [0, 1)
 *  u_sample     fp32 [B] uniforms in [0, 1)
 *  accepted_len int32 [B] (written) k in 0..gamma
 *  out_tokens   int32 [B, gamma+1] (written): x_0..x_{k-1}, the correction or
 *               bonus token, then -1
 *  near_boundary uint8 [B] or NULL: 1 when u_sample lay within 1e-6 of a
 *               boundary of the fp32 cumulative sum (a draw whose token fp32
 *               and exact arithmetic may resolve differently)
 *  gamma 1..32, V >= 1.
 */
svpa_status svpa_spec_accept(int32_t batch, int32_t gamma, int32_t vocab,
                             const float *p_probs, const float *q_probs,
                             const int32_t *draft_tokens,
                             const float *u_accept, const float *u_sample,
                             int32_t *accepted_len, int32_t *out_tokens,
                             uint8_t *near_boundary, void *workspace,
                             size_t workspace_bytes, int32_t *error_flag,
                             void *stream);

/*
 * The linear sampler fed by logits: P_i = softmax(target_logits_i / T) and
 * Q_i = softmax(draft_logits_i / T_draft) are formed inside the kernel and
 * never written out.  Q must be the distribution the drafts were drawn from.
 * Then the rule of svpa_spec_accept, with P(x) and Q(x) formed in fp32 as for
 * the residual (accept iff fp32(u * Q(x)) <= P(x)) and the residual
 * max(0, P_k - Q_k) formed in fp32.
 *
 * Sources: "Speculative Decoding and KV-Cache Compression", section 2.3 (the
 * acceptance ratio takes softmax(logits)[x] of the target pass); "LOW-LATENCY
 * INFERENCE: SPECULATIVE DECODING & PAGING", architecture (target logits
 * checked against draft logits); the same first page's alert table treats
 * the draft's temperature as its own knob.
 *
 *  temperature, draft_temperature  > 0 and finite (log2(e)/T must fit fp32)
 *  target_logits fp32 [B, gamma+1, V]; draft_logits fp32 [B, gamma, V]:
 *               finite or -inf (a masked token); every row needs a finite
 *               entry, else SVPA_DEVERR_BAD_VALUE is raised
 *  draft_tokens, u_accept, u_sample, accepted_len, out_tokens: as in
 *               svpa_spec_accept
 *  near_boundary uint8 [B] or NULL: 1 when a decision lay within 5e-5 of its
 *               threshold, where forming P and Q in fp32 (relative error up
 *               to ~2.5e-5) may decide it the other way: an acceptance test
 *               with |u Q - P| <= 5e-5 max(P, u Q), a residual of mass below
 *               5e-5, or u * (mass) within 5e-5 of a running sum.  With
 *               large vocabularies the running sums are closer together than
 *               that, so most draws are flagged.
 *  workspace    16-byte aligned device buffer of at least
 *               svpa_spec_accept_logits_workspace_size() bytes: the (max,
 *               sum) pair of every 8192-token slab of every row, written by
 *               the first kernel and read by the second
 *  gamma 1..32; 1 <= V <= 262144, else SVPA_ERR_UNSUPPORTED.
 * Two kernels on `stream`: the slab statistics (one CTA per slab of a row),
 * then the sampler clusters (a programmatic dependent launch of the first).
 */
svpa_status svpa_spec_accept_logits_workspace_size(int32_t batch, int32_t gamma,
                                                   int32_t vocab, size_t *bytes);

svpa_status svpa_spec_accept_logits(int32_t batch, int32_t gamma, int32_t vocab,
                                    float temperature, float draft_temperature,
                                    const float *target_logits,
                                    const float *draft_logits,
                                    const int32_t *draft_tokens,
                                    const float *u_accept, const float *u_sample,
                                    int32_t *accepted_len, int32_t *out_tokens,
                                    uint8_t *near_boundary, void *workspace,
                                    size_t workspace_bytes, int32_t *error_flag,
                                    void *stream);

/*
 * Draft-tree rejection sampler (recursive residual rejection over the
 * children of a node, in index order; identical to svpa_spec_accept on a
 * chain).  At a node: R = P[node], Z = 1; child c with token x_c is accepted
 * iff u_accept[c] * Q[node](x_c) * Z <= R(x_c) (for the first child this is
 * the fp32 test of svpa_spec_accept); on rejection R <- max(0, R - Z*Q[node])
 * and Z <- sum(R).  The walk descends into an accepted child; when every child
 * is rejected the correction token is drawn from R, and at a leaf a bonus
 * token is drawn from P[leaf], both with u_sample.
 *
 * Sources: "The Sub-Millisecond Speculative Decoding Meltdown" (draft trees
 * verified in one pass: "Tree-Attention Verification", "Draft Tree Rejection
 * Cascades"); the per-token rule of "LOW-LATENCY INFERENCE: SPECULATIVE
 * DECODING & PAGING".  The pages do not spell out the multi-child rule; this
 * is the recursive form that keeps the output distributed as P.
 *
 *  parent       HOST int32 [n_nodes]: parent[0] = -1, 0 <= parent[i] < i
 *  p_probs      fp32 [B, n_nodes, V]   target distribution at every node
 *  q_probs      fp32 [B, n_internal, V] draft distribution of the children of
 *               each internal node (a node with a child), in node order
 *  node_tokens  int32 [B, n_nodes] (entry 0 unused)
 *  u_accept     fp32 [B, n_nodes] (entry c drives child c's test)
 *  u_sample     fp32 [B]
 *  accepted_len int32 [B]; path_nodes int32 [B, W]; out_tokens int32 [B, W]
 *               with W = tree depth + 1: the root, the accepted nodes, -1...;
 *               the accepted tokens, the correction/bonus token, -1...
 *  near_boundary uint8 [B] or NULL: a later-child test or the final draw fell
 *               within 1e-6 (normalised units) of its threshold.
 *  n_nodes 1..64; V <= 262144 (the residual row is held in the shared memory
 *  of one thread-block cluster), else SVPA_ERR_UNSUPPORTED.
 */
svpa_status svpa_spec_accept_tree(int32_t batch, int32_t n_nodes, int32_t vocab,
                                  const int32_t *parent, const float *p_probs,
                                  const float *q_probs,
                                  const int32_t *node_tokens,
                                  const float *u_accept, const float *u_sample,
                                  int32_t *accepted_len, int32_t *path_nodes,
                                  int32_t *out_tokens, uint8_t *near_boundary,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *error_flag, void *stream);

/*
 * Draft-tree rejection sampler fed by logits: the recursion of
 * svpa_spec_accept_tree on P[node] = softmax(target_logits[node] /
 * temperature) and Q[node] = softmax(draft_logits[row of node] /
 * draft_temperature), formed in the kernel and never written out.  The walk
 * forms the softmax statistics (max and normaliser) of the rows it visits
 * only: one target row per node on the accepted path and the draft row of
 * each internal node on it, read from memory once for the statistics and
 * again (from L2) for a residual update or draw; the rows of nodes off the
 * path are never read.  Every test is made in fp32, P and Q formed as for
 * the residual: child c, after j rejected siblings, is accepted iff
 * u_accept[c] * Q(x_c) * Z <= R(x_c), with R = P, Z = 1 for the first child
 * (the products rounded in that order); the residual R <- max(0, R - Z Q) is
 * fp32 and its mass Z is summed in fp64.
 *
 * Sources: "Speculative Decoding and KV-Cache Compression", section 2.3 (the
 * acceptance ratio takes softmax(logits)[x]); "The Sub-Millisecond
 * Speculative Decoding Meltdown" (the target scores every node of the draft
 * tree in one pass); the multi-child rule as for svpa_spec_accept_tree.
 *
 *  parent       HOST int32 [n_nodes]: parent[0] = -1, 0 <= parent[i] < i
 *  target_logits fp32 [B, n_nodes, V]; -inf entries are masked tokens; a row
 *               the walk visits that has no finite entry, a NaN or +inf
 *               raises SVPA_DEVERR_BAD_VALUE
 *  draft_logits fp32 [B, n_internal, V]: the draft logits of the children of
 *               each internal node, in node order
 *  temperature, draft_temperature  > 0 and finite (log2(e)/T must be finite
 *               in fp32), else SVPA_ERR_INVALID_ARG
 *  node_tokens, u_accept, u_sample, accepted_len, path_nodes, out_tokens as
 *               for svpa_spec_accept_tree
 *  near_boundary uint8 [B] or NULL: 1 when a decision lay where forming P and
 *               Q in fp32 may take it the other way; after j rejected
 *               siblings the band is s_j = 2^(j+1) * 5e-5: a test with
 *               |u Q Z - R(x)| <= s_j max(P(x), Q(x)), a residual of mass
 *               below s_j, a draw with u * Z within s_j (within 5e-5 for a
 *               draw from P) of a running sum.
 *  n_nodes 1..64; V <= 262144, else SVPA_ERR_UNSUPPORTED.  Needs no
 *  workspace.  One kernel on `stream` (a thread-block cluster per sequence).
 */
svpa_status svpa_spec_accept_tree_logits(int32_t batch, int32_t n_nodes, int32_t vocab,
                                         const int32_t *parent, float temperature,
                                         float draft_temperature,
                                         const float *target_logits,
                                         const float *draft_logits,
                                         const int32_t *node_tokens,
                                         const float *u_accept, const float *u_sample,
                                         int32_t *accepted_len, int32_t *path_nodes,
                                         int32_t *out_tokens, uint8_t *near_boundary,
                                         int32_t *error_flag, void *stream);

/*
 * Commit the accepted tokens of every sequence and roll back the rest.
 *
 * With L = context_lens[b] and k = accepted_len[b] (0 <= k < n_q):
 *  - tree (path_nodes != NULL): for d = 1..k the K and V rows (all kv heads)
 *    of speculative slot L + path_nodes[b][d] are copied to slot L + d, so the
 *    accepted path becomes a linear continuation of the history;
 *  - context_lens[b] becomes L + k + 1 (the last committed token and the k
 *    accepted drafts; the correction/bonus token is written next step);
 *  - logical pages i with ceil((L+k+1)/16) <= i < ceil((L+n_q)/16) are
 *    dropped: block_table[b][i] = -1 and refcount[block] -= 1; a block whose
 *    count reaches 0 is pushed on the free stack (free_stack[(*free_top)++]).
 * The order of pushes within one call is unspecified.
 * A sequence whose length, k or tree path is invalid (path_nodes[b][d] < d or
 * >= n_q, k >= path_width, a page of the moved rows without a block) raises a
 * device error bit and is left untouched: no row moves, no page is dropped
 * and its length stays L.
 *
 * Sources: "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING",
 * architecture diagram (commit to the KV-cache block table; discard the KV
 * blocks of rejected tokens; rollback through block tables); "Speculative
 * Decoding & KV-Cache PagedAttention in Enterprise LLM Serving",
 * PagedKVCacheManager (reference counts, shared prefix blocks, release to the
 * free pool at count zero, block size 16).
 *
 *  block_table  int32 [B, max_blocks_per_seq] (in/out)
 *  context_lens int32 [B] (in/out)
 *  accepted_len int32 [B]
 *  refcount     int32 [num_blocks] (in/out)
 *  free_stack   int32 [num_blocks] (in/out), free_top int32 [1] (in/out)
 *  path_nodes   int32 [B, path_width] or NULL (linear)
 *  k_pool, v_pool  the pools (only read/written for a tree; bf16 only)
 */
svpa_status svpa_block_table_commit(int32_t batch, int32_t n_q,
                                    int32_t block_size,
                                    int32_t max_blocks_per_seq,
                                    int32_t num_blocks, int32_t *block_table,
                                    int32_t *context_lens,
                                    const int32_t *accepted_len,
                                    int32_t *refcount, int32_t *free_stack,
                                    int32_t *free_top,
                                    const int32_t *path_nodes,
                                    int32_t path_width, void *k_pool,
                                    void *v_pool, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t kv_dtype,
                                    int32_t *error_flag, void *stream);

/*
 * Append n_new K/V rows to every sequence's pages (the write that precedes
 * verification: the draft tokens' keys and values must be in the cache before
 * the verify attention reads them).
 *
 * Sources: "Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM
 * Serving", PagedKVCacheManager.EnsureCapacityAndAppendToken (a page past the
 * table's end comes from the free pool with reference count 1; a page whose
 * count is above 1 is cloned before the write and the shared block loses one
 * reference) and its shared-prefix section; "The Sub-Millisecond Speculative
 * Decoding Meltdown", "Custom FP8 Quantized Memory Block Layout" (E4M3 pages
 * with per-block K and V scales).
 *
 * With L = context_lens[b] (read only; svpa_block_table_commit sets the new
 * length), row t of sequence b goes to position L + t, t = 0..n_new-1, for
 * every kv head.  For each logical page i from L/16 to (L+n_new-1)/16:
 *  - block_table[b][i] == -1: a block is popped (free_stack[--*free_top]),
 *    its count set to 1 and stored in the table.  A page that holds history
 *    (i*16 < L) without a block raises SVPA_DEVERR_BAD_VALUE.
 *  - a mapped block whose count is above 1: when other sequences of the same
 *    call also write into it, exactly one of them (which one is unspecified)
 *    keeps it and writes in place; every other holder pops a fresh block,
 *    copies the whole page (and, for FP8, its two scales) into it, stores it
 *    in its table and the shared block loses one reference.  A block shared
 *    with a sequence outside the call is always cloned.
 *  - otherwise the rows are written in place.
 * Blocks popped, and which holder keeps a shared page, may differ from a
 * sequential pass in sequence order; each sequence's gathered content,
 * the counts of the blocks it maps and the number of blocks popped do not.
 *
 * FP8 pools (kv_dtype = SVPA_KV_FP8_E4M3) are requantised on write, per
 * (page, kv head) and separately for K and V:
 *   amax  = max |x| over the page's history values (stored code x current
 *           scale, one fp32 product) and the new bf16 values;
 *   scale = amax / 448 (one fp32 division; 1 when amax is 0);
 *   history codes are re-encoded from their values only when the scale
 *   changes; new codes = e4m3(x / scale), round to nearest even, saturating
 *   at +-448; slots past the last row of the page are set to 0.
 * FP8 pools with scale_tile 64 (one scale per 64 consecutive elements of a
 * row; scales [num_blocks, Hkv, 16, head_dim / 64]): each 64-value tile of a
 * new row gets scale = amax / 448 of its own values (1 when amax is 0) and
 * codes e4m3(value / scale); history rows keep their codes and scales; codes
 * past the last row are 0.  ("The Sub-Millisecond Speculative Decoding
 * Meltdown", implementation checklist: block scales per 64-element tile.)
 * bf16 pools receive the row bits unchanged; their slots past the last row
 * are left as they were.
 *
 *  new_k, new_v  bf16 [B, n_new, Hkv, D], 16-byte aligned
 *  block_table   int32 [B, max_blocks_per_seq] (in/out)
 *  context_lens  int32 [B]
 *  refcount      int32 [num_blocks] (in/out)
 *  free_stack    int32 [num_blocks] (in/out), free_top int32 [1] (in/out)
 *  k_pool, v_pool [num_blocks, Hkv, 16, D] bf16 or E4M3 bytes (in/out),
 *                16-byte aligned
 *  k_scale, v_scale fp32 [num_blocks, Hkv], or [num_blocks, Hkv, 16,
 *                head_dim / 64] with scale_tile 64 (in/out; FP8 only, else NULL)
 *  scale_tile    0, or 64 (FP8 with head_dim a multiple of 64)
 *  error_flag    int32 [1], zero before the call
 * Limits: 1 <= n_new <= 4096, 1 <= num_kv_heads <= 4096, block_size 16;
 * head_dim a multiple of 8 up to 1024 (bf16) or of 16 up to 256 (FP8); else
 * SVPA_ERR_INVALID_ARG before anything is enqueued.
 * Device errors: an empty free stack sets SVPA_DEVERR_FREE_OVERFLOW
 * (svpa_check_error: SVPA_ERR_OUT_OF_BLOCKS); a block id outside the pool
 * SVPA_DEVERR_BAD_BLOCK; a bad length or a mapped block with count 0
 * SVPA_DEVERR_BAD_VALUE.  When any bit is set no row is written; the blocks
 * already popped stay mapped with count 1, so tables, counts and the free
 * stack remain consistent.  Two kernels on `stream` (the second a
 * programmatic dependent launch of the first).
 */
svpa_status svpa_kv_append(int32_t batch, int32_t n_new, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size,
                           int32_t max_blocks_per_seq, int32_t num_blocks,
                           int32_t kv_dtype, int32_t scale_tile,
                           const void *new_k,
                           const void *new_v, int32_t *block_table,
                           const int32_t *context_lens, int32_t *refcount,
                           int32_t *free_stack, int32_t *free_top,
                           void *k_pool, void *v_pool, float *k_scale,
                           float *v_scale, int32_t *error_flag, void *stream);

/*
 * Acceptance telemetry and the adaptive draft length, from the accepted
 * lengths a sampler call left in device memory (no host round trip).
 *
 * Sources: "Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM
 * Serving" (the lookahead follows a moving-average acceptance rate: above
 * 0.85 -> 5 drafts, above 0.70 -> 4, above 0.50 -> 3, otherwise 2); "The
 * Sub-Millisecond Speculative Decoding Meltdown", production failure
 * scenarios (when the moving average collapses below 0.25, fall back to one
 * token) and its telemetry checklist; "LOW-LATENCY INFERENCE: SPECULATIVE
 * DECODING & PAGING", acceptance math (E[K], speed-up).
 *
 * A sequence that accepted k of gamma drafts ran k + (k < gamma) acceptance
 * tests.  Per sequence (when seq_state is given), in fp32 with every product
 * and sum rounded separately:
 *   A = decay * A + k;  N = decay * N + tests;  alpha = A / N
 *   seq_gamma_next[b] = 5 if alpha > 0.85, 4 if > 0.70, 3 if > 0.50,
 *                       2 if >= 0.25, else 1
 * The batch keeps its own (A, N) in batch_state, updated with the step's
 * integer totals (sum of k, sum of tests), and batch_gamma_next[0] is the
 * same table at its alpha (one draft length for the next call, whose kernels
 * take one n_q).  telemetry[4] (fp32): the batch alpha, the mean accepted
 * count of this step, E[K] = sum_{i=1..g} alpha^i and the speed-up
 * (E[K] + 1) / (g * draft_cost_ratio + 1) at the batch's g.
 *
 *  accepted_len     int32 [B] (from svpa_spec_accept / _tree)
 *  seq_state        fp32 [B][2] (A, N), in/out, zero for a new sequence; or NULL
 *  seq_gamma_next   int32 [B] or NULL (requires seq_state)
 *  batch_state      fp32 [2], in/out; batch_gamma_next int32 [1]; telemetry fp32 [4]
 *  decay            in [0, 1] (weight of the past; 0.9 in the Python binding)
 *  draft_cost_ratio r >= 0 (draft step time / target step time)
 * Limits: batch >= 1, 1 <= gamma <= 63; else SVPA_ERR_INVALID_ARG.  An
 * accepted length outside [0, gamma] sets SVPA_DEVERR_BAD_VALUE (the batch
 * state is then left unchanged).  One kernel (one CTA) on `stream`.
 */
svpa_status svpa_gamma_update(int32_t batch, int32_t gamma,
                              const int32_t *accepted_len, float *seq_state,
                              int32_t *seq_gamma_next, float *batch_state,
                              int32_t *batch_gamma_next, float *telemetry,
                              float decay, float draft_cost_ratio,
                              int32_t *error_flag, void *stream);

/*
 * svpa_paged_verify_attn without a caller workspace, for callers that may not
 * allocate device memory: code running inside a host framework that owns all
 * device allocations and forbids cudaMalloc/cudaFree on its hot path (an
 * allocation there can synchronise the device and fragments the framework's
 * pool), or plugin code that is handed only its input and output buffers.
 * The pages this library follows have no counterpart of this entry point.
 *
 * Same arguments and result as svpa_paged_verify_attn minus the workspace.
 * Its scratch is a fixed 32 MiB array inside the library, present on every
 * GPU that loads it until the process exits; a shape whose workspace
 * (svpa_attn_workspace_size) exceeds 32 MiB is rejected with
 * SVPA_ERR_WORKSPACE before anything is enqueued, as is any call that
 * svpa_paged_verify_attn would reject.  No call makes an allocation: no
 * cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current).  Under CUDA's lazy module loading
 *    (the default) that lookup loads the library's module on the device,
 *    and loading reserves the 32 MiB array there: the driver's one
 *    reservation for this entry point, which may block.  Make one call per
 *    device at initialisation (a batch of 0 does not count: it returns
 *    before the lookup), outside any stream capture, before the hot path.
 *  - Only the runtime's primary context of each device is supported (the
 *    address is cached per device index).
 *  - Every call on a device shares the one array and starts by clearing its
 *    counter words on `stream`; calls that overlap on the GPU (other streams,
 *    or other threads) race on it and must be serialised by the caller.
 */
svpa_status svpa_paged_verify_attn_noalloc(const svpa_attn_params *p, const void *q,
                                           const void *k_pool, const void *v_pool,
                                           const float *k_scale, const float *v_scale,
                                           const int32_t *block_table,
                                           const int32_t *context_lens,
                                           const uint64_t *ancestor_mask, void *out,
                                           float *lse, int32_t *error_flag,
                                           void *stream);

/* Synchronise `stream`, read the device error word and map it to a status
 * (SVPA_OK when it is zero).  Does not clear the word. */
svpa_status svpa_check_error(const int32_t *error_flag, void *stream);

/*
 * Diagnostic of the device-side wait limit.  Every wait inside the library's
 * kernels is bounded in wall time: when the limit passes, the kernel sets
 * SVPA_DEVERR_TIMEOUT in its error word, releases what it holds (tensor
 * memory, copies in flight) and returns, so the GPU stays usable and
 * svpa_check_error reports SVPA_ERR_TIMEOUT.  This call exercises that path on
 * purpose: one CTA allocates tensor memory, waits with the kernels' own
 * bounded mbarrier wait, under limit_ns, on a barrier that no thread ever
 * arrives on (no copy is in flight), frees the tensor memory and returns.
 * The pages this library follows have no counterpart of this entry point;
 * they name stalls in production ("The Sub-Millisecond Speculative Decoding
 * Meltdown", production failure scenarios) but no detection mechanism.
 *  limit_ns    the wait's limit, 1 ns .. 10 s (the kernels use 2 s)
 *  error_flag  int32 [1], device, zero before the call: SVPA_DEVERR_TIMEOUT
 *              is OR-ed in when the wait runs out (always, by construction)
 *  reached     int32 [1], device, zero before the call: 1 is added when the
 *              wait returned as timed out (2 if it had completed)
 * SVPA_ERR_INVALID_ARG for a null pointer or a limit outside that range.
 * One kernel of one CTA on `stream`.
 */
svpa_status svpa_wait_selftest(uint64_t limit_ns, int32_t *error_flag, int32_t *reached, void *stream);

/* Static description of a status code. */
const char *svpa_status_string(svpa_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t svpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SVPA_H */
