/*
 * tsv.h — C ABI of libtsv, token-tree speculative verification for GB300 (sm_103a).
 *
 * One LLM pass scores every node of a speculated token tree; this library runs
 * the data-parallel part of that pass and of the acceptance step:
 *
 *   tsv_tree_prepare            parent array -> per-node ancestor bitsets + depth
 *   tsv_tree_attention          every tree node attends to the shared prefix KV
 *                               plus its own ancestors (topology-aware mask)
 *   tsv_tree_verify_greedy      greedy acceptance walk over the tree
 *   tsv_tree_verify_stochastic  multi-step speculative sampling over the tree
 *   tsv_tree_verify_stochastic_warped  the same against a top-k / top-p warped LLM distribution
 *   tsv_tree_expand, tsv_tree_merge  token-tree construction on the GPU
 *   tsv_kv_commit               move the accepted path's K/V rows behind the prefix
 *
 * Sources: "SpecInfer: Accelerating Generative Large Language Model Serving
 * with Tree-based Speculative Inference and Verification" — §2 Overview (tree
 * verification: each token sees all its ancestors), §4 Token Tree Verifier
 * (Tree Attention; Tree-Based Parallel Decoding: one shared KV cache holding
 * verified and speculated tokens, topology-aware causal masking fused into one
 * kernel; Token Verification: multi-step speculative sampling), §6 Evaluation
 * (greedy verification reproduces incremental decoding); "Accelerating LLM
 * Inference with Staged Speculative Decoding" — §3 Methods, Implementation
 * (attention split between the KV cache and the in-batch tree, positions set
 * per tree node).
 *
 * Conventions for every call:
 *   - Trees.  A batch holds B requests; request b owns the N-array rows
 *     node_offsets[b] .. node_offsets[b+1]-1 (N = node_offsets[B]).  parent[]
 *     holds request-local indices in topological order: parent[i] == -1 (a
 *     root) or 0 <= parent[i] < i.  Any other value makes the request a bad
 *     tree: status_d[b] = TSV_ERR_BAD_TREE, its outputs are undefined, and no
 *     kernel traps.  Verification also needs exactly one root, at node 0; the
 *     root's token is the last already-verified token and is always on the
 *     path.  At most TSV_MAX_NODES nodes per request, TSV_MAX_BATCH requests.
 *   - KV cache.  Tree node i of request b lives at cache row prefix_len[b] + i
 *     (the caller has written it there before the call).  The library never
 *     appends to, moves or compacts the cache.
 *   - Memory.  The caller owns every buffer.  Pointers marked _d are device
 *     pointers, _host are host pointers read during the call only.  Scratch
 *     memory is a caller-provided device workspace whose size the matching
 *     *_workspace_size query returns.  Zero-fill a workspace once before its
 *     first use (it holds completion counters); every call that completes
 *     leaves them zero again, so it may be reused by later calls on one stream
 *     as is (re-zero it after a TSV_ERR_TIMEOUT).  Calls that overlap on the
 *     GPU must not share a workspace.
 *   - Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Calls are asynchronous on it.  The return value reports only the
 *     synchronous host-side checks and launch errors; device-side results and
 *     per-request errors are in status_d.
 *   - Errors.  Invalid arguments return TSV_ERR_INVALID_ARG before anything is
 *     launched; shapes the kernels do not implement return TSV_ERR_UNSUPPORTED;
 *     a CUDA launch error returns TSV_ERR_CUDA.  Device-side waits are bounded:
 *     a wait that runs out writes TSV_ERR_TIMEOUT to status_d and the kernel
 *     returns normally.
 */
#ifndef TSV_H_
#define TSV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TSV_MAX_NODES 256   /* nodes per request */
#define TSV_MAX_BATCH 128   /* requests per call */
#define TSV_ANC_WORDS 8     /* u32 words per ancestor bitset row (TSV_MAX_NODES / 32) */

typedef enum {
  TSV_OK = 0,
  TSV_ERR_INVALID_ARG = 1,
  TSV_ERR_BAD_TREE = 2,
  TSV_ERR_UNSUPPORTED = 3,
  TSV_ERR_CUDA = 4,
  TSV_ERR_TIMEOUT = 5,
  TSV_ERR_SCRATCH_LIMIT = 6  /* the call needs more than the fixed scratch of a _noalloc entry point */
} tsv_status;

typedef enum { TSV_F32 = 0, TSV_BF16 = 1 } tsv_dtype;

/* Flags for tsv_tree_attention. */
#define TSV_ATTN_DEFAULT 0u   /* bf16: tensor-core kernel; f32: CUDA-core kernel */
#define TSV_ATTN_SIMT 1u      /* force the CUDA-core kernel (any dtype) */

typedef struct tsv_handle_s* tsv_handle;

/* Human-readable name of a status code (static storage, never NULL). */
const char* tsv_status_string(int status);

/* ABI version of this library (major * 10000 + minor * 100 + patch). */
int tsv_version(void);

/*
 * Handle: caches the device's properties and the kernels' launch attributes.
 * tsv_create makes `device` current on the calling thread and must be called
 * before any other call on that device; returns TSV_ERR_CUDA when no such
 * device exists.  A handle may be used from one host thread at a time.
 */
tsv_status tsv_create(tsv_handle* out, int device);
tsv_status tsv_destroy(tsv_handle h);

/*
 * tsv_set_verify_overlap — how this handle's verification calls are ordered
 * against the kernel launched before them on the same stream.  `kinds` is a
 * set of flags; a call of a kind not in it (the default: none) waits for that
 * kernel's results before it reads.  A call of a kind in it starts while that
 * kernel still runs, in the CTAs its flag names below (the attention kernels'
 * trigger lets it launch once every attention CTA is resident), and completes
 * only after that kernel completes, so every later launch on the stream still
 * sees both finished.  The caller guarantees the call's inputs were complete
 * before that kernel began: the verification of one batch then runs in the
 * shadow of the attention launch of another.  Results are identical either
 * way, except that the full-size walk of TSV_OVERLAP_STOCHASTIC_FULL may run
 * in smaller clusters, whose sums go in another order: a decision within
 * rounding of a tie (what the oracle reports as a near tie) can then differ.
 *   TSV_OVERLAP_GREEDY       tsv_tree_verify_greedy (and _noalloc), in small
 *                            CTAs that fit on an SM beside a running
 *                            keys-on-lanes tree-attention CTA; while it is set,
 *                            a stochastic call in full-size CTAs also leaves
 *                            room for a greedy CTA beside each of them, so
 *                            greedy launched after it runs during its walk
 *   TSV_OVERLAP_STOCHASTIC   tsv_tree_verify_stochastic (unwarped; in two-warp
 *                            CTAs reading their slices from global memory, so
 *                            a walk is several times slower than alone: worth
 *                            it only when the kernel before it runs longer)
 *   TSV_OVERLAP_STOCHASTIC_FULL
 *                            tsv_tree_verify_stochastic (warped or not) in its
 *                            usual full-size CTAs, which need whole SMs, in
 *                            clusters of at most 4 so that they find room: for
 *                            a kernel before it that leaves SMs idle (the
 *                            rows-on-lanes tree attention on fewer units than
 *                            SMs) or frees them one by one as it ends (the
 *                            persistent tree attention's tail); the walk's
 *                            clusters start wherever SMs are free.  Takes
 *                            precedence over TSV_OVERLAP_STOCHASTIC.
 *   Takes effect for calls made (or captured into a CUDA graph) after it;
 *   TSV_ERR_INVALID_ARG for other bits.
 */
#define TSV_OVERLAP_GREEDY 1u
#define TSV_OVERLAP_STOCHASTIC 2u
#define TSV_OVERLAP_STOCHASTIC_FULL 4u
tsv_status tsv_set_verify_overlap(tsv_handle h, uint32_t kinds);

/*
 * tsv_tree_prepare — ancestor bitsets of every tree node (the topology-aware
 * causal mask of SpecInfer §4, Tree-Based Parallel Decoding, stored as one bit
 * per (node, tree key)).
 *   parent_d        int32 [N]       request-local parent indices
 *   node_offsets_d  int32 [B+1]     row ranges of the requests
 *   B               1 .. TSV_MAX_BATCH
 *   anc_d   (out)   uint32 [N][TSV_ANC_WORDS]: bit j of row i set iff node j is i
 *                   or an ancestor of i (bits >= n_b are zero)
 *   depth_d (out)   int32 [N]: number of strict ancestors (RoPE position of the
 *                   node is prefix_len[b] + depth[i]; positions are the caller's)
 *                   may be NULL
 *   status_d (out)  int32 [B]: TSV_OK or TSV_ERR_BAD_TREE (anc rows of a bad
 *                   request are zero)
 * Needs no workspace.  Run once per verification step; the result serves every
 * layer's tsv_tree_attention call.
 */
tsv_status tsv_tree_prepare(tsv_handle h, const int32_t* parent_d, const int32_t* node_offsets_d,
                            int32_t B, uint32_t* anc_d, int32_t* depth_d, int32_t* status_d,
                            void* stream);

/*
 * Workspace bytes tsv_tree_attention needs for this batch shape (depends on
 * the split of the prefix into chunks, which the call plans from the host
 * copies of prefix_len and node_offsets).  Returns TSV_ERR_INVALID_ARG on a bad
 * shape, TSV_ERR_UNSUPPORTED on a shape no kernel implements.
 */
tsv_status tsv_tree_attention_workspace_size(tsv_handle h, tsv_dtype dtype, int32_t B,
                                             const int32_t* prefix_len_host,
                                             const int32_t* node_offsets_host, int32_t Hq,
                                             int32_t Hkv, int32_t D, int anc_given,
                                             uint32_t flags, size_t* bytes);

/*
 * tsv_tree_attention — tree attention (SpecInfer §4 "Tree Attention"): for
 * request b, node i, query head h, KV head g = h / (Hq/Hkv),
 *   J(i)     = {0 .. P_b-1} U {P_b + a : a = i or an ancestor of i}
 *   out[i,h] = sum_{j in J(i)} softmax_j(scale * <q[i,h], k[b,j,g]>) v[b,j,g]
 * computed in one pass over the cache: each CTA streams a chunk of one KV
 * head's rows from HBM once for all tree nodes of the request, and chunks are
 * merged by their log-sum-exp (the cache / in-tree split of Staged Speculative
 * Decoding §3, generalised to any number of chunks).
 *   dtype              TSV_BF16 (tensor cores, fp32 accumulate) or TSV_F32
 *   q_d                [N, Hq, D] contiguous, dtype
 *   k_cache_d, v_cache_d  element (b, l, g, d) at b*kv_stride_b + l*kv_stride_l
 *                      + g*kv_stride_h + d (strides in elements; d contiguous).
 *                      Rows 0 .. prefix_len[b]+n_b-1 of request b are read;
 *                      other rows may hold anything (even NaN).  For bf16 the
 *                      base pointers must be 16-byte aligned and the strides
 *                      multiples of 8 elements.
 *   out_d       (out)  [N, Hq, D] contiguous, dtype
 *   prefix_len_host, node_offsets_host  host copies (used to plan the grid);
 *   prefix_len_d, node_offsets_d        the same values on the device
 *   parent_d           int32 [N]
 *   anc_d              from tsv_tree_prepare on the same parent_d (16-byte
 *                      aligned), or NULL: the bitsets are then computed from
 *                      parent_d inside the call, which also validates the tree
 *   B, Hq, Hkv, D      Hq % Hkv == 0, D in {64, 128}, Hq*N rows fit in int32;
 *                      the tensor-core path also needs Hq/Hkv to divide 128
 *                      (TSV_ERR_UNSUPPORTED otherwise)
 *   scale              softmax scale; 0 means 1/sqrt(D)
 *   workspace_d, workspace_bytes   at least tsv_tree_attention_workspace_size
 *   status_d    (out)  int32 [B]: TSV_OK or TSV_ERR_BAD_TREE when anc_d is NULL
 *                      (else left alone); TSV_ERR_TIMEOUT on a device-side
 *                      timeout
 *   flags              TSV_ATTN_DEFAULT or TSV_ATTN_SIMT
 */
tsv_status tsv_tree_attention(tsv_handle h, tsv_dtype dtype, const void* q_d, const void* k_cache_d,
                              const void* v_cache_d, int64_t kv_stride_b, int64_t kv_stride_l,
                              int64_t kv_stride_h, void* out_d, const int32_t* prefix_len_host,
                              const int32_t* node_offsets_host, const int32_t* prefix_len_d,
                              const int32_t* node_offsets_d, const int32_t* parent_d,
                              const uint32_t* anc_d, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                              float scale, void* workspace_d, size_t workspace_bytes,
                              int32_t* status_d, uint32_t flags, void* stream);

/* Workspace bytes for tsv_tree_verify_greedy on N rows of V logits. */
tsv_status tsv_tree_verify_greedy_workspace_size(tsv_handle h, int32_t B, int32_t N, int64_t V,
                                                 size_t* bytes);

/*
 * tsv_tree_verify_greedy — greedy token-tree verification (SpecInfer §4 Token
 * Tree Verification; §6: emits exactly the incremental-decoding tokens).  Row u
 * of logits is the LLM's next-token score after node u's sequence.
 *   u = 0; repeat { a = argmax logits[u] (lowest index on ties);
 *                   c = lowest-index child of u with tree_tokens[c] == a;
 *                   stop if none; u = c }; bonus = argmax at the stop node.
 *   logits_d        float32 [N, V] (finite values)
 *   tree_tokens_d   int32 [N]; parent_d int32 [N]; node_offsets_d int32 [B+1]
 *   path_d    (out) int32 [N]: request b's segment holds 0, then the accepted
 *                   nodes (request-local indices), then -1
 *   accept_len_d (out) int32 [B]: accepted nodes after the root
 *   bonus_d   (out) int32 [B]: the token emitted after the accepted ones
 *   status_d  (out) int32 [B]: TSV_OK or TSV_ERR_BAD_TREE (then path -1,
 *                   accept_len 0, bonus -1)
 * Emitted tokens of request b: tree_tokens[path[1 .. accept_len]] then bonus.
 */
tsv_status tsv_tree_verify_greedy(tsv_handle h, const float* logits_d, int64_t V,
                                  const int32_t* tree_tokens_d, const int32_t* parent_d,
                                  const int32_t* node_offsets_d, int32_t B, int32_t N,
                                  int32_t* path_d, int32_t* accept_len_d, int32_t* bonus_d,
                                  void* workspace_d, size_t workspace_bytes, int32_t* status_d,
                                  void* stream);

/* Workspace bytes for tsv_tree_verify_stochastic on N rows over a vocabulary of V. */
tsv_status tsv_tree_verify_stochastic_workspace_size(tsv_handle h, int32_t B, int32_t N, int64_t V,
                                                     size_t* bytes);

/*
 * tsv_tree_verify_stochastic — multi-step speculative sampling (SpecInfer §1
 * Correctness, §4 Token Verification): the emitted tokens follow the LLM's own
 * distribution.  p = softmax(llm_logits[u] / temperature); for each child c of
 * u in increasing index, x = tree_tokens[c], q = ssm_probs[c]:
 *   accept iff u_accept[c] * q[x] < p[x]      (probability min(1, p[x]/q[x]))
 *     -> move to c with p = softmax(llm_logits[c] / temperature)
 *   else p <- max(0, p - q) / sum(max(0, p - q))   (kept if that sum is 0)
 * With no child accepted the walk stops and the bonus token is the smallest x
 * with cumsum(p)[x] > u_sample[u] * sum(p).
 *   llm_logits_d    float32 [N, V], finite
 *   ssm_probs_d     float32 [N, V]: row c is the distribution node c's token
 *                   was drawn from (used as given, not renormalised)
 *   u_accept_d, u_sample_d  float32 [N] in [0, 1)
 *   temperature     > 0
 *   n_tried_d (out) int32 [B]: children tested (may be NULL)
 *   other arguments and outputs as in tsv_tree_verify_greedy.
 * Arithmetic is fp32 with compensated sums; a decision whose margin is below
 * about 1e-6 may go either way relative to an exact computation.
 */
tsv_status tsv_tree_verify_stochastic(tsv_handle h, const float* llm_logits_d,
                                      const float* ssm_probs_d, int64_t V,
                                      const int32_t* tree_tokens_d, const int32_t* parent_d,
                                      const int32_t* node_offsets_d, const float* u_accept_d,
                                      const float* u_sample_d, float temperature, int32_t B,
                                      int32_t N, int32_t* path_d, int32_t* accept_len_d,
                                      int32_t* bonus_d, int32_t* n_tried_d, void* workspace_d,
                                      size_t workspace_bytes, int32_t* status_d, void* stream);

/*
 * tsv_tree_verify_stochastic_warped — tsv_tree_verify_stochastic against the
 * warped LLM distribution that top-k / top-p sampling draws from (the pages'
 * evaluation samples with top-k): p = softmax(llm_logits[u] / temperature),
 * then
 *   top_k > 0    keep the top_k tokens of the ranking (larger logit first,
 *                equal logits by lower token index), all when top_k >= V;
 *   top_p < 1    then keep the shortest prefix of that ranking whose share of
 *                the kept mass reaches top_p;
 * and renormalise over the kept tokens, zero elsewhere.  Acceptance, residual
 * and bonus follow the same rules on this p, so the emitted tokens follow it.
 * ssm_probs rows are used as given: they are the proposal distributions the
 * proposer actually sampled from (warped or not).
 *   top_k   0 (off) or 1 .. 1024; top_p in (0, 1] (1 = off); top_p < 1 needs
 *           top_k >= 1 (TSV_ERR_UNSUPPORTED otherwise, as for top_k > 1024)
 *   other arguments, workspace and outputs as in tsv_tree_verify_stochastic.
 * A top-p cut within about 1e-6 of top_p may go either way relative to an
 * exact computation.
 */
tsv_status tsv_tree_verify_stochastic_warped(
    tsv_handle h, const float* llm_logits_d, const float* ssm_probs_d, int64_t V,
    const int32_t* tree_tokens_d, const int32_t* parent_d, const int32_t* node_offsets_d,
    const float* u_accept_d, const float* u_sample_d, float temperature, int32_t top_k, float top_p,
    int32_t B, int32_t N, int32_t* path_d, int32_t* accept_len_d, int32_t* bonus_d,
    int32_t* n_tried_d, void* workspace_d, size_t workspace_bytes, int32_t* status_d,
    void* stream);

/*
 * tsv_tree_expand — one expansion step of token-tree construction (SpecInfer
 * §3, expansion-based token trees: every node of the current frontier gets
 * the small model's top-k tokens as children).
 *   ssm_logits_d  float32 [F, V]: the small model's logits at the F frontier nodes
 *   k             1 .. min(V, 1024)
 *   tokens_d (out) int32 [F, k]: row f lists the k tokens of largest logit,
 *                 larger first, equal logits by lower token index; child j of
 *                 frontier node f carries tokens[f][j] (the caller appends the
 *                 children, F*k nodes, after the current tree)
 * Needs no workspace.
 */
tsv_status tsv_tree_expand(tsv_handle h, const float* ssm_logits_d, int64_t V, int32_t F, int32_t k,
                           int32_t* tokens_d, void* stream);

/*
 * tsv_tree_merge — merge-based token-tree construction (SpecInfer §3: the
 * trees of several speculators are merged into one token tree to verify).
 * All input trees of a request share its root (node 0 of each, the last
 * verified token; the first tree's root token is kept).  A node is identified
 * by its token path from the root, so nodes with equal paths become one.
 *   parent_d, tokens_d  int32 [M]: the input trees one after another, parent
 *                       indices local to each tree (parent[0] = -1, parent[i] < i)
 *   tree_offsets_d      int32 [T+1]: node range of input tree t
 *   request_trees_d     int32 [B+1]: input trees request_trees[b] .. [b+1]-1
 *                       belong to request b (at least one each)
 *   out_parent_d, out_tokens_d (out) int32 [M]: request b's union at rows
 *                       tree_offsets[request_trees[b]] .. + out_count[b] - 1,
 *                       in creation order (trees in order, nodes in order; a
 *                       node appears where its path is first seen, so parents
 *                       come first); the rest of the request's rows are -1
 *   out_source_d (out)  int32 [M]: the input node (row of parent_d) that
 *                       created each union node; may be NULL
 *   out_count_d (out)   int32 [B]
 *   status_d (out)      int32 [B]: TSV_OK, TSV_ERR_BAD_TREE (an input breaks
 *                       the tree rules), TSV_ERR_UNSUPPORTED (more than 1024
 *                       input nodes, or a union of more than TSV_MAX_NODES)
 * Needs no workspace.
 */
tsv_status tsv_tree_merge(tsv_handle h, const int32_t* parent_d, const int32_t* tokens_d,
                          const int32_t* tree_offsets_d, const int32_t* request_trees_d, int32_t B,
                          int32_t* out_parent_d, int32_t* out_tokens_d, int32_t* out_source_d,
                          int32_t* out_count_d, int32_t* status_d, void* stream);

/*
 * tsv_kv_commit — commits the accepted path to the KV cache (SpecInfer §4,
 * Token Tree Verifier: the verified and speculated tokens share one cache,
 * and the accepted tokens become the next part of the verified sequence).
 * Tree node i of request b sits at cache row prefix_len[b] + i; node 0 (the
 * root) is the last verified token.  For the path returned by verification,
 * path[0] = 0, path[1], ..., path[L] (L = accept_len[b]), row
 * prefix_len[b] + k receives the K and V rows of node path[k], k = 1 .. L, in
 * place; no other row changes.
 *   dtype, k_cache_d, v_cache_d, kv_stride_*, Hkv, D   as in tsv_tree_attention
 *                   (the caches are written); rows, strides and pointers must
 *                   be 16-byte aligned
 *   prefix_len_d    int32 [B]   device copy of the prefix lengths
 *   node_offsets_d  int32 [B+1]
 *   path_d          int32 [N]   per request as written by the verify calls
 *   accept_len_d    int32 [B]
 *   new_len_d (out) int32 [B]: prefix_len[b] + 1 + L, the verified length
 *                   (-1 when the request's path is rejected); may be NULL
 *   status_d (out)  int32 [B]: TSV_OK, or TSV_ERR_INVALID_ARG when the path
 *                   does not start at node 0, does not rise strictly or leaves
 *                   the request's nodes (that request's rows are not touched)
 * Needs no workspace.  Rows of rejected branches past prefix_len + L keep
 * whatever they held.
 */
tsv_status tsv_kv_commit(tsv_handle h, tsv_dtype dtype, void* k_cache_d, void* v_cache_d,
                         int64_t kv_stride_b, int64_t kv_stride_l, int64_t kv_stride_h, int32_t B,
                         int32_t Hkv, int32_t D, const int32_t* prefix_len_d,
                         const int32_t* node_offsets_d, const int32_t* path_d,
                         const int32_t* accept_len_d, int32_t* new_len_d, int32_t* status_d,
                         void* stream);

/*
 * tsv_tree_verify_greedy_noalloc — the same greedy verification as
 * tsv_tree_verify_greedy, for callers that cannot provide device scratch
 * memory: code running where it may not allocate (an engine or plugin whose
 * allocator owns all device memory, a latency-critical loop that must never
 * enter the CUDA allocator) or a binding with no device-memory management of
 * its own.  The pages describe no such interface; it has no counterpart there.
 *   Arguments and outputs as in tsv_tree_verify_greedy, without the workspace.
 *   Scratch: one fixed 1 MiB array in device memory, allocated when the library
 *   is loaded and held by every GPU that loads it until the process exits; this
 *   call allocates and frees nothing.  A shape whose scratch would exceed it
 *   returns TSV_ERR_SCRATCH_LIMIT (no shape within TSV_MAX_BATCH x
 *   TSV_MAX_NODES does).
 *   The first call on a device looks up the array's device address (a host-side
 *   set-up step, with that device current), and so does the first call after
 *   the device's context was reset (cudaDeviceReset): make each such call
 *   before any stream capture.
 *   All calls on a device share the array: each call clears the part that must
 *   start at zero on its stream, but calls that overlap on the GPU (streams not
 *   ordered with each other) race on it and give wrong results.
 */
tsv_status tsv_tree_verify_greedy_noalloc(tsv_handle h, const float* logits_d, int64_t V,
                                          const int32_t* tree_tokens_d, const int32_t* parent_d,
                                          const int32_t* node_offsets_d, int32_t B, int32_t N,
                                          int32_t* path_d, int32_t* accept_len_d, int32_t* bonus_d,
                                          int32_t* status_d, void* stream);

/*
 * tsv_selftest_bounded_wait — checks on the caller's device that a device-side
 * wait which never completes ends in TSV_ERR_TIMEOUT and a usable context,
 * not a hang.  The pages have no counterpart; it exercises the bounded wait
 * every kernel of this library uses for its mbarriers (about 1 s of wall
 * clock, then an abort flag that every other waiting role of the CTA sees).
 *   arrive          nonzero: the barriers are completed before the waits, so
 *                   they return at once and status is TSV_OK; zero: nothing
 *                   arrives, the waits run out and status is TSV_ERR_TIMEOUT
 *   status_d (out)  int32 [1]
 *   elapsed_ns_d (out)  int64 [1]: wall-clock nanoseconds from the start of
 *                   the waits to the status write; may be NULL
 * One CTA; allocates nothing; asynchronous on `stream`.
 */
tsv_status tsv_selftest_bounded_wait(tsv_handle h, int32_t arrive, int32_t* status_d,
                                     int64_t* elapsed_ns_d, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TSV_H_ */
