// tsv_internal.h — declarations shared by the library's translation units
// (launch wrappers and the attention work plan).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tsv.h"

namespace tsv {

constexpr int kBM = 128;  // query rows (node x head-in-group) per attention CTA = TMEM lanes
constexpr int kBN = 128;  // keys per pipeline block

// How one tsv_tree_attention call is cut into CTAs.  Passed by value as a
// kernel parameter (no host-to-device copy, so a launch can be captured).
// A unit (CTA) is (request b, KV head g, chunk c, M-tile mt); inside request b
// the unit index is ((g * n_chunks + c) * mtiles + mt), so the M-tiles of one
// KV chunk run next to each other and share its rows through L2.  Requests
// take consecutive unit ranges in slot order: slot s holds request
// slot_req[s], longest key range first, so that the block scheduler starts
// the longest CTAs first (longest-processing-time list scheduling).
struct AttnPlan {
  int32_t B, Hq, Hkv, G, D;
  int32_t n_units;
  int32_t chunk_keys;  // keys per chunk (multiple of kBN), same for every request
  float scale_log2;    // softmax scale * log2(e)
  int32_t unit_start[TSV_MAX_BATCH + 1];  // per slot
  int32_t slot_req[TSV_MAX_BATCH];
  int32_t n_chunks[TSV_MAX_BATCH];
  int32_t mtiles[TSV_MAX_BATCH];
  int32_t prefix[TSV_MAX_BATCH];
  int32_t nodes[TSV_MAX_BATCH];
  int32_t node_off[TSV_MAX_BATCH];
  int64_t part_row[TSV_MAX_BATCH];  // first partial row of request b, -1 when n_chunks == 1
  int32_t ctr_base[TSV_MAX_BATCH];  // first merge counter of request b (one per KV head x M-tile)
  int64_t part_rows_total;
  int32_t n_counters;
  // Keys-on-lanes kernel: every request is cut into n_chunks[b] == cluster
  // chunks of chunk_len[b] keys (a multiple of 128); the chunks of one (KV
  // head, M-tile) group are consecutive units and form one cluster.
  // Tile-pair rows kernel: cluster == n_chunks[b] (2 .. 8, the same for every
  // request) when the chunks of a (KV head, tile pair) merge in a cluster,
  // else 0.
  int32_t chunk_len[TSV_MAX_BATCH];
  int32_t cluster;
  int32_t keys_kernel;  // 1: keys-on-lanes kernel, 0: rows-on-lanes kernel
  // Keys-on-lanes kernel: every unit runs in the first wave (n_units <= SMs),
  // so each CTA pulls its first K/V blocks into L2 before waiting for the
  // previous kernel; with later waves the prefetch would only add traffic.
  int32_t prefetch_l2;
  // Keys-on-lanes kernel with one chunk per request and more units than SMs:
  // a persistent launch of `grid` CTAs (one per SM), each taking a sequence of
  // units, so that its producer streams the next unit's K/V while the key
  // lanes finish the previous unit.
  int32_t persistent;
  int32_t grid;
  // Rows-on-lanes kernel: 1 = two 128-row query tiles per CTA (units are
  // tile pairs), 0 = one tile per CTA (every request has mtiles <= 1).
  int32_t tc_tile_pairs;
};

// Launches a kernel with programmatic stream serialization (it may be
// scheduled while the previous kernel in the stream drains; the kernel waits
// for it with pdl_wait() before touching global memory) and, when cluster > 0,
// thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct Workspace {
  char* base;
  size_t size;
  size_t used;
  void* take(size_t bytes) {
    size_t off = (used + 255) & ~(size_t)255;
    if (off + bytes > size) return nullptr;
    used = off + bytes;
    return base + off;
  }
};

// Launch wrappers (defined next to their kernels); return the launch error.
cudaError_t launch_tree_prepare(const int32_t* parent, const int32_t* node_offsets, int32_t B,
                                uint32_t* anc, int32_t* depth, int32_t* status, cudaStream_t st);

cudaError_t launch_attention_tc(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const AttnPlan& plan,
                                const int32_t* parent, const uint32_t* anc, void* out,
                                float* part_o, float* part_lse, int32_t* counters,
                                int32_t* status, cudaStream_t st);
cudaError_t attention_tc_set_attributes(int D);
size_t attention_tc_smem_bytes(int D);
// The same with one query tile per CTA (plans with tc_tile_pairs == 0).
cudaError_t launch_attention_tc1(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                 const CUtensorMap& tmap_v, const AttnPlan& plan,
                                 const int32_t* parent, const uint32_t* anc, void* out,
                                 float* part_o, float* part_lse, int32_t* counters,
                                 int32_t* status, cudaStream_t st);
cudaError_t attention_tc1_set_attributes(int D);
size_t attention_tc1_smem_bytes(int D);

constexpr int kKeysBlockKeys = 128;  // keys per block of the keys-on-lanes kernel
constexpr int kKeysTileRows = 64;    // query rows per CTA of the keys-on-lanes kernel
constexpr int kKeysMaxUnitsPerCta = 48;  // units one CTA of a persistent keys launch may take
cudaError_t launch_attention_keys(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, const AttnPlan& plan,
                                  const int32_t* parent, const uint32_t* anc, void* out,
                                  int32_t* status, cudaStream_t st);
cudaError_t attention_keys_set_attributes(int D);
size_t attention_keys_smem_bytes(int D);

cudaError_t launch_attention_simt(bool bf16, const void* q, const void* k, const void* v,
                                  int64_t sb, int64_t sl, int64_t sh, void* out,
                                  const int32_t* prefix_len, const int32_t* node_offsets,
                                  const uint32_t* anc, int32_t B, int32_t N, int32_t Hq,
                                  int32_t Hkv, int32_t D, float scale, cudaStream_t st);

// Greedy verification: argmax over vocab slices folded into one 64-bit word
// per row, the last CTA of a request walks.
int greedy_splits(int64_t V, int32_t N, int num_sms);
cudaError_t launch_greedy_verify(const float* logits, int64_t V, int32_t N, int splits,
                                 const int32_t* tokens, const int32_t* parent,
                                 const int32_t* node_offsets, int32_t B, unsigned long long* rowbest,
                                 int32_t* counters, int32_t* path, int32_t* accept_len, int32_t* bonus,
                                 int32_t* status, int beside, cudaStream_t st);
cudaError_t launch_greedy_walk(unsigned long long* rowbest, const int32_t* tokens, const int32_t* parent,
                               const int32_t* node_offsets, int32_t B, int32_t* path,
                               int32_t* accept_len, int32_t* bonus, int32_t* status,
                               cudaStream_t st);

// Layout of a greedy verification workspace (the one tsv_tree_verify_greedy
// uses): B int32 completion counters, then N 64-bit row argmax words; both
// start at zero and every call leaves them at zero.
inline size_t greedy_counter_bytes(int32_t B) { return ((size_t)B * 4 + 255) & ~(size_t)255; }
inline size_t greedy_row_word_bytes(int32_t N) { return ((size_t)N * 8 + 255) & ~(size_t)255; }
inline size_t greedy_workspace_bytes(int32_t B, int32_t N) {
  return greedy_counter_bytes(B) + greedy_row_word_bytes(N);
}

// Stochastic verification: one cluster of mss_cluster_size(V, B, ...) CTAs
// per request, each owning a slice of the vocabulary.  `beside`: 0 waits for
// the previous kernel on the stream before reading; kMssBesideCompact and
// kMssBesideFull start beside it (two-warp CTAs that fit next to an attention
// CTA, or the full-size CTAs on SMs it leaves free) and complete after it.
// `room`: the full-size CTAs leave registers for a greedy CTA beside each.
constexpr int kMssClusterSizes = 9;  // entries of the resident-cluster table (sizes 0..8)
constexpr int kMssBesideCompact = 1, kMssBesideFull = 2;
// Largest cluster of the full-size CTAs beside a running kernel: a cluster
// needs that many idle SMs in one GPC, which a running grid seldom leaves
// (measured beside the GQA rows-on-lanes launch: clusters of 8 started only as
// it ended, clusters of 4 or 2 ran beside it).
constexpr int kMssBesideMaxCluster = 4;
int mss_cluster_size(int64_t V, int32_t B, const int* max_clusters, int cap);
cudaError_t launch_mss_verify(const float* llm_logits, const float* ssm_probs, int64_t V,
                              const int32_t* tokens, const int32_t* parent,
                              const int32_t* node_offsets, const float* u_acc, const float* u_smp,
                              float inv_t, int32_t top_k, float top_p, int32_t B, float* resid,
                              int32_t* path, int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                              int32_t* status, size_t staged_limit, const int* max_clusters,
                              int beside, int room, cudaStream_t st);
// Sets the MSS kernels' dynamic shared-memory limit on `device` to all that is
// left beside their static shared memory, returns the staged kernel's limit
// (the largest staged slice set a launch may use) and fills
// max_clusters[0..kMssClusterSizes-1] with the clusters of each size the
// device holds at once.
cudaError_t mss_set_attributes(int device, size_t* staged_limit, int* max_clusters);
constexpr int kMssMaxTopK = 1024;  // largest top_k of the warped stochastic verification

// Token-tree construction: expansion (top-k children per frontier row) and
// merge of several trees per request.
constexpr int kTreeMergeMaxInput = 1024;  // input nodes of one request's merge
cudaError_t launch_tree_expand(const float* logits, int64_t V, int32_t F, int32_t k, int32_t* tokens,
                               int num_sms, cudaStream_t st);
cudaError_t launch_tree_merge(const int32_t* parent, const int32_t* tokens, const int32_t* tree_offsets,
                              const int32_t* request_trees, int32_t B, int32_t* out_parent,
                              int32_t* out_tokens, int32_t* out_source, int32_t* out_count,
                              int32_t* status, cudaStream_t st);

// KV commit of the accepted path: rows hold row_chunks 16-byte chunks per
// cache row (Hkv x D x element size / 16); strides in bytes.
cudaError_t launch_kv_commit(uint8_t* k, uint8_t* v, int64_t sb, int64_t sl, int64_t sh, int32_t B,
                             int32_t Hkv, int32_t d_chunks, const int32_t* prefix_len,
                             const int32_t* node_offsets, const int32_t* path,
                             const int32_t* accept_len, int32_t* new_len, int32_t* status,
                             cudaStream_t st);

}  // namespace tsv
