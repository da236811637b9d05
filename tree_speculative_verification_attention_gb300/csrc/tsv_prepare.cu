// tsv_prepare.cu — parent array -> per-node ancestor bitsets and depths.
//
// The topology-aware causal mask of SpecInfer (§4 Token Tree Verifier,
// Tree-Based Parallel Decoding) lets tree node i see tree key j iff j is i or
// one of i's ancestors (§2: each token's activations account for all of its
// ancestors).  It is stored as one bit per (node, tree key): TSV_ANC_WORDS u32
// words per node.  One CTA per request computes the reflexive-transitive
// closure of the parent relation by pointer jumping: after round k every node
// knows its ancestors within distance 2^k, so 8 rounds cover 256 nodes.
#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

__global__ void __launch_bounds__(TSV_MAX_NODES)
    tree_prepare_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                        uint32_t* __restrict__ anc, int32_t* __restrict__ depth,
                        int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ uint32_t A[2][TSV_MAX_NODES][TSV_ANC_WORDS];
  __shared__ int32_t J[2][TSV_MAX_NODES];
  __shared__ int bad;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  if (tid == 0) bad = (n < 0) ? 1 : (n > TSV_MAX_NODES ? 2 : 0);
  __syncthreads();
  if (bad == 0 && tid < n) {
    const int p = parent[off + tid];
    if (p < -1 || p >= tid) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (bad) {
    for (int i = tid; i < n; i += blockDim.x) {
      for (int w = 0; w < TSV_ANC_WORDS; ++w) anc[(size_t)(off + i) * TSV_ANC_WORDS + w] = 0u;
      if (depth) depth[off + i] = -1;
    }
    if (tid == 0) status[b] = (bad & 1) ? TSV_ERR_BAD_TREE : TSV_ERR_UNSUPPORTED;
    return;
  }
  const int i = tid;
  if (i < n) {
    const int p = parent[off + i];
#pragma unroll
    for (int w = 0; w < TSV_ANC_WORDS; ++w) A[0][i][w] = 0u;
    A[0][i][i >> 5] |= 1u << (i & 31);
    if (p >= 0) A[0][i][p >> 5] |= 1u << (p & 31);
    J[0][i] = p;
  }
  // Round r reads buffer r&1 and writes the other; after 8 rounds the result is in buffer 0.
#pragma unroll 1
  for (int r = 0; r < 8; ++r) {
    __syncthreads();
    const int cur = r & 1, nxt = cur ^ 1;
    if (i < n) {
      const int j = J[cur][i];
#pragma unroll
      for (int w = 0; w < TSV_ANC_WORDS; ++w) A[nxt][i][w] = A[cur][i][w] | (j >= 0 ? A[cur][j][w] : 0u);
      J[nxt][i] = j >= 0 ? J[cur][j] : -1;
    }
  }
  __syncthreads();
  if (i < n) {
    int pop = 0;
#pragma unroll
    for (int w = 0; w < TSV_ANC_WORDS; ++w) {
      anc[(size_t)(off + i) * TSV_ANC_WORDS + w] = A[0][i][w];
      pop += __popc(A[0][i][w]);
    }
    if (depth) depth[off + i] = pop - 1;
  }
  if (tid == 0) status[b] = TSV_OK;
}

cudaError_t launch_tree_prepare(const int32_t* parent, const int32_t* node_offsets, int32_t B,
                                uint32_t* anc, int32_t* depth, int32_t* status, cudaStream_t st) {
  return launch_pdl(tree_prepare_kernel, dim3(B), dim3(TSV_MAX_NODES), 0, st, 0u, parent, node_offsets, anc, depth,
                    status);
}

}  // namespace tsv
