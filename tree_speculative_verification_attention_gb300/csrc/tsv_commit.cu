// tsv_commit.cu — KV commit of the accepted path.
//
// After verification the accepted nodes path[1..L] of a request become the
// next L tokens of its verified sequence (SpecInfer §4, Token Tree Verifier:
// one cache holds the verified tokens and the speculated tree).  Tree node i
// sits at cache row P + i, so the commit copies row P + path[k] to row P + k
// for k = 1 .. L, in place, for K and V.
//
// grid (B, column blocks): a thread owns one 16-byte chunk of the (KV head, d)
// columns and walks k upwards.  In place is safe in that order: the path
// rises strictly, so path[k'] >= k' and a source row P + path[k'] never lies
// at or below an earlier destination P + k (k < k').  Eight rows are loaded
// before any of them is stored, for memory-level parallelism.
#include <cuda_runtime.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kCommitBatch = 8;

__global__ void __launch_bounds__(kCommitThreads)
    kv_commit_kernel(uint8_t* __restrict__ k, uint8_t* __restrict__ v, int64_t sb, int64_t sl,
                     int64_t sh, int32_t Hkv, int32_t d_chunks, const int32_t* __restrict__ prefix_len,
                     const int32_t* __restrict__ node_offsets, const int32_t* __restrict__ path,
                     const int32_t* __restrict__ accept_len, int32_t* __restrict__ new_len,
                     int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ int32_t spath[TSV_MAX_NODES];
  __shared__ int bad;
  const int b = blockIdx.x;
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  const int L = accept_len[b];
  const int P = prefix_len[b];
  if (threadIdx.x == 0) bad = (L < 0 || L >= n || n > TSV_MAX_NODES) ? 1 : 0;
  __syncthreads();
  if (!bad) {
    for (int i = threadIdx.x; i <= L; i += blockDim.x) spath[i] = path[off + i];
  }
  __syncthreads();
  if (!bad) {
    for (int i = threadIdx.x; i <= L; i += blockDim.x) {
      const int x = spath[i];
      const bool ok = (i == 0) ? (x == 0) : (x > spath[i - 1] && x < n);
      if (!ok) bad = 1;
    }
  }
  __syncthreads();
  if (blockIdx.y == 0 && threadIdx.x == 0) {
    if (new_len) new_len[b] = bad ? -1 : P + 1 + L;
    status[b] = bad ? TSV_ERR_INVALID_ARG : TSV_OK;
  }
  if (bad) return;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= Hkv * d_chunks) return;
  const int g = c / d_chunks, dc = c - g * d_chunks;
  const int64_t col = (int64_t)b * sb + (int64_t)g * sh + (int64_t)dc * 16;
  uint8_t* kc = k + col;
  uint8_t* vc = v + col;
  for (int k0 = 1; k0 <= L; k0 += kCommitBatch) {
    uint4 kr[kCommitBatch], vr[kCommitBatch];
#pragma unroll
    for (int u = 0; u < kCommitBatch; ++u) {
      const int kk = k0 + u;
      if (kk <= L && spath[kk] != kk) {
        const int64_t src = (int64_t)(P + spath[kk]) * sl;
        kr[u] = *reinterpret_cast<const uint4*>(kc + src);
        vr[u] = *reinterpret_cast<const uint4*>(vc + src);
      }
    }
#pragma unroll
    for (int u = 0; u < kCommitBatch; ++u) {
      const int kk = k0 + u;
      if (kk <= L && spath[kk] != kk) {
        const int64_t dst = (int64_t)(P + kk) * sl;
        *reinterpret_cast<uint4*>(kc + dst) = kr[u];
        *reinterpret_cast<uint4*>(vc + dst) = vr[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_commit(uint8_t* k, uint8_t* v, int64_t sb, int64_t sl, int64_t sh, int32_t B,
                             int32_t Hkv, int32_t d_chunks, const int32_t* prefix_len,
                             const int32_t* node_offsets, const int32_t* path,
                             const int32_t* accept_len, int32_t* new_len, int32_t* status,
                             cudaStream_t st) {
  const int chunks = Hkv * d_chunks;
  dim3 grid(B, (chunks + kCommitThreads - 1) / kCommitThreads);
  return launch_pdl(kv_commit_kernel, grid, dim3(kCommitThreads), 0, st, 0u, k, v, sb, sl, sh, Hkv, d_chunks,
                    prefix_len, node_offsets, path, accept_len, new_len, status);
}

}  // namespace tsv
