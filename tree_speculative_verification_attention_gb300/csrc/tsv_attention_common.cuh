// tsv_attention_common.cuh — pieces shared by the two tensor-core tree-attention
// kernels: named barriers, the per-block visibility mask built from an ancestor
// bitset, and the in-kernel ancestor computation by pointer jumping.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

// Named barriers (0 is __syncthreads).
constexpr int kBarSetup = 1;    // warps 0-3 + warp 5: TMEM address published
constexpr int kBarSoftmax = 2;  // warps 0-3

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Visibility of the 64 keys key0 .. key0+63 for one query row, given o =
// key0 - P (its tree index of column 0, may be negative) and the row's
// ancestor bitset (kAncWords words, zero past the tree).  Bit c set iff the
// key is in the prefix or is the node itself or one of its ancestors.
__device__ __forceinline__ uint64_t block_visibility(const uint32_t* arow, int o) {
  if (o >= 0) {
    const int w = o >> 5, sh = o & 31;
    const uint64_t lo = ((uint64_t)arow[w + 1] << 32) | arow[w];
    const uint64_t hi = arow[w + 2];
    return sh ? ((lo >> sh) | (hi << (64 - sh))) : lo;
  }
  const int pre = -o;  // columns 0 .. pre-1 are prefix keys
  if (pre >= 64) return ~0ull;
  const uint64_t tb = ((uint64_t)arow[1] << 32) | arow[0];
  return (tb << pre) | ((1ull << pre) - 1ull);
}

// Ancestor bitsets of all n nodes of a request, computed by the 128 softmax
// threads from parent[] (topological order) by pointer jumping: after round k
// each node holds its ancestors within distance 2^k.  Returns the buffer that
// holds the result; *bad is set when parent[] breaks the convention.
__device__ __forceinline__ const uint32_t* ancestors_by_pointer_jumping(
    const int32_t* __restrict__ par, int n, uint32_t* scratch, int* bad) {
  uint32_t* const A0 = scratch;
  uint32_t* const A1 = scratch + TSV_MAX_NODES * TSV_ANC_WORDS;
  int32_t* const J0 = reinterpret_cast<int32_t*>(scratch + 2 * TSV_MAX_NODES * TSV_ANC_WORDS);
  int32_t* const J1 = J0 + TSV_MAX_NODES;
  const int tid = threadIdx.x;
  for (int i = tid; i < n; i += 128) {
    const int p = __ldg(par + i);
    const bool ok = p >= -1 && p < i;
    if (!ok) atomicOr(bad, 1);
    const int pp = ok ? p : -1;
#pragma unroll
    for (int w = 0; w < TSV_ANC_WORDS; ++w) A0[i * TSV_ANC_WORDS + w] = 0u;
    A0[i * TSV_ANC_WORDS + (i >> 5)] |= 1u << (i & 31);
    if (pp >= 0) A0[i * TSV_ANC_WORDS + (pp >> 5)] |= 1u << (pp & 31);
    J0[i] = pp;
  }
  const int rounds = n > 1 ? 32 - __clz(n - 1) : 0;
  for (int r = 0; r < rounds; ++r) {
    named_bar(kBarSoftmax, 128);
    const uint32_t* Ac = (r & 1) ? A1 : A0;
    uint32_t* An = (r & 1) ? A0 : A1;
    const int32_t* Jc = (r & 1) ? J1 : J0;
    int32_t* Jn = (r & 1) ? J0 : J1;
    for (int i = tid; i < n; i += 128) {
      const int j = Jc[i];
#pragma unroll
      for (int w = 0; w < TSV_ANC_WORDS; ++w)
        An[i * TSV_ANC_WORDS + w] = Ac[i * TSV_ANC_WORDS + w] | (j >= 0 ? Ac[j * TSV_ANC_WORDS + w] : 0u);
      Jn[i] = j >= 0 ? Jc[j] : -1;
    }
  }
  named_bar(kBarSoftmax, 128);
  return (rounds & 1) ? A1 : A0;
}

}  // namespace tsv
