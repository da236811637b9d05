// tsv_attention_common.cuh — pieces shared by the two tensor-core tree-attention
// kernels: named barriers and the per-block visibility mask built from an
// ancestor bitset.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

// Named barrier `id` (0 is __syncthreads) over `count` threads.
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

}  // namespace tsv
