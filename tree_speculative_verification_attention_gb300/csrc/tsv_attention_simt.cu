// tsv_attention_simt.cu — tree attention on CUDA cores.
//
// The fp32 path (tensor cores take no fp32 operands) and an independent
// cross-check of the tensor-core path for bf16.  One CTA per (node, query
// head); its four warps stride over the node's visible keys (the whole prefix,
// then the tree keys whose bit is set in the node's ancestor bitset), each lane
// owning D/32 dimensions; per-warp online softmax, merged across warps at the
// end.  SpecInfer §4 "Tree Attention" defines the result: attention over the
// token sequence the node stands for.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

namespace {

constexpr int kSimtWarps = 4;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32)
    tree_attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ kc,
                          const T* __restrict__ vc, int64_t sb, int64_t sl, int64_t sh,
                          T* __restrict__ out, const int32_t* __restrict__ prefix_len,
                          const int32_t* __restrict__ node_offsets,
                          const uint32_t* __restrict__ anc, int32_t B, int32_t Hq, int32_t Hkv,
                          float scale_log2) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  constexpr int E = D / 32;
  const int h = blockIdx.x;
  const int gi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Request of this node: last b with node_offsets[b] <= gi.
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (node_offsets[mid] <= gi) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  const int i = gi - off;
  const int P = prefix_len[b];
  const int g = h / (Hq / Hkv);

  float qv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) qv[e] = to_f(q[((size_t)gi * Hq + h) * D + lane * E + e]) * scale_log2;
  uint32_t bits[TSV_ANC_WORDS];
#pragma unroll
  for (int w = 0; w < TSV_ANC_WORDS; ++w) bits[w] = anc[(size_t)gi * TSV_ANC_WORDS + w];

  const T* kb = kc + (int64_t)b * sb + (int64_t)g * sh;
  const T* vb = vc + (int64_t)b * sb + (int64_t)g * sh;
  float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;

  auto visit = [&](int64_t row) {
    const T* kr = kb + row * sl + lane * E;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot += qv[e] * to_f(kr[e]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
    const float m_new = fmaxf(m, dot);
    const float alpha = exp2f(m - m_new);
    const float p = exp2f(dot - m_new);
    l = l * alpha + p;
    const T* vr = vb + row * sl + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * alpha + p * to_f(vr[e]);
    m = m_new;
  };
  for (int j = warp; j < P; j += kSimtWarps) visit(j);
  if (i < n && n <= TSV_MAX_NODES) {
    for (int j = warp; j < n; j += kSimtWarps)
      if ((bits[j >> 5] >> (j & 31)) & 1u) visit((int64_t)P + j);
  }

  __shared__ float sm_m[kSimtWarps], sm_l[kSimtWarps];
  __shared__ float sm_o[kSimtWarps][D];
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) sm_o[warp][lane * E + e] = o[e];
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, sm_m[w]);
    float L = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) {
      const float f = sm_m[w] == -INFINITY ? 0.f : exp2f(sm_m[w] - M);
      L += sm_l[w] * f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += sm_o[w][lane * E + e] * f;
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < E; ++e) out[((size_t)gi * Hq + h) * D + lane * E + e] = from_f<T>(acc[e] * inv);
  }
}

cudaError_t launch_attention_simt(bool bf16, const void* q, const void* k, const void* v,
                                  int64_t sb, int64_t sl, int64_t sh, void* out,
                                  const int32_t* prefix_len, const int32_t* node_offsets,
                                  const uint32_t* anc, int32_t B, int32_t N, int32_t Hq,
                                  int32_t Hkv, int32_t D, float scale, cudaStream_t st) {
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(Hq, N), block(kSimtWarps * 32);
  if (bf16) {
    using T = __nv_bfloat16;
    if (D == 64)
      return launch_pdl(tree_attn_simt_kernel<T, 64>, grid, block, 0, st, 0u,
          (const T*)q, (const T*)k, (const T*)v, sb, sl, sh, (T*)out, prefix_len,
          node_offsets, anc, B, Hq, Hkv, scale_log2);
    else
      return launch_pdl(tree_attn_simt_kernel<T, 128>, grid, block, 0, st, 0u,
          (const T*)q, (const T*)k, (const T*)v, sb, sl, sh, (T*)out, prefix_len,
          node_offsets, anc, B, Hq, Hkv, scale_log2);
  } else {
    using T = float;
    if (D == 64)
      return launch_pdl(tree_attn_simt_kernel<T, 64>, grid, block, 0, st, 0u,
          (const T*)q, (const T*)k, (const T*)v, sb, sl, sh, (T*)out, prefix_len,
          node_offsets, anc, B, Hq, Hkv, scale_log2);
    else
      return launch_pdl(tree_attn_simt_kernel<T, 128>, grid, block, 0, st, 0u,
          (const T*)q, (const T*)k, (const T*)v, sb, sl, sh, (T*)out, prefix_len,
          node_offsets, anc, B, Hq, Hkv, scale_log2);
  }
}

}  // namespace tsv
