// tsv_verify.cu — token-tree verification kernels.
//
// Greedy (SpecInfer §4 Token Tree Verification; §6: the output equals
// incremental decoding):
//   greedy_verify_kernel   grid (splits, N): each CTA streams one vocab slice
//                          of one logits row with 16-byte loads and reduces
//                          (max, lowest index) with warp shuffles; the last
//                          CTA of each request merges the slices per row, marks
//                          for every node u its next node = the lowest-index
//                          child whose token is argmax(u), and follows those
//                          links from the root.
// Stochastic, multi-step speculative sampling (SpecInfer §1 Correctness, §4
// Token Verification):
//   mss_verify_kernel      one cluster of up to 8 CTAs per request, each CTA
//                          owning a slice of the vocabulary.  The walk is
//                          sequential; every vocab-wide step in it is split
//                          over the cluster: the softmax statistics of each
//                          row the walk visits (only those rows are read), the
//                          residual pass max(0, p - q) after a rejection, and
//                          the inverse-CDF draw of the bonus token.  Partial
//                          results meet in distributed shared memory.
#include <float.h>
#include <math.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kMinSlice = 4096;  // vocab entries per CTA at least

struct ArgMax {
  float v;
  int32_t i;
};

// Larger value wins; equal values go to the lower index.
__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = better(a, b);
  }
  return a;
}

__device__ __forceinline__ int64_t slice_len(int64_t V, int splits) {
  int64_t per = (V + splits - 1) / splits;
  return (per + 3) & ~int64_t(3);
}

}  // namespace

// Argmax (lowest index on ties) of vocab slice s of logits row `row`, reduced
// over the CTA; the result is valid in thread 0.  `red` holds one entry per warp.
__device__ __forceinline__ ArgMax slice_argmax(const float* __restrict__ logits, int64_t V, int splits,
                                               int row, int s, ArgMax* red) {
  const int64_t per = slice_len(V, splits);
  const int64_t lo = (int64_t)s * per;
  const int64_t hi = min(V, lo + per);
  const float* x = logits + (size_t)row * (size_t)V;
  ArgMax best{-INFINITY, INT32_MAX};
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t lo4 = lo >> 2, hi4 = hi >> 2;
    int64_t k = lo4 + threadIdx.x;
    // Four independent 16-byte loads in flight per thread.
    for (; k + 3 * kArgmaxThreads < hi4; k += 4 * kArgmaxThreads) {
      float4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = __ldcs(x4 + k + u * kArgmaxThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int32_t base = (int32_t)((k + u * kArgmaxThreads) << 2);
        best = better(best, ArgMax{a[u].x, base});
        best = better(best, ArgMax{a[u].y, base + 1});
        best = better(best, ArgMax{a[u].z, base + 2});
        best = better(best, ArgMax{a[u].w, base + 3});
      }
    }
    for (; k < hi4; k += kArgmaxThreads) {
      const float4 a = __ldcs(x4 + k);
      const int32_t base = (int32_t)(k << 2);
      best = better(best, ArgMax{a.x, base});
      best = better(best, ArgMax{a.y, base + 1});
      best = better(best, ArgMax{a.z, base + 2});
      best = better(best, ArgMax{a.w, base + 3});
    }
  } else {
    for (int64_t k = lo + threadIdx.x; k < hi; k += kArgmaxThreads)
      best = better(best, ArgMax{__ldcs(x + k), (int32_t)k});
  }
  best = warp_argmax(best);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = best;
  __syncthreads();
  if (warp == 0) {
    best = lane < kArgmaxThreads / 32 ? red[lane] : ArgMax{-INFINITY, INT32_MAX};
    best = warp_argmax(best);
  }
  return best;
}

// Validates one request's tree for verification: a single root at node 0,
// every other parent earlier in the order.  Returns a TSV status.
__device__ int validate_verify_tree(const int32_t* par_g, int n, int* bad_flag) {
  if (threadIdx.x == 0) *bad_flag = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
  __syncthreads();
  if (*bad_flag == 0) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int p = par_g[i];
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
      if (!ok) atomicMax(bad_flag, TSV_ERR_BAD_TREE);
    }
  }
  __syncthreads();
  return *bad_flag;
}

__device__ void fail_request(int32_t* path, int n, int32_t* accept_len, int32_t* bonus,
                             int32_t* n_tried, int32_t* status, int code) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) path[i] = -1;
  if (threadIdx.x == 0) {
    *accept_len = 0;
    *bonus = -1;
    if (n_tried) *n_tried = 0;
    *status = code;
  }
}

// Shared scratch of one greedy walk: the request's parents, tokens and
// per-node results, and its (row, slice) argmax partials when they fit.
constexpr int kWalkPartials = 1024;
struct WalkSmem {
  int32_t par[TSV_MAX_NODES];
  int32_t tok[TSV_MAX_NODES];
  int32_t am[TSV_MAX_NODES];
  int32_t nxt[TSV_MAX_NODES];
  ArgMax part[kWalkPartials];
  int bad, len;
};

// The greedy walk of request b from its per-slice argmax partials: every
// child c whose token equals argmax(parent(c)) proposes itself to its parent
// with atomicMin (lowest index wins), then the chain is followed from the root.
// Parents, tokens and partials are loaded in one parallel step.  Run by one
// whole CTA of up to 256 threads.
__device__ void greedy_walk_request(int b, int off, int n, const float* part_val,
                                    const int32_t* part_idx, int splits, const int32_t* tokens,
                                    const int32_t* parent, int32_t* path, int32_t* accept_len,
                                    int32_t* bonus, int32_t* status, WalkSmem& w) {
  const int T = blockDim.x;
  if (threadIdx.x == 0) w.bad = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
  __syncthreads();
  const int items = n * splits;  // rows of a request are consecutive, so its partials are too
  const bool staged = items <= kWalkPartials;
  if (w.bad == 0) {
    for (int i = threadIdx.x; i < n; i += T) {
      w.par[i] = parent[off + i];
      w.tok[i] = tokens[off + i];
    }
    if (staged)
      for (int i = threadIdx.x; i < items; i += T)
        w.part[i] = ArgMax{__ldcg(part_val + (size_t)off * splits + i), __ldcg(part_idx + (size_t)off * splits + i)};
  }
  __syncthreads();
  if (w.bad == 0) {
    for (int i = threadIdx.x; i < n; i += T) {
      const int p = w.par[i];
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
      if (!ok) atomicMax(&w.bad, TSV_ERR_BAD_TREE);
    }
  }
  __syncthreads();
  if (w.bad) {
    fail_request(path + off, n, accept_len + b, bonus + b, nullptr, status + b, w.bad);
    return;
  }
  for (int u = threadIdx.x; u < n; u += T) {
    ArgMax best{-INFINITY, INT32_MAX};
    for (int s = 0; s < splits; ++s) {
      const size_t k = (size_t)(off + u) * splits + s;
      best = better(best, staged ? w.part[u * splits + s] : ArgMax{__ldcg(part_val + k), __ldcg(part_idx + k)});
    }
    w.am[u] = best.i;
    w.nxt[u] = INT32_MAX;
  }
  __syncthreads();
  for (int c = 1 + threadIdx.x; c < n; c += T) {
    const int p = w.par[c];
    if (w.tok[c] == w.am[p]) atomicMin(&w.nxt[p], c);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int u = 0, len = 0;
    path[off + len++] = 0;
    while (w.nxt[u] != INT32_MAX) {
      u = w.nxt[u];
      path[off + len++] = u;
    }
    accept_len[b] = len - 1;
    bonus[b] = w.am[u];
    status[b] = TSV_OK;
    w.len = len;
  }
  __syncthreads();
  for (int i = w.len + threadIdx.x; i < n; i += T) path[off + i] = -1;
}

// Walk-only kernel: one CTA per request (used when N == 0, where no argmax CTA exists).
__global__ void __launch_bounds__(TSV_MAX_NODES)
    greedy_walk_kernel(const float* __restrict__ part_val, const int32_t* __restrict__ part_idx,
                       int splits, const int32_t* __restrict__ tokens,
                       const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                       int32_t* __restrict__ path, int32_t* __restrict__ accept_len,
                       int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  __shared__ WalkSmem w;
  const int b = blockIdx.x;
  const int off = node_offsets[b];
  greedy_walk_request(b, off, node_offsets[b + 1] - off, part_val, part_idx, splits, tokens, parent,
                      path, accept_len, bonus, status, w);
}

// Fused greedy verification: grid (splits, N).  Each CTA reduces one vocab
// slice of one row; the last CTA to finish among a request's rows x slices
// (atomic counter, no waiting) walks that request's tree.  CTA (0, 0) also
// reports requests that own no rows.  Counters start at zero and are reset.
__global__ void __launch_bounds__(kArgmaxThreads)
    greedy_verify_kernel(const float* __restrict__ logits, int64_t V, int splits,
                         const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                         const int32_t* __restrict__ node_offsets, int B,
                         float* __restrict__ part_val, int32_t* __restrict__ part_idx,
                         int32_t* __restrict__ counters, int32_t* __restrict__ path,
                         int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                         int32_t* __restrict__ status) {
  __shared__ int32_t offs[TSV_MAX_BATCH + 1];
  __shared__ WalkSmem w;
  __shared__ ArgMax red[kArgmaxThreads / 32];
  __shared__ int last;
  const int row = blockIdx.y, s = blockIdx.x;
  for (int i = threadIdx.x; i <= B; i += blockDim.x) offs[i] = node_offsets[i];
  const ArgMax best = slice_argmax(logits, V, splits, row, s, red);
  if (threadIdx.x == 0) {
    part_val[(size_t)row * splits + s] = best.v;
    part_idx[(size_t)row * splits + s] = best.i;
  }
  __syncthreads();  // offs loaded
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offs[mid] <= row) lo = mid; else hi = mid;
  }
  while (lo + 1 < B && offs[lo + 1] <= row) ++lo;  // skip empty requests sharing the offset
  const int b = lo;
  const int off = offs[b], n = offs[b + 1] - off;
  if (row == 0 && s == 0) {
    for (int e = threadIdx.x; e < B; e += blockDim.x)
      if (offs[e + 1] == offs[e]) {
        accept_len[e] = 0;
        bonus[e] = -1;
        status[e] = TSV_ERR_BAD_TREE;
      }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(counters + b, 1) == n * splits - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  greedy_walk_request(b, off, n, part_val, part_idx, splits, tokens, parent, path, accept_len, bonus,
                      status, w);
  if (threadIdx.x == 0) counters[b] = 0;
}

int greedy_splits(int64_t V, int32_t N, int num_sms) {
  int64_t s = (2LL * num_sms + N - 1) / (N > 0 ? N : 1);
  const int64_t cap = (V + kMinSlice - 1) / kMinSlice;
  s = s < cap ? s : cap;
  return (int)(s < 1 ? 1 : s);
}

cudaError_t launch_greedy_verify(const float* logits, int64_t V, int32_t N, int splits,
                                 const int32_t* tokens, const int32_t* parent,
                                 const int32_t* node_offsets, int32_t B, float* part_val,
                                 int32_t* part_idx, int32_t* counters, int32_t* path,
                                 int32_t* accept_len, int32_t* bonus, int32_t* status,
                                 cudaStream_t st) {
  dim3 grid(splits, N);
  greedy_verify_kernel<<<grid, kArgmaxThreads, 0, st>>>(logits, V, splits, tokens, parent,
                                                        node_offsets, B, part_val, part_idx,
                                                        counters, path, accept_len, bonus, status);
  return cudaGetLastError();
}

cudaError_t launch_greedy_walk(const float* part_val, const int32_t* part_idx, int splits,
                               const int32_t* tokens, const int32_t* parent,
                               const int32_t* node_offsets, int32_t B, int32_t* path,
                               int32_t* accept_len, int32_t* bonus, int32_t* status,
                               cudaStream_t st) {
  greedy_walk_kernel<<<B, TSV_MAX_NODES, 0, st>>>(part_val, part_idx, splits, tokens, parent,
                                                  node_offsets, path, accept_len, bonus, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ stochastic

namespace {

constexpr int kMssThreads = 256;
constexpr int kMssWarps = kMssThreads / 32;
constexpr int kMssMaxCluster = 8;
constexpr int64_t kMssMinSlice = 4096;  // vocab entries per CTA at least
constexpr int kMssGroups = 4;           // 4-float groups in flight per thread

// exp(a - m) with the subtraction's rounding error folded back in (TwoSum:
// a - m = d + err exactly), so the result is as accurate as expf itself even
// when a - m is large in magnitude.  Requires finite a and m.
__device__ __forceinline__ float exp_diff(float a, float m) {
  const float d = a - m;
  const float bb = d - a;
  const float err = (a - (d - bb)) + (-m - bb);
  return expf(d) * (1.0f + err);
}

// Sums are carried as unevaluated pairs of floats, hi + lo with |lo| at most
// half an ulp of hi (about 44 significant bits), built from the error-free
// TwoSum and FMA-based product transformations.  This GPU's fp64 rate is a
// small fraction of its fp32 rate, so the walk keeps fp64 out of its loops.
struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const F2 s = two_sum(a.hi, b.hi);
  return two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ F2 f2_scale(F2 a, float f) {  // a * f
  const float p = __fmul_rn(a.hi, f);
  const float e = fmaf(a.hi, f, -p);  // exact: a.hi * f = p + e
  return two_sum(p, fmaf(a.lo, f, e));
}

__device__ __forceinline__ bool f2_lt(F2 a, F2 b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// 1 / (hi + lo), to about one ulp.
__device__ __forceinline__ float f2_inv(F2 a) {
  const float r = 1.0f / a.hi;
  return fmaf(-__fmul_rn(r, a.lo), r, r);
}

__device__ __forceinline__ F2 comp_value(const CompSum& c) { return two_sum(c.s, c.c); }

__device__ __forceinline__ F2 shfl_xor_f2(F2 v, int o) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

// Block-wide sum of a pair sum and two plain floats (every thread gets them;
// the floats are sums of one nonzero value and zeros, so exact).
// `red` holds 4 x 32 floats.
__device__ void block_sum(F2& a, float& b, float& c, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = f2_add(a, shfl_xor_f2(a, o));
    b += __shfl_xor_sync(0xffffffffu, b, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
  }
  __syncthreads();  // red is free
  if (lane == 0) {
    red[warp] = a.hi;
    red[32 + warp] = a.lo;
    red[64 + warp] = b;
    red[96 + warp] = c;
  }
  __syncthreads();
  // Every warp adds the per-warp values in warp order: the same result everywhere.
  a = F2{0.f, 0.f};
  b = 0.f;
  c = 0.f;
  for (int w = 0; w < kMssWarps; ++w) {
    a = f2_add(a, F2{red[w], red[32 + w]});
    b += red[64 + w];
    c += red[96 + w];
  }
}

__device__ float block_max(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = -INFINITY;
  for (int w = 0; w < kMssWarps; ++w) v = fmaxf(v, red[w]);
  return v;
}

// Four consecutive floats at p[y] (16-byte load when rows are 16-byte aligned).
template <int kind>  // 0: read-only, 1: streamed once, 2: read-write scratch
__device__ __forceinline__ float4 load4(const float* p, int64_t y, bool vec) {
  if (vec) {
    const float4* q = reinterpret_cast<const float4*>(p + y);
    return kind == 0 ? __ldg(q) : kind == 1 ? __ldcs(q) : *q;
  }
  return make_float4(p[y], p[y + 1], p[y + 2], p[y + 3]);
}

__device__ __forceinline__ float at(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// u * q < p exactly, for floats u, q >= 0 and p (the product is formed
// without rounding as p0 + e).
__device__ __forceinline__ bool accept_test(float u, float q, float p) {
  const float p0 = __fmul_rn(u, q);
  const float e = fmaf(u, q, -p0);
  return p0 < p || (p0 == p && e < 0.f);
}

}  // namespace

// Multi-step speculative sampling: one cluster of `ncl` CTAs per request, CTA
// rank r owning vocab slice r.  All walk decisions are taken identically by
// every CTA from values every CTA holds: the children, their tokens, accept
// uniforms, proposal probabilities q_c(x_c) and parent logits l(x_c) (read
// once, in parallel, at the start), the row statistics and residual sums
// (combined in rank order through distributed shared memory), and p at the
// next child's token, which the residual pass of the CTA owning that token
// publishes with the sums.  A CTA streams only its own slice of the logits,
// proposals and residual rows.
__global__ void __launch_bounds__(kMssThreads, 2)
    mss_verify_kernel(const float* __restrict__ llm_logits, const float* __restrict__ ssm_probs,
                      int64_t V, const int32_t* __restrict__ tokens,
                      const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                      const float* __restrict__ u_acc, const float* __restrict__ u_smp, float inv_t,
                      int ncl, int vec, float* __restrict__ resid_all, int32_t* __restrict__ path,
                      int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                      int32_t* __restrict__ n_tried, int32_t* __restrict__ status) {
  __shared__ int32_t first_child[TSV_MAX_NODES];
  __shared__ int32_t next_sib[TSV_MAX_NODES];
  __shared__ int32_t tok_s[TSV_MAX_NODES];
  __shared__ float ua_s[TSV_MAX_NODES], qx_s[TSV_MAX_NODES], lx_s[TSV_MAX_NODES];
  __shared__ float red[128];
  __shared__ F2 scan_s[kMssWarps];
  __shared__ __align__(16) float pub[2][4];  // exchange slots, alternating
  __shared__ int bad;
  __shared__ int pick_s, last_s;
  const int b = blockIdx.x / ncl;
  const int rank = blockIdx.x - b * ncl;  // == %cluster_ctarank for 1-D clusters of ncl
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  if (tid == 0) {
    pick_s = INT32_MAX;
    last_s = -1;
  }
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  const int code = validate_verify_tree(parent + off, n, &bad);
  if (code) {
    if (rank == 0)
      fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                   status + b, code);
    return;  // uniform over the cluster: every CTA sees the same tree
  }
  const int32_t* par = parent + off;
  // Per child c: its token (rejected before any access when out of range),
  // accept uniform, q_c(x_c) and the parent row's logit at x_c.
  for (int c = 1 + tid; c < n; c += T) {
    const int x = tokens[off + c];
    tok_s[c] = x;
    if (x < 0 || (int64_t)x >= V) {
      atomicMax(&bad, TSV_ERR_INVALID_ARG);
    } else {
      ua_s[c] = __ldg(u_acc + off + c);
      qx_s[c] = __ldg(ssm_probs + (size_t)(off + c) * (size_t)V + x);
      lx_s[c] = __ldg(llm_logits + (size_t)(off + par[c]) * (size_t)V + x);
    }
  }
  __syncthreads();
  if (bad) {
    if (rank == 0)
      fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                   status + b, bad);
    return;
  }
  // Sibling lists in increasing index order.
  for (int c = tid; c < n; c += T) first_child[c] = INT32_MAX;
  __syncthreads();
  for (int c = 1 + tid; c < n; c += T) {
    const int p = par[c];
    atomicMin(&first_child[p], c);
    int nx = -1;
    for (int c2 = c + 1; c2 < n; ++c2) {
      if (par[c2] == p) {
        nx = c2;
        break;
      }
    }
    next_sib[c] = nx;
  }
  __syncthreads();

  // This CTA's slice (a multiple of 4 long, so 16-byte aligned rows stay aligned).
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t lo = min(V, (int64_t)rank * per), hi = min(V, lo + per);
  const int64_t n4 = (hi - lo) >> 2;  // full groups
  float* resid[2] = {resid_all + (size_t)b * 2 * (size_t)V, resid_all + ((size_t)b * 2 + 1) * (size_t)V};
  int xk = 0;  // exchanges so far (the same count in every CTA)
  // Publishes four floats, then waits for the whole cluster.
  auto exchange = [&](float v0, float v1, float v2, float v3) {
    if (tid == 0) {
      pub[xk & 1][0] = v0;
      pub[xk & 1][1] = v1;
      pub[xk & 1][2] = v2;
      pub[xk & 1][3] = v3;
    }
    cluster_sync_all();
  };
  auto peer = [&](int slot, int r) {
    return ld_dsmem_f32(mapa_shared(smem_u32(&pub[xk & 1][slot]), (uint32_t)r));
  };
  const int lane = tid & 31;

  // Row statistics of node u's logits: m = max(l / T), s = sum exp(l / T - m).
  float m_u = 0.f, inv_s = 0.f;
  auto row_stats = [&](int u) {
    const float* lrow = llm_logits + (size_t)(off + u) * (size_t)V;
    float m = -INFINITY;
    for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
      float4 v[kMssGroups];
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k) {
        const int64_t g = g0 + (int64_t)k * T;
        if (g < n4) v[k] = load4<0>(lrow, lo + 4 * g, vec);
      }
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k)
        if (g0 + (int64_t)k * T < n4)
#pragma unroll
          for (int e = 0; e < 4; ++e) m = fmaxf(m, at(v[k], e) * inv_t);
    }
    for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) m = fmaxf(m, lrow[y] * inv_t);
    m = block_max(m, red);
    CompSum acc;
    for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
      float4 v[kMssGroups];
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k) {
        const int64_t g = g0 + (int64_t)k * T;
        if (g < n4) v[k] = load4<0>(lrow, lo + 4 * g, vec);
      }
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k)
        if (g0 + (int64_t)k * T < n4)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc.add(exp_diff(at(v[k], e) * inv_t, m));
    }
    for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) acc.add(exp_diff(lrow[y] * inv_t, m));
    F2 s = comp_value(acc);
    float z1 = 0.f, z2 = 0.f;
    block_sum(s, z1, z2, red);
    exchange(m, s.hi, s.lo, 0.f);
    // Combine in rank order (identical in every CTA): M = max m_r, S = sum s_r e^(m_r - M).
    const float mr = lane < ncl ? peer(0, lane) : -INFINITY;
    const float sh = lane < ncl ? peer(1, lane) : 0.f;
    const float sl = lane < ncl ? peer(2, lane) : 0.f;
    float M = -INFINITY;
    for (int r = 0; r < ncl; ++r) M = fmaxf(M, __shfl_sync(0xffffffffu, mr, r));
    F2 S{0.f, 0.f};
    for (int r = 0; r < ncl; ++r) {
      const float m_r = __shfl_sync(0xffffffffu, mr, r);
      const F2 s_r{__shfl_sync(0xffffffffu, sh, r), __shfl_sync(0xffffffffu, sl, r)};
      if (m_r != -INFINITY) S = f2_add(S, f2_scale(s_r, exp_diff(m_r, M)));
    }
    ++xk;
    m_u = M;
    inv_s = f2_inv(S);
  };

  int u = 0, len = 1, cur = 0, tried = 0;
  bool from_resid = false;  // false: p = softmax(row u); true: p = resid[cur] / Z
  bool px_known = false;    // p at the current child's token came with the last exchange
  float px_next = 0.f;
  F2 Z{0.f, 0.f};
  if (rank == 0 && tid == 0) path[off] = 0;
  row_stats(0);
  while (true) {
    int accepted = -1;
    int c = first_child[u];
    if (c == INT32_MAX) c = -1;
    const float* lrow = llm_logits + (size_t)(off + u) * (size_t)V;
    while (c >= 0) {
      const float* q = ssm_probs + (size_t)(off + c) * (size_t)V;
      // p(x) of the current distribution (fp32, ~2 ulp); the test is exact.
      const float px = px_known ? px_next : exp_diff(lx_s[c] * inv_t, m_u) * inv_s;
      ++tried;
      if (accept_test(ua_s[c], qx_s[c], px)) {
        accepted = c;
        break;
      }
      // Rejected: residual pass over the slice, r = max(0, p - q).  The owner
      // of the next child's token records r and p there for the exchange.
      const int cn = next_sib[c];
      const int64_t xn = cn >= 0 ? (int64_t)tok_s[cn] : -1;
      const int nxt = cur ^ 1;
      const float inv_z = f2_inv(Z);
      const float* rin = resid[cur];
      float* rout = resid[nxt];
      CompSum acc;
      float r_x = 0.f, p_x = 0.f;
      for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
        float4 a[kMssGroups], qq[kMssGroups];
#pragma unroll
        for (int k = 0; k < kMssGroups; ++k) {
          const int64_t g = g0 + (int64_t)k * T;
          if (g < n4) {
            a[k] = from_resid ? load4<2>(rin, lo + 4 * g, vec) : load4<0>(lrow, lo + 4 * g, vec);
            qq[k] = load4<1>(q, lo + 4 * g, vec);
          }
        }
#pragma unroll
        for (int k = 0; k < kMssGroups; ++k) {
          const int64_t g = g0 + (int64_t)k * T;
          if (g < n4) {
            const int64_t y = lo + 4 * g;
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float py = from_resid ? at(a[k], e) * inv_z : exp_diff(at(a[k], e) * inv_t, m_u) * inv_s;
              r[e] = fmaxf(py - at(qq[k], e), 0.0f);
              acc.add(r[e]);
              if (y + e == xn) {
                r_x = r[e];
                p_x = py;
              }
            }
            if (vec) {
              *reinterpret_cast<float4*>(rout + y) = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) rout[y + e] = r[e];
            }
          }
        }
      }
      for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) {
        const float py = from_resid ? rin[y] * inv_z : exp_diff(__ldg(lrow + y) * inv_t, m_u) * inv_s;
        const float r = fmaxf(py - __ldcs(q + y), 0.0f);
        rout[y] = r;
        acc.add(r);
        if (y == xn) {
          r_x = r;
          p_x = py;
        }
      }
      F2 zs = comp_value(acc);
      block_sum(zs, r_x, p_x, red);
      exchange(zs.hi, zs.lo, r_x, p_x);
      const float zh = lane < ncl ? peer(0, lane) : 0.f;
      const float zl = lane < ncl ? peer(1, lane) : 0.f;
      const float rr = lane < ncl ? peer(2, lane) : 0.f;
      const float pr = lane < ncl ? peer(3, lane) : 0.f;
      F2 Znew{0.f, 0.f};
      float rxn = 0.f, pxn = 0.f;
      for (int r = 0; r < ncl; ++r) {
        Znew = f2_add(Znew, F2{__shfl_sync(0xffffffffu, zh, r), __shfl_sync(0xffffffffu, zl, r)});
        rxn += __shfl_sync(0xffffffffu, rr, r);  // one owner, the rest add zeros
        pxn += __shfl_sync(0xffffffffu, pr, r);
      }
      ++xk;
      if (Znew.hi > 0.f) {  // else p = q up to rounding: keep p
        cur = nxt;
        Z = Znew;
        from_resid = true;
        px_next = rxn * f2_inv(Znew);
      } else {
        px_next = pxn;
      }
      px_known = true;
      c = cn;
    }
    if (accepted < 0) break;
    u = accepted;
    if (rank == 0 && tid == 0) path[off + len] = u;
    ++len;
    from_resid = false;
    px_known = false;
    row_stats(u);
  }

  // Bonus token: smallest y with cumsum(w)[y] > u_smp[u] * sum(w), w = the
  // unnormalised current distribution.  Each thread owns a contiguous run of
  // its CTA's slice; runs and slices are in vocabulary order.
  {
    const float* lrow = llm_logits + (size_t)(off + u) * (size_t)V;
    const float* rin = resid[cur];
    const int64_t per_t = ((((hi - lo) + T - 1) / T) + 3) & ~int64_t(3);
    const int64_t tlo = min(hi, lo + (int64_t)tid * per_t), thi = min(hi, tlo + per_t);
    auto weight = [&](float a) { return from_resid ? a : exp_diff(a * inv_t, m_u); };
    CompSum acc;
    int64_t last_pos = -1;
    {
      int64_t y = tlo;
      for (; y + 4 <= thi; y += 4) {
        const float4 a = from_resid ? load4<2>(rin, y, vec) : load4<0>(lrow, y, vec);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w = weight(at(a, e));
          acc.add(w);
          if (w > 0.0f) last_pos = y + e;
        }
      }
      for (; y < thi; ++y) {
        const float w = weight(from_resid ? rin[y] : lrow[y]);
        acc.add(w);
        if (w > 0.0f) last_pos = y;
      }
    }
    const F2 mine = comp_value(acc);
    // Exclusive prefix over the CTA's threads: warp scan, then across warps.
    const int warp = tid >> 5;
    F2 incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const F2 t{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
      if (lane >= o) incl = f2_add(t, incl);
    }
    F2 wexcl{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    if (lane == 0) wexcl = F2{0.f, 0.f};
    if (lane == 31) scan_s[warp] = incl;
    if (last_pos >= 0) atomicMax(&last_s, (int)last_pos);
    __syncthreads();
    F2 wbase{0.f, 0.f}, cta_total{0.f, 0.f};
    for (int w = 0; w < kMssWarps; ++w) {
      if (w < warp) wbase = f2_add(wbase, scan_s[w]);
      cta_total = f2_add(cta_total, scan_s[w]);
    }
    exchange(cta_total.hi, cta_total.lo, __int_as_float(last_s), 0.f);
    const float th = lane < ncl ? peer(0, lane) : 0.f;
    const float tl = lane < ncl ? peer(1, lane) : 0.f;
    const int lr = lane < ncl ? __float_as_int(peer(2, lane)) : -1;
    F2 base{0.f, 0.f}, total{0.f, 0.f};
    int last_all = -1;
    for (int r = 0; r < ncl; ++r) {
      const F2 t{__shfl_sync(0xffffffffu, th, r), __shfl_sync(0xffffffffu, tl, r)};
      if (r < rank) base = f2_add(base, t);
      total = f2_add(total, t);
      last_all = max(last_all, __shfl_sync(0xffffffffu, lr, r));
    }
    ++xk;
    const F2 excl = f2_add(f2_add(base, wbase), wexcl);
    const F2 target = f2_scale(total, __ldg(u_smp + off + u));
    if (mine.hi > 0.f && !f2_lt(target, excl) && f2_lt(target, f2_add(excl, mine))) {
      // This run holds the crossing; walk it in order.
      int64_t pick = -1;
      CompSum run;
      for (int64_t y = tlo; y < thi; ++y) {
        const float w = weight(from_resid ? rin[y] : lrow[y]);
        run.add(w);
        if (f2_lt(target, f2_add(excl, comp_value(run)))) {
          pick = y;
          break;
        }
      }
      if (pick < 0) pick = last_pos;  // rounding inside the run
      atomicMin(&pick_s, (int)pick);
    }
    __syncthreads();
    exchange(__int_as_float(pick_s), 0.f, 0.f, 0.f);
    if (rank == 0 && tid == 0) {
      int pick = INT32_MAX;
      for (int r = 0; r < ncl; ++r) pick = min(pick, __float_as_int(peer(0, r)));
      // No crossing (rounding left the target at the total): last positive entry.
      bonus[b] = pick != INT32_MAX ? pick : last_all;
      accept_len[b] = len - 1;
      if (n_tried) n_tried[b] = tried;
      status[b] = TSV_OK;
    }
    cluster_sync_all();  // peers keep their exchange slots until rank 0 has read them
  }
  if (rank == 0)
    for (int i = len + tid; i < n; i += T) path[off + i] = -1;
}

int mss_cluster_size(int64_t V) {
  const int64_t c = (V + kMssMinSlice - 1) / kMssMinSlice;
  return (int)(c < 1 ? 1 : (c > kMssMaxCluster ? kMssMaxCluster : c));
}

cudaError_t launch_mss_verify(const float* llm_logits, const float* ssm_probs, int64_t V,
                              const int32_t* tokens, const int32_t* parent,
                              const int32_t* node_offsets, const float* u_acc, const float* u_smp,
                              float inv_t, int32_t B, float* resid, int32_t* path,
                              int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                              int32_t* status, cudaStream_t st) {
  const int ncl = mss_cluster_size(V);
  const int vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(llm_logits) |
                                    reinterpret_cast<uintptr_t>(ssm_probs) |
                                    reinterpret_cast<uintptr_t>(resid)) & 15) == 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ncl));
  cfg.blockDim = dim3(kMssThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mss_verify_kernel, llm_logits, ssm_probs, V, tokens, parent,
                            node_offsets, u_acc, u_smp, inv_t, ncl, vec, resid, path, accept_len,
                            bonus, n_tried, status);
}

}  // namespace tsv
