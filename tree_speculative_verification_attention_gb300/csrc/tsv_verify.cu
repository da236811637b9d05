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
//   row_stats_kernel       grid (splits, N): per row max and compensated
//                          sum of exp(l/T - max) over a vocab slice.
//   mss_walk_kernel        grid B, 1024 threads: the sequential walk.  An
//                          accept test needs only p(x) and q(x); a rejection
//                          makes one vocab-wide pass that writes the residual
//                          max(0, p - q) into the workspace and sums it; the
//                          bonus token is drawn by a block-wide inverse-CDF
//                          scan.
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

// The greedy walk of request b from its per-slice argmax partials: every
// child c whose token equals argmax(parent(c)) proposes itself to its parent
// with atomicMin (lowest index wins), then the chain is followed from the root.
// Run by one whole CTA of up to 256 threads.
__device__ void greedy_walk_request(int b, int off, int n, const float* part_val,
                                    const int32_t* part_idx, int splits, const int32_t* tokens,
                                    const int32_t* parent, int32_t* path, int32_t* accept_len,
                                    int32_t* bonus, int32_t* status, int* sh_bad, int32_t* am,
                                    int32_t* nxt, int* len_s) {
  const int code = validate_verify_tree(parent + off, n, sh_bad);
  if (code) {
    fail_request(path + off, n, accept_len + b, bonus + b, nullptr, status + b, code);
    return;
  }
  for (int u = threadIdx.x; u < n; u += blockDim.x) {
    ArgMax best{-INFINITY, INT32_MAX};
    for (int s = 0; s < splits; ++s) {
      const size_t k = (size_t)(off + u) * splits + s;
      best = better(best, ArgMax{__ldcg(part_val + k), __ldcg(part_idx + k)});
    }
    am[u] = best.i;
    nxt[u] = INT32_MAX;
  }
  __syncthreads();
  for (int c = 1 + threadIdx.x; c < n; c += blockDim.x) {
    const int p = parent[off + c];
    if (tokens[off + c] == am[p]) atomicMin(&nxt[p], c);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int u = 0, len = 0;
    path[off + len++] = 0;
    while (nxt[u] != INT32_MAX) {
      u = nxt[u];
      path[off + len++] = u;
    }
    accept_len[b] = len - 1;
    bonus[b] = am[u];
    status[b] = TSV_OK;
    *len_s = len;
  }
  __syncthreads();
  for (int i = *len_s + threadIdx.x; i < n; i += blockDim.x) path[off + i] = -1;
}

// Walk-only kernel: one CTA per request (used when N == 0, where no argmax CTA exists).
__global__ void __launch_bounds__(TSV_MAX_NODES)
    greedy_walk_kernel(const float* __restrict__ part_val, const int32_t* __restrict__ part_idx,
                       int splits, const int32_t* __restrict__ tokens,
                       const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                       int32_t* __restrict__ path, int32_t* __restrict__ accept_len,
                       int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  __shared__ int32_t am[TSV_MAX_NODES];
  __shared__ int32_t nxt[TSV_MAX_NODES];
  __shared__ int bad, len_s;
  const int b = blockIdx.x;
  const int off = node_offsets[b];
  greedy_walk_request(b, off, node_offsets[b + 1] - off, part_val, part_idx, splits, tokens, parent,
                      path, accept_len, bonus, status, &bad, am, nxt, &len_s);
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
  __shared__ int32_t am[TSV_MAX_NODES];
  __shared__ int32_t nxt[TSV_MAX_NODES];
  __shared__ ArgMax red[kArgmaxThreads / 32];
  __shared__ int bad, len_s, last;
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
                      status, &bad, am, nxt, &len_s);
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

constexpr int kStatsThreads = 256;
constexpr int kWalkThreads = 1024;

// exp(a - m) with the subtraction's rounding error folded back in (TwoSum:
// a - m = d + err exactly), so the result is as accurate as expf itself even
// when a - m is large in magnitude.  Requires finite a and m.
__device__ __forceinline__ float exp_diff(float a, float m) {
  const float d = a - m;
  const float bb = d - a;
  const float err = (a - (d - bb)) + (-m - bb);
  return expf(d) * (1.0f + err);
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide sum in fp64 (every thread gets the result).  `scratch` holds 32 doubles.
__device__ double block_sum_d(double v, double* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  v = warp_sum_d(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  double t = lane < nw ? scratch[lane] : 0.0;
  t = warp_sum_d(t);
  return t;
}

}  // namespace

__global__ void __launch_bounds__(kStatsThreads)
    row_stats_kernel(const float* __restrict__ logits, int64_t V, int splits, float inv_t,
                     float* __restrict__ part_m, double* __restrict__ part_s) {
  const int row = blockIdx.y, s = blockIdx.x;
  const int64_t per = slice_len(V, splits);
  const int64_t lo = (int64_t)s * per, hi = min(V, lo + per);
  const float* x = logits + (size_t)row * (size_t)V;
  // Pass 1: max of the slice.
  float m = -INFINITY;
  for (int64_t k = lo + threadIdx.x; k < hi; k += kStatsThreads) m = fmaxf(m, __ldg(x + k) * inv_t);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float redm[kStatsThreads / 32];
  __shared__ double reds[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) redm[warp] = m;
  __syncthreads();
  m = -INFINITY;
#pragma unroll
  for (int w = 0; w < kStatsThreads / 32; ++w) m = fmaxf(m, redm[w]);
  // Pass 2 (the slice is now in L1/L2): compensated sum of exp(z - m).
  CompSum acc;
  for (int64_t k = lo + threadIdx.x; k < hi; k += kStatsThreads)
    acc.add(exp_diff(__ldg(x + k) * inv_t, m));
  const double tot = block_sum_d(acc.value(), reds);
  if (threadIdx.x == 0) {
    part_m[(size_t)row * splits + s] = m;
    part_s[(size_t)row * splits + s] = tot;
  }
}

int stats_splits(int64_t V, int32_t N, int num_sms) { return greedy_splits(V, N, num_sms); }

cudaError_t launch_row_stats(const float* logits, int64_t V, int32_t N, int splits, float inv_t,
                             float* part_m, double* part_s, cudaStream_t st) {
  dim3 grid(splits, N);
  row_stats_kernel<<<grid, kStatsThreads, 0, st>>>(logits, V, splits, inv_t, part_m, part_s);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(kWalkThreads)
    mss_walk_kernel(const float* __restrict__ llm_logits, const float* __restrict__ ssm_probs,
                    int64_t V, const int32_t* __restrict__ tokens,
                    const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                    const float* __restrict__ u_acc, const float* __restrict__ u_smp, float inv_t,
                    int splits, const float* __restrict__ part_m, const double* __restrict__ part_s,
                    float* __restrict__ resid_all, int32_t* __restrict__ path,
                    int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                    int32_t* __restrict__ n_tried, int32_t* __restrict__ status) {
  __shared__ int32_t first_child[TSV_MAX_NODES];
  __shared__ int32_t next_sib[TSV_MAX_NODES];
  __shared__ float row_m[TSV_MAX_NODES];
  __shared__ double row_s[TSV_MAX_NODES];
  __shared__ double scratch[32];
  __shared__ double scan_s[kWalkThreads / 32];
  __shared__ int bad;
  __shared__ int pick_s, last_s;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0) {
    pick_s = INT32_MAX;
    last_s = -1;
  }
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  const int code = validate_verify_tree(parent + off, n, &bad);
  if (code) {
    fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                 status + b, code);
    return;
  }
  const int32_t* par = parent + off;
  // Tokens index the vocabulary rows: reject out-of-range ones before any access.
  for (int c = 1 + tid; c < n; c += blockDim.x) {
    const int x = tokens[off + c];
    if (x < 0 || (int64_t)x >= V) atomicMax(&bad, TSV_ERR_INVALID_ARG);
  }
  __syncthreads();
  if (bad) {
    fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                 status + b, bad);
    return;
  }
  // Sibling lists in increasing index order.
  for (int c = tid; c < n; c += blockDim.x) first_child[c] = INT32_MAX;
  __syncthreads();
  for (int c = 1 + tid; c < n; c += blockDim.x) {
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
  // Row statistics of every node: merge the vocab slices.
  for (int u = tid; u < n; u += blockDim.x) {
    float m = -INFINITY;
    for (int s = 0; s < splits; ++s) m = fmaxf(m, part_m[(size_t)(off + u) * splits + s]);
    double sum = 0.0;
    for (int s = 0; s < splits; ++s) {
      const size_t k = (size_t)(off + u) * splits + s;
      if (part_m[k] != -INFINITY) sum += part_s[k] * (double)exp_diff(part_m[k], m);
    }
    row_m[u] = m;
    row_s[u] = sum;
  }
  __syncthreads();

  float* resid[2] = {resid_all + (size_t)b * 2 * (size_t)V, resid_all + ((size_t)b * 2 + 1) * (size_t)V};
  int u = 0, len = 1, cur = 0, tried = 0;
  bool from_resid = false;  // false: p = softmax(row u); true: p = resid[cur] / Z
  double Z = 0.0;
  if (tid == 0) path[off] = 0;
  while (true) {
    int accepted = -1;
    int c = first_child[u];
    if (c == INT32_MAX) c = -1;
    const float* lrow = llm_logits + (size_t)(off + u) * (size_t)V;
    const float m_u = row_m[u];
    const float inv_s = (float)(1.0 / row_s[u]);
    while (c >= 0 && accepted < 0) {
      const int x = tokens[off + c];
      const float* q = ssm_probs + (size_t)(off + c) * (size_t)V;
      const float inv_z = (float)(1.0 / Z);
      // p(x) of the current distribution (fp32, ~2 ulp), compared in fp64.
      const float px = from_resid ? resid[cur][x] * inv_z
                                  : exp_diff(__ldg(lrow + x) * inv_t, m_u) * inv_s;
      ++tried;
      if ((double)__ldg(u_acc + off + c) * (double)__ldg(q + x) < (double)px) {
        accepted = c;
        break;
      }
      // Rejected: residual pass over the vocabulary, r = max(0, p - q).
      const int nxt = cur ^ 1;
      CompSum acc;
      for (int64_t y = tid; y < V; y += blockDim.x) {
        const float py = from_resid ? resid[cur][y] * inv_z
                                    : exp_diff(__ldg(lrow + y) * inv_t, m_u) * inv_s;
        const float r = fmaxf(py - __ldcs(q + y), 0.0f);
        resid[nxt][y] = r;
        acc.add(r);
      }
      const double Znew = block_sum_d(acc.value(), scratch);
      if (Znew > 0.0) {  // else p = q up to rounding: keep p
        cur = nxt;
        Z = Znew;
        from_resid = true;
      }
      __syncthreads();  // residual row complete before anyone reads it
      c = next_sib[c];
    }
    if (accepted < 0) break;
    u = accepted;
    if (tid == 0) path[off + len] = u;
    ++len;
    from_resid = false;
  }
  // Bonus token: smallest y with cumsum(w)[y] > u_smp[u] * sum(w), w = the
  // unnormalised current distribution.  Each thread owns a contiguous slice.
  {
    const float* lrow = llm_logits + (size_t)(off + u) * (size_t)V;
    const float m_u = row_m[u];
    const int64_t per = (V + blockDim.x - 1) / blockDim.x;
    const int64_t lo = (int64_t)tid * per, hi = min(V, lo + per);
    CompSum acc;
    int64_t last_pos = -1;
    for (int64_t y = lo; y < hi; ++y) {
      const float w = from_resid ? resid[cur][y] : exp_diff(__ldg(lrow + y) * inv_t, m_u);
      acc.add(w);
      if (w > 0.0f) last_pos = y;
    }
    const double mine = acc.value();
    // Exclusive prefix over threads (fp64): warp scan, then across warps.
    const int warp = tid >> 5, lane = tid & 31;
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) scan_s[warp] = incl;
    if (last_pos >= 0) atomicMax(&last_s, (int)last_pos);
    __syncthreads();
    double wbase = 0.0, total = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      if (w < warp) wbase += scan_s[w];
      total += scan_s[w];
    }
    const double excl = wbase + incl - mine;
    const double target = (double)__ldg(u_smp + off + u) * total;
    if (mine > 0.0 && excl <= target && target < excl + mine) {
      // This slice holds the crossing; walk it in order.
      int64_t pick = -1;
      CompSum run;
      for (int64_t y = lo; y < hi; ++y) {
        const float w = from_resid ? resid[cur][y] : exp_diff(__ldg(lrow + y) * inv_t, m_u);
        run.add(w);
        if (excl + run.value() > target) {
          pick = y;
          break;
        }
      }
      if (pick < 0) pick = last_pos;  // rounding inside the slice
      atomicMin(&pick_s, (int)pick);
    }
    __syncthreads();
    if (tid == 0) {
      // No crossing (rounding left the target at the total): last positive entry.
      bonus[b] = pick_s != INT32_MAX ? pick_s : last_s;
      accept_len[b] = len - 1;
      if (n_tried) n_tried[b] = tried;
      status[b] = TSV_OK;
    }
  }
  for (int i = len + tid; i < n; i += blockDim.x) path[off + i] = -1;
}

cudaError_t launch_mss_walk(const float* llm_logits, const float* ssm_probs, int64_t V,
                            const int32_t* tokens, const int32_t* parent,
                            const int32_t* node_offsets, const float* u_acc, const float* u_smp,
                            float inv_t, int32_t B, int splits, const float* part_m,
                            const double* part_s, float* resid, int32_t* path,
                            int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                            int32_t* status, cudaStream_t st) {
  mss_walk_kernel<<<B, kWalkThreads, 0, st>>>(llm_logits, ssm_probs, V, tokens, parent,
                                              node_offsets, u_acc, u_smp, inv_t, splits, part_m,
                                              part_s, resid, path, accept_len, bonus, n_tried,
                                              status);
  return cudaGetLastError();
}

}  // namespace tsv
