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
constexpr int kArgmaxInFlight = 8;
constexpr uint32_t kArgmaxPrefetchMax = 32768;  // largest slice pulled into L2 ahead of the wait
constexpr int kMinSlice = 2048;  // vocab entries per CTA at least

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
    // Eight independent 16-byte loads in flight per thread (32 KB per CTA).
    for (; k + (kArgmaxInFlight - 1) * kArgmaxThreads < hi4; k += kArgmaxInFlight * kArgmaxThreads) {
      float4 a[kArgmaxInFlight];
#pragma unroll
      for (int u = 0; u < kArgmaxInFlight; ++u) a[u] = __ldcs(x4 + k + u * kArgmaxThreads);
#pragma unroll
      for (int u = 0; u < kArgmaxInFlight; ++u) {
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
};

// The greedy walk of request b from its per-slice argmax partials: every
// child c whose token equals argmax(parent(c)) proposes itself to its parent
// with atomicMin (lowest index wins), then the chain is followed from the
// root.  Run by one whole CTA of kArgmaxThreads threads: one load step
// (parents, tokens, partials), then three barriers — partials staged; every
// node's argmax known and the tree checked; proposals made — and warp 0
// follows the chain and writes the path.
__device__ void greedy_walk_request(int b, int off, int n, const float* part_val,
                                    const int32_t* part_idx, int splits, const int32_t* tokens,
                                    const int32_t* parent, int32_t* path, int32_t* accept_len,
                                    int32_t* bonus, int32_t* status, WalkSmem& w) {
  const int T = blockDim.x;
  const int i = threadIdx.x;
  static_assert(kWalkPartials <= 4 * kArgmaxThreads && TSV_MAX_NODES <= kArgmaxThreads, "one pass");
  const int size_code = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
  if (size_code) {  // uniform: n is the same for every thread
    fail_request(path + off, n, accept_len + b, bonus + b, nullptr, status + b, size_code);
    return;
  }
  const int items = n * splits;  // rows of a request are consecutive, so its partials are too
  const bool staged = items <= kWalkPartials;
  // Every load is issued before the first shared-memory store, so they all
  // travel together.
  int pv = 0, tv = 0;
  if (i < n) {
    pv = parent[off + i];
    tv = tokens[off + i];
  }
  float pval[4];
  int32_t pidx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = i + k * T;
    if (staged && e < items) {
      pval[k] = __ldcg(part_val + (size_t)off * splits + e);
      pidx[k] = __ldcg(part_idx + (size_t)off * splits + e);
    }
  }
  if (i < n) {
    w.par[i] = pv;
    w.tok[i] = tv;
    w.nxt[i] = INT32_MAX;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int e = i + k * T;
    if (staged && e < items) w.part[e] = ArgMax{pval[k], pidx[k]};
  }
  __syncthreads();
  // Node i: its parent is checked (a single root at 0, every other parent
  // earlier) and its row's slices merged into its argmax.
  bool bad = false;
  if (i < n) {
    bad = !((i == 0) ? (pv == -1) : (pv >= 0 && pv < i));
    ArgMax best{-INFINITY, INT32_MAX};
    for (int sl = 0; sl < splits; ++sl) {
      const size_t k = (size_t)(off + i) * splits + sl;
      best = better(best, staged ? w.part[i * splits + sl] : ArgMax{__ldcg(part_val + k), __ldcg(part_idx + k)});
    }
    w.am[i] = best.i;
  }
  if (__syncthreads_or(bad)) {
    fail_request(path + off, n, accept_len + b, bonus + b, nullptr, status + b, TSV_ERR_BAD_TREE);
    return;
  }
  if (i >= 1 && i < n && tv == w.am[pv]) atomicMin(&w.nxt[pv], i);
  __syncthreads();
  if (i < 32) {  // warp 0: lane 0 follows the chain, the warp writes the rest
    int len = 0;
    if (i == 0) {
      int u = 0;
      path[off + len++] = 0;
      while (w.nxt[u] != INT32_MAX) {
        u = w.nxt[u];
        path[off + len++] = u;
      }
      accept_len[b] = len - 1;
      bonus[b] = w.am[u];
      status[b] = TSV_OK;
    }
    len = __shfl_sync(0xffffffffu, len, 0);
    for (int k = len + i; k < n; k += 32) path[off + k] = -1;
  }
}

// Walk-only kernel: one CTA per request (used when N == 0, where no argmax CTA exists).
__global__ void __launch_bounds__(TSV_MAX_NODES)
    greedy_walk_kernel(const float* __restrict__ part_val, const int32_t* __restrict__ part_idx,
                       int splits, const int32_t* __restrict__ tokens,
                       const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                       int32_t* __restrict__ path, int32_t* __restrict__ accept_len,
                       int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
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
// Thread 0 writes the CTA's partial and counts it with one acquire-release
// atomic, so the last CTA sees every partial without a separate fence.
__global__ void __launch_bounds__(kArgmaxThreads, 4)  // <= 64 registers: the loads stay in flight
    greedy_verify_kernel(const float* __restrict__ logits, int64_t V, int splits,
                         const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                         const int32_t* __restrict__ node_offsets, int B,
                         float* __restrict__ part_val, int32_t* __restrict__ part_idx,
                         int32_t* __restrict__ counters, int32_t* __restrict__ path,
                         int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                         int32_t* __restrict__ status) {
  // A small slice (short rows spread over many CTAs) is pulled into L2 while
  // the previous kernel finishes: a prefetch reads no value, so it may run
  // ahead of that kernel's writes.
  if (threadIdx.x == 0 && (V & 3) == 0) {
    const int64_t per = slice_len(V, splits);
    const int64_t lo = min(V, (int64_t)blockIdx.x * per), hi = min(V, lo + per);
    const float* src = logits + (size_t)blockIdx.y * (size_t)V + lo;
    const uint32_t bytes = (uint32_t)((hi - lo) * 4);
    if (bytes > 0 && bytes <= kArgmaxPrefetchMax && (reinterpret_cast<uintptr_t>(src) & 15) == 0)
      bulk_prefetch_l2(src, bytes);
  }
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ int32_t offs[TSV_MAX_BATCH + 1];
  __shared__ WalkSmem w;
  __shared__ ArgMax red[kArgmaxThreads / 32];
  __shared__ int last;
  const int row = blockIdx.y, s = blockIdx.x;
  // The offsets travel with the first logits loads: stored after the slice.
  static_assert(TSV_MAX_BATCH < kArgmaxThreads, "one offset per thread");
  const int my_off = threadIdx.x <= B ? node_offsets[threadIdx.x] : 0;
  const ArgMax best = slice_argmax(logits, V, splits, row, s, red);
  pdl_trigger();  // this CTA's share of the logits is read: let the next kernel be scheduled
  if (threadIdx.x <= B) offs[threadIdx.x] = my_off;
  __syncthreads();
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
  if (threadIdx.x == 0) {
    part_val[(size_t)row * splits + s] = best.v;
    part_idx[(size_t)row * splits + s] = best.i;
    last = atom_add_acq_rel_gpu(counters + b, 1) == n * splits - 1;
  }
  __syncthreads();
  if (!last) return;
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
  return launch_pdl(greedy_verify_kernel, grid, dim3(kArgmaxThreads), 0, st, 0u, logits, V, splits, tokens, parent,
                    node_offsets, B, part_val, part_idx, counters, path, accept_len, bonus, status);
}

cudaError_t launch_greedy_walk(const float* part_val, const int32_t* part_idx, int splits,
                               const int32_t* tokens, const int32_t* parent,
                               const int32_t* node_offsets, int32_t B, int32_t* path,
                               int32_t* accept_len, int32_t* bonus, int32_t* status,
                               cudaStream_t st) {
  return launch_pdl(greedy_walk_kernel, dim3(B), dim3(TSV_MAX_NODES), 0, st, 0u, part_val, part_idx, splits, tokens,
                    parent, node_offsets, path, accept_len, bonus, status);
}

// ------------------------------------------------------------------ stochastic

namespace {

constexpr int kMssThreads = 256;
constexpr int kMssWarps = kMssThreads / 32;
constexpr int kMssMaxCluster = 8;
constexpr int64_t kMssMinSlice = 4096;  // vocab entries per CTA at least
constexpr int kMssGroups = 4;           // 4-float groups in flight per thread
constexpr uint32_t kBulkChunk = 32768;  // bytes per bulk copy instruction
constexpr int kMaxTopK = kMssMaxTopK;   // largest top-k the warped support handles

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

// Sum over the warp's lanes, the same in every lane (butterfly; f2_add is
// commutative, so partners compute identical sums).
__device__ __forceinline__ F2 warp_sum_f2(F2 a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = f2_add(a, shfl_xor_f2(a, o));
  return a;
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

// A CTA's view of one vocabulary row restricted to its slice: element y of
// the row is p[y - off].  p points either into global memory (off = 0, the
// whole row) or at the slice staged in shared memory (off = the slice's first
// index); loads are generic, so both work.
struct Slice {
  const float* p;
  int64_t off;
  __device__ __forceinline__ float operator[](int64_t y) const { return p[y - off]; }
  __device__ __forceinline__ float4 ld4(int64_t y, bool vec) const {
    const float* q = p + (y - off);
    if (vec) return *reinterpret_cast<const float4*>(q);
    return make_float4(q[0], q[1], q[2], q[3]);
  }
};

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

// Order-preserving 32-bit key of a float (-0 counts as +0): larger logit,
// larger key.
__device__ __forceinline__ uint32_t order_key(float l) {
  const uint32_t u = __float_as_uint(l + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ int ld_dsmem_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Token y of the row is kept by the warp iff its logit l ranks before the
// boundary: l > tau, or l == tau and y <= ycut (ranking: larger logit first,
// equal logits by lower index).
__device__ __forceinline__ bool kept(float l, int64_t y, float tau, int ycut) {
  return l > tau || (l == tau && y <= ycut);
}

// Shared scratch of the warped support.
static_assert(kMssThreads == 256, "one histogram bin per thread");
struct SelSmem {
  int hist[2][256];  // per-CTA digit histograms, alternating with the exchanges
  int wsum[kMssThreads / 32];
  int ints[8];
  float cand_v[kMaxTopK];
  int cand_i[kMaxTopK];
  float srt_v[kMaxTopK];
  int srt_i[kMaxTopK];
  F2 tsum[kMssWarps];
  F2 s_cut;
};

struct Support {
  float tau;
  int ycut;
  F2 S;
};

// The warped support of one LLM row (top-k, then top-p, as the oracle defines
// them), found by the whole cluster: its boundary (tau, ycut) in the ranking
// and the kept mass S = sum exp(l / T - M) over kept tokens.  Radix selection
// of the k-th key (four 8-bit digits, histograms summed over the cluster),
// then, for equal logits at the boundary, the cut by token index; the kept
// tokens (at most kMaxTopK) are gathered into every CTA and sorted there, the
// same way in every CTA, for the top-p cut and the mass.  Every CTA of the
// cluster runs it in lockstep; `xk` counts the exchanges.
__device__ __noinline__ Support warped_support(const Slice lrow, int64_t V, int64_t lo,
                                               int64_t hi, float inv_t, float M, int top_k, float top_p,
                                               int ncl, int rank, int& xk, float (*pub)[4], SelSmem& w) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Kt = (int64_t)top_k < V ? top_k : (int)V;
  uint32_t prefix = 0;
  float tau = -INFINITY;
  int ycut = INT32_MAX;
  if (Kt < V) {
    int r = Kt, ties_total = 0;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* h = w.hist[xk & 1];
      h[tid] = 0;  // kMssThreads == 256 bins
      __syncthreads();
      for (int64_t y = lo + tid; y < hi; y += kMssThreads) {
        const uint32_t k = order_key(lrow[y]);
        if (pass == 0 || (k >> (shift + 8)) == prefix) atomicAdd(&h[(k >> shift) & 255], 1);
      }
      __syncthreads();
      cluster_sync_all();
      int cnt = 0;
      for (int rr = 0; rr < ncl; ++rr) cnt += ld_dsmem_s32(mapa_shared(smem_u32(&h[tid]), (uint32_t)rr));
      ++xk;
      // Suffix sums over the digits (larger digit = larger logit).
      int sfx = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, sfx, o);
        if (lane + o < 32) sfx += t;
      }
      if (lane == 0) w.wsum[warp] = sfx;
      __syncthreads();
      for (int ww = warp + 1; ww < kMssWarps; ++ww) sfx += w.wsum[ww];
      if (sfx >= r && sfx - cnt < r) {
        w.ints[0] = tid;
        w.ints[1] = sfx - cnt;
        w.ints[2] = cnt;
      }
      __syncthreads();
      r -= w.ints[1];
      ties_total = w.ints[2];
      prefix = (prefix << 8) | (uint32_t)w.ints[0];
      __syncthreads();
    }
    tau = key_value(prefix);
    if (r < ties_total) {
      // Keep the r lowest-index tokens among those equal to tau.
      if (tid == 0) w.ints[3] = 0;
      __syncthreads();
      int c = 0;
      for (int64_t y = lo + tid; y < hi; y += kMssThreads) c += order_key(lrow[y]) == prefix;
      atomicAdd(&w.ints[3], c);
      __syncthreads();
      if (tid == 0) pub[xk & 1][0] = __int_as_float(w.ints[3]);
      cluster_sync_all();
      int before = 0, mine = 0;
      for (int rr = 0; rr < ncl; ++rr) {
        const int t = __float_as_int(ld_dsmem_f32(mapa_shared(smem_u32(&pub[xk & 1][0]), (uint32_t)rr)));
        if (rr < rank) before += t;
        if (rr == rank) mine = t;
      }
      ++xk;
      int found = -1;
      if (warp == 0 && before < r && r <= before + mine) {
        int need = r - before;
        for (int64_t base = lo; base < hi; base += 32) {
          const int64_t y = base + lane;
          const bool tie = y < hi && order_key(lrow[y]) == prefix;
          const uint32_t bal = __ballot_sync(0xffffffffu, tie);
          const int n = __popc(bal);
          if (need <= n) {
            uint32_t b2 = bal;
            for (int q = 1; q < need; ++q) b2 &= b2 - 1;
            found = (int)(base + __ffs(b2) - 1);
            break;
          }
          need -= n;
        }
      }
      if (tid == 0) pub[xk & 1][0] = __int_as_float(found);
      cluster_sync_all();
      ycut = -1;
      for (int rr = 0; rr < ncl; ++rr)
        ycut = max(ycut, __float_as_int(ld_dsmem_f32(mapa_shared(smem_u32(&pub[xk & 1][0]), (uint32_t)rr))));
      ++xk;
    }
  }
  // Gather the kept tokens of every CTA, then sort them (larger logit first,
  // equal logits by lower index) identically in every CTA.
  if (tid == 0) w.ints[4] = 0;
  __syncthreads();
  for (int64_t y = lo + tid; y < hi; y += kMssThreads) {
    const float l = lrow[y];
    if (kept(l, y, tau, ycut)) {
      const int j = atomicAdd(&w.ints[4], 1);
      if (j < kMaxTopK) {  // at most min(top_k, V) <= kMaxTopK tokens are kept
        w.cand_v[j] = l;
        w.cand_i[j] = (int)y;
      }
    }
  }
  __syncthreads();
  if (tid == 0) pub[xk & 1][0] = __int_as_float(w.ints[4]);
  cluster_sync_all();
  int cnt_r[kMssMaxCluster], K = 0;
  for (int rr = 0; rr < ncl; ++rr) {
    cnt_r[rr] = __float_as_int(ld_dsmem_f32(mapa_shared(smem_u32(&pub[xk & 1][0]), (uint32_t)rr)));
    K += cnt_r[rr];
  }
  ++xk;
  int P2 = 1;
  while (P2 < K) P2 <<= 1;
  for (int j = tid; j < P2; j += kMssThreads) {
    float v = -INFINITY;
    int id = INT32_MAX;
    if (j < K) {
      int rr = 0, jl = j;
      while (jl >= cnt_r[rr]) jl -= cnt_r[rr++];
      v = ld_dsmem_f32(mapa_shared(smem_u32(&w.cand_v[jl]), (uint32_t)rr));
      id = ld_dsmem_s32(mapa_shared(smem_u32(&w.cand_i[jl]), (uint32_t)rr));
    }
    w.srt_v[j] = v;
    w.srt_i[j] = id;
  }
  __syncthreads();
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P2; i += kMssThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const float a = w.srt_v[i], bv = w.srt_v[ixj];
          const int ai = w.srt_i[i], bi = w.srt_i[ixj];
          const bool a_first = a > bv || (a == bv && ai < bi);
          if (((i & k) == 0) != a_first) {
            w.srt_v[i] = bv;
            w.srt_v[ixj] = a;
            w.srt_i[i] = bi;
            w.srt_i[ixj] = ai;
          }
        }
      }
      __syncthreads();
    }
  }
  // Cumulative mass in ranking order: thread t owns a run of consecutive entries.
  const int per = (K + kMssThreads - 1) / kMssThreads;
  const int j0 = min(K, tid * per), j1 = min(K, j0 + per);
  F2 run{0.f, 0.f};
  for (int j = j0; j < j1; ++j) run = f2_add(run, F2{exp_diff(w.srt_v[j] * inv_t, M), 0.f});
  F2 incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const F2 t{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
    if (lane >= o) incl = f2_add(t, incl);
  }
  if (lane == 31) w.tsum[warp] = incl;
  if (tid == 0) w.ints[5] = INT32_MAX;
  __syncthreads();
  F2 base{0.f, 0.f}, total{0.f, 0.f};
  for (int ww = 0; ww < kMssWarps; ++ww) {
    if (ww < warp) base = f2_add(base, w.tsum[ww]);
    total = f2_add(total, w.tsum[ww]);
  }
  // Exclusive prefix of this thread's run (all threads shuffle, then branch).
  const F2 up{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  const F2 excl = lane == 0 ? base : f2_add(base, up);
  int J = K;
  F2 S = total;
  if (top_p < 1.0f) {
    // Shortest prefix whose share of the kept mass reaches top_p.
    const F2 target = f2_scale(total, top_p);
    F2 cum = excl;
    for (int j = j0; j < j1; ++j) {
      cum = f2_add(cum, F2{exp_diff(w.srt_v[j] * inv_t, M), 0.f});
      if (!f2_lt(cum, target)) {
        atomicMin(&w.ints[5], j);
        break;
      }
    }
    __syncthreads();
    J = min(K, w.ints[5] + 1);
    // The mass up to the cut, from the thread that owns entry J-1.
    if (J - 1 >= j0 && J - 1 < j1) {
      F2 c2 = excl;
      for (int j = j0; j < J; ++j) c2 = f2_add(c2, F2{exp_diff(w.srt_v[j] * inv_t, M), 0.f});
      w.s_cut = c2;
    }
    __syncthreads();
    S = w.s_cut;
  }
  Support out;
  out.tau = w.srt_v[J - 1];
  out.ycut = w.srt_i[J - 1];
  out.S = S;
  __syncthreads();  // the scratch may be rewritten by the next call
  return out;
}

}  // namespace

// Multi-step speculative sampling: one cluster of `ncl` CTAs per request, CTA
// rank r owning vocab slice r.  All walk decisions are taken identically by
// every CTA from values every CTA holds: the children, their tokens, accept
// uniforms, proposal probabilities q_c(x_c) and parent logits l(x_c) (read
// once, in parallel, at the start), the row statistics and residual sums
// (combined in a fixed order from partials every CTA pushes into every
// other's shared memory), and p at the next child's token, which the residual
// pass of the CTA owning that token publishes with the sums.  A CTA reads only
// its own slice of the logits, proposals and residual rows.
//
// Exchanges: each CTA (or each warp of each CTA) stores its 16-byte partial
// into a slot of every CTA of the cluster with st.async, which completes the
// receiver's mbarrier transaction count; a CTA waits on its own mbarrier and
// reads the slots locally.  Two slot sets alternate: a CTA pushes exchange
// k + 2 only after exchange k + 1 completed, that is after every CTA pushed
// k + 1, which each does only after its threads have read exchange k.
//
// Staged (`staged`, when the slices fit): each CTA holds three slice buffers
// in shared memory.  One holds the row the current distribution comes from
// (the logits of the node being expanded, or the last residual); the others
// hold the proposals of the child being tested and of its next sibling,
// fetched ahead.  A rejection writes the residual max(0, p - q) over the
// tested child's proposals, which are not needed again, and that buffer
// becomes the distribution's row; the old row's buffer is free.  Slices move
// by bulk asynchronous copies counted on one mbarrier per buffer.  Otherwise
// the slices are read from global memory and the residual rows live in the
// workspace.
__global__ void __launch_bounds__(kMssThreads, 2)
    mss_verify_kernel(const float* __restrict__ llm_logits, const float* __restrict__ ssm_probs,
                      int64_t V, const int32_t* __restrict__ tokens,
                      const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                      const float* __restrict__ u_acc, const float* __restrict__ u_smp, float inv_t,
                      int top_k, float top_p, int ncl, int vec, int staged,
                      float* __restrict__ resid_all, int32_t* __restrict__ path,
                      int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                      int32_t* __restrict__ n_tried, int32_t* __restrict__ status) {
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ int32_t tok_s[TSV_MAX_NODES], par_s[TSV_MAX_NODES];
  __shared__ float ua_s[TSV_MAX_NODES], qx_s[TSV_MAX_NODES], lx_s[TSV_MAX_NODES];
  __shared__ float red[128];
  __shared__ F2 scan_s[kMssWarps];
  __shared__ __align__(16) float pub[2][4];  // exchange slots, alternating
  __shared__ int bad, bad_tok;
  __shared__ int pick_s, last_s;
  __shared__ __align__(8) uint64_t cbar[3];  // staged copies: one barrier per slice buffer
  __shared__ __align__(8) uint64_t xbar[2];  // exchanges, alternating
  __shared__ __align__(16) float4 xslot[2][kMssMaxCluster * kMssWarps];
  __shared__ SelSmem sel;
  extern __shared__ __align__(128) float mss_dyn[];
  const bool warped = top_k > 0 || top_p < 1.0f;
  const int b = blockIdx.x / ncl;
  const int rank = blockIdx.x - b * ncl;  // == %cluster_ctarank for 1-D clusters of ncl
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const int lane = tid & 31;
  if (tid == 0) {
    pick_s = INT32_MAX;
    last_s = -1;
    if (staged)
      for (int i = 0; i < 3; ++i) mbar_init(&cbar[i], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_fence_init();
  }
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;

  // This CTA's slice (a multiple of 4 long, so 16-byte aligned rows stay aligned).
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t lo = min(V, (int64_t)rank * per), hi = min(V, lo + per);
  const int64_t n4 = (hi - lo) >> 2;  // full groups
  const int64_t per_al = (per + 31) & ~int64_t(31);
  const uint32_t slice_bytes = (uint32_t)((hi - lo) * 4);  // a multiple of 16 when staged
  // Staged buffers (bookkeeping identical in every thread): buffer pb holds
  // the distribution's row; node_of[j] is the child whose proposals buffer j
  // holds or receives (-1: none); pend[j]: a copy into j not yet waited for;
  // par[j]: parity of the next phase of j's barrier.
  auto buf = [&](int j) { return mss_dyn + (size_t)j * (size_t)per_al; };
  int pb = 0;
  int node_of[3] = {-1, -1, -1};
  bool pend[3] = {false, false, false};
  uint32_t par_bar[3] = {0u, 0u, 0u};
  bool tmo = false;
  auto ready = [&](int j) {  // the copy into buffer j (if any) has landed
    if (pend[j]) {
      if (!mbar_wait(&cbar[j], par_bar[j], nullptr)) tmo = true;
      par_bar[j] ^= 1u;
      pend[j] = false;
    }
  };
  // Thread 0 copies this CTA's slice of a global row into buffer j.  Every
  // thread is done reading j (a barrier since) and has fenced its writes.
  auto issue_copy = [&](int j, const float* row) {
    if (pend[j]) {  // a copy still in flight into j lands first ...
      ready(j);
      // ... and every thread has seen that phase complete before the next
      // one can (a waiter that slept through both would wait for a third).
      __syncthreads();
    }
    if (tid == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&cbar[j], slice_bytes);
      for (uint32_t o = 0; o < slice_bytes; o += kBulkChunk)
        bulk_copy_g2s(buf(j) + o / 4, row + lo + o / 4, min(kBulkChunk, slice_bytes - o), &cbar[j]);
    }
    pend[j] = true;
  };
  auto q_buffer_of = [&](int c) {
    for (int j = 0; j < 3; ++j)
      if (j != pb && node_of[j] == c) return j;
    return -1;
  };
  // A buffer other than pb and `not_j`, preferring one with no copy in flight.
  auto free_buffer = [&](int not_j) {
    int pick = -1;
    for (int j = 0; j < 3; ++j)
      if (j != pb && j != not_j && (pick < 0 || (pend[pick] && !pend[j]))) pick = j;
    return pick;
  };
  auto q_issue = [&](int j, int c) {
    issue_copy(j, ssm_probs + (size_t)(off + c) * (size_t)V);
    node_of[j] = c;
  };
  // Row of node u into buffer pb, and the proposals of its first child c.
  auto stage_row = [&](int u, int c) {
    issue_copy(pb, llm_logits + (size_t)(off + u) * (size_t)V);
    node_of[pb] = -1;
    if (c >= 0 && q_buffer_of(c) < 0) q_issue(free_buffer(-1), c);
  };
  auto drain = [&]() {  // no copy may be in flight when the CTA leaves
    if (!staged) return;
    for (int j = 0; j < 3; ++j) ready(j);
  };
  __syncthreads();  // barriers initialised ...
  cluster_sync_all();  // ... in every CTA of the cluster, before anyone pushes
  // Node 0 is the root and node 1 (if any) its first child in every valid
  // tree: their slices travel while the tree is read and checked.
  if (staged && n >= 1) stage_row(0, n >= 2 ? 1 : -1);

  // One parallel step reads every node's parent, token and accept uniform,
  // and checks them: a single root at node 0, every other parent earlier in
  // the order (else TSV_ERR_BAD_TREE), tokens in [0, V) (else
  // TSV_ERR_INVALID_ARG; tree errors take precedence).
  if (tid == 0) {
    bad = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
    bad_tok = 0;
  }
  __syncthreads();
  if (bad == 0) {
    for (int i = tid; i < n; i += T) {
      const int p = parent[off + i];
      const int x = i > 0 ? tokens[off + i] : 0;
      const float ua = i > 0 ? u_acc[off + i] : 0.f;
      par_s[i] = p;
      if (!((i == 0) ? (p == -1) : (p >= 0 && p < i))) atomicMax(&bad, TSV_ERR_BAD_TREE);
      if (i > 0) {
        tok_s[i] = x;
        ua_s[i] = ua;
        if (x < 0 || (int64_t)x >= V) bad_tok = TSV_ERR_INVALID_ARG;
      }
    }
  }
  __syncthreads();
  const int code = bad ? bad : bad_tok;
  if (code) {
    drain();
    if (rank == 0)
      fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                   status + b, code);
    return;  // uniform over the cluster: every CTA sees the same tree
  }
  // Per child c: q_c(x_c) and the parent row's logit at x_c, loaded now and
  // stored once the root's row statistics are done (the loads travel
  // meanwhile; the first accept test is the first use).
  static_assert(kMssThreads >= TSV_MAX_NODES, "one child per thread");
  float my_qx = 0.f, my_lx = 0.f;
  if (tid >= 1 && tid < n) {
    my_qx = __ldg(ssm_probs + (size_t)(off + tid) * (size_t)V + tok_s[tid]);
    my_lx = __ldg(llm_logits + (size_t)(off + par_s[tid]) * (size_t)V + tok_s[tid]);
  }
  // The lowest-index child of p after node `from` (children follow their
  // parent in the order), or -1: a ballot scan by the calling warp; every
  // warp finds the same node.
  auto next_child = [&](int p, int from) {
    for (int base = from + 1; base < n; base += 32) {
      const int c = base + lane;
      const uint32_t bal = __ballot_sync(0xffffffffu, c < n && par_s[c] == p);
      if (bal) return base + __ffs(bal) - 1;
    }
    return -1;
  };

  float* resid[2] = {resid_all + (size_t)b * 2 * (size_t)V, resid_all + ((size_t)b * 2 + 1) * (size_t)V};
  int xk = 0;  // exchanges of the warped support so far (the same count in every CTA)
  int xp = 0;  // pushed exchanges so far (the same count in every CTA)
  uint32_t xpar = 0u;  // bit s: parity of the next phase of xbar[s]
  // Pushed exchange: `per_warp` false, one float4 per CTA (slot = rank);
  // true, one per warp of every CTA (slot = rank * kMssWarps + warp).
  // Returns the slots once all have landed.
  auto push = [&](float4 v, bool per_warp) -> const float4* {
    const int s = xp & 1;
    const int slots = per_warp ? ncl * kMssWarps : ncl;
    if (tid == 0) mbar_arrive_expect_tx(&xbar[s], (uint32_t)slots * 16u);
    const int w = tid >> 5;
    if (per_warp ? lane < ncl : tid < ncl) {
      const int dst = per_warp ? lane : tid;
      const int slot = per_warp ? rank * kMssWarps + w : rank;
      st_async_v4(mapa_shared(smem_u32(&xslot[s][slot]), (uint32_t)dst), v,
                  mapa_shared(smem_u32(&xbar[s]), (uint32_t)dst));
    }
    if (!mbar_wait(&xbar[s], (xpar >> s) & 1u, nullptr)) tmo = true;
    xpar ^= 1u << s;
    ++xp;
    return xslot[s];
  };
  // Node u's logits, this CTA's slice.
  auto logits_of = [&](int u) {
    return staged ? Slice{buf(pb), lo} : Slice{llm_logits + (size_t)(off + u) * (size_t)V, 0};
  };

  // Row statistics of node u's logits: m = max(l / T), s = sum exp(l / T - m)
  // over the kept tokens (all tokens unless warped), and the boundary
  // (tau, ycut) of the kept set.  Staged, the row's slice is left holding
  // weights w(y) with p(y) = w(y) * wscale: exp(l / T - m_local) (0 for tokens
  // the warp drops), so later passes multiply instead of exponentiating.
  float m_u = 0.f, inv_s = 0.f, tau = -INFINITY, wscale = 0.f;
  int ycut = INT32_MAX;
  auto row_stats = [&](int u) {
    if (staged) ready(pb);
    const Slice lrow = logits_of(u);
    float m = -INFINITY;
    for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
      float4 v[kMssGroups];
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k) {
        const int64_t g = g0 + (int64_t)k * T;
        if (g < n4) v[k] = lrow.ld4(lo + 4 * g, vec);
      }
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k)
        if (g0 + (int64_t)k * T < n4)
#pragma unroll
          for (int e = 0; e < 4; ++e) m = fmaxf(m, at(v[k], e) * inv_t);
    }
    for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) m = fmaxf(m, lrow[y] * inv_t);
    m = block_max(m, red);
    if (warped) {
      const float4* e = push(make_float4(m, 0.f, 0.f, 0.f), false);
      float M = -INFINITY;
      for (int r = 0; r < ncl; ++r) M = fmaxf(M, e[r].x);
      const Support sp = warped_support(lrow, V, lo, hi, inv_t, M, top_k, top_p, ncl, rank, xk, pub, sel);
      m_u = M;
      inv_s = f2_inv(sp.S);
      tau = sp.tau;
      ycut = sp.ycut;
      if (staged) {  // weights relative to the row maximum M
        float* w = buf(pb);
        for (int64_t y = lo + tid; y < hi; y += T) {
          const float l = w[y - lo];
          w[y - lo] = kept(l, y, tau, ycut) ? exp_diff(l * inv_t, M) : 0.f;
        }
        wscale = inv_s;
        fence_proxy_async_smem();  // the slice may be overwritten by a later copy
        __syncthreads();
      }
      return;
    }
    CompSum acc;
    for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
      float4 v[kMssGroups];
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k) {
        const int64_t g = g0 + (int64_t)k * T;
        if (g < n4) v[k] = lrow.ld4(lo + 4 * g, vec);
      }
#pragma unroll
      for (int k = 0; k < kMssGroups; ++k) {
        const int64_t g = g0 + (int64_t)k * T;
        if (g < n4) {
          float4 w;
          w.x = exp_diff(v[k].x * inv_t, m);
          w.y = exp_diff(v[k].y * inv_t, m);
          w.z = exp_diff(v[k].z * inv_t, m);
          w.w = exp_diff(v[k].w * inv_t, m);
          acc.add(w.x);
          acc.add(w.y);
          acc.add(w.z);
          acc.add(w.w);
          if (staged) *reinterpret_cast<float4*>(buf(pb) + 4 * g) = w;
        }
      }
    }
    for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) {
      const float w = exp_diff(lrow[y] * inv_t, m);
      acc.add(w);
      if (staged) buf(pb)[y - lo] = w;
    }
    if (staged) fence_proxy_async_smem();  // the slice may be overwritten by a later copy
    F2 s = warp_sum_f2(comp_value(acc));
    // Combine the warp partials (identical in every CTA):
    // M = max m_i, S = sum s_i e^(m_i - M).
    const float4* e = push(make_float4(m, s.hi, s.lo, 0.f), true);
    const int cnt = ncl * kMssWarps;
    const float4 e0 = lane < cnt ? e[lane] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    const float4 e1 = lane + 32 < cnt ? e[lane + 32] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    float M = fmaxf(e0.x, e1.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    F2 S{0.f, 0.f};
    if (e0.x != -INFINITY) S = f2_scale(F2{e0.y, e0.z}, exp_diff(e0.x, M));
    if (e1.x != -INFINITY) S = f2_add(S, f2_scale(F2{e1.y, e1.z}, exp_diff(e1.x, M)));
    S = warp_sum_f2(S);
    const float own = m != -INFINITY ? exp_diff(m, M) : 0.f;  // e^(m - M) of this CTA
    m_u = M;
    inv_s = f2_inv(S);
    wscale = own * inv_s;
    tau = -INFINITY;
    ycut = INT32_MAX;
  };

  int u = 0, len = 1, cur = 0, tried = 0;
  bool from_resid = false;  // false: p = softmax(row u); true: p = residual / Z
  bool px_known = false;    // p at the current child's token came with the last exchange
  float px_next = 0.f;
  F2 Z{0.f, 0.f};
  if (rank == 0 && tid == 0) path[off] = 0;
  row_stats(0);
  if (tid >= 1 && tid < n) {
    qx_s[tid] = my_qx;
    lx_s[tid] = my_lx;
  }
  __syncthreads();
  while (true) {
    int accepted = -1;
    int c = next_child(u, u);
    while (c >= 0) {
      // p(x) of the current distribution (fp32, ~2 ulp); the test is exact.
      const float px = px_known ? px_next
                                : (kept(lx_s[c], tok_s[c], tau, ycut) ? exp_diff(lx_s[c] * inv_t, m_u) * inv_s : 0.f);
      ++tried;
      if (accept_test(ua_s[c], qx_s[c], px)) {
        accepted = c;
        break;
      }
      // Rejected: residual pass over the slice, r = max(0, p - q).  The owner
      // of the next child's token records r and p there for the exchange.
      const int cn = next_child(u, c);
      const int64_t xn = cn >= 0 ? (int64_t)tok_s[cn] : -1;
      const int nxt = cur ^ 1;
      // p(y) = source(y) * pscale, except on a logits row read from global
      // memory, where it is exponentiated here.
      const float pscale = from_resid ? f2_inv(Z) : wscale;
      Slice src, q;
      float* rout;
      int64_t rout_off;
      int qj = -1;  // staged: the buffer of c's proposals, then of the residual
      if (staged) {
        qj = q_buffer_of(c);
        if (qj < 0) {  // not fetched ahead
          qj = free_buffer(-1);
          q_issue(qj, c);
        }
        if (cn >= 0 && q_buffer_of(cn) < 0) q_issue(free_buffer(qj), cn);  // the next sibling's, ahead
        ready(qj);
        src = Slice{buf(pb), lo};
        q = Slice{buf(qj), lo};
        rout = buf(qj);  // over q: every element is read, then written, by one thread
        rout_off = lo;
      } else {
        src = from_resid ? Slice{resid[cur], 0} : logits_of(u);
        q = Slice{ssm_probs + (size_t)(off + c) * (size_t)V, 0};
        rout = resid[nxt];
        rout_off = 0;
      }
      CompSum acc;
      float r_x = 0.f, p_x = 0.f;
      for (int64_t g0 = tid; g0 < n4; g0 += (int64_t)T * kMssGroups) {
        float4 a[kMssGroups], qq[kMssGroups];
#pragma unroll
        for (int k = 0; k < kMssGroups; ++k) {
          const int64_t g = g0 + (int64_t)k * T;
          if (g < n4) {
            a[k] = src.ld4(lo + 4 * g, vec);
            qq[k] = q.ld4(lo + 4 * g, vec);
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
              const float py = staged || from_resid
                                   ? at(a[k], e) * pscale
                                   : (kept(at(a[k], e), y + e, tau, ycut)
                                          ? exp_diff(at(a[k], e) * inv_t, m_u) * inv_s : 0.f);
              r[e] = fmaxf(py - at(qq[k], e), 0.0f);
              acc.add(r[e]);
              if (y + e == xn) {
                r_x = r[e];
                p_x = py;
              }
            }
            float* o = rout + (y - rout_off);
            if (vec) {
              *reinterpret_cast<float4*>(o) = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) o[e] = r[e];
            }
          }
        }
      }
      for (int64_t y = lo + 4 * n4 + tid; y < hi; y += T) {
        const float a = src[y];
        const float py = staged || from_resid
                             ? a * pscale
                             : (kept(a, y, tau, ycut) ? exp_diff(a * inv_t, m_u) * inv_s : 0.f);
        const float r = fmaxf(py - q[y], 0.0f);
        rout[y - rout_off] = r;
        acc.add(r);
        if (y == xn) {
          r_x = r;
          p_x = py;
        }
      }
      if (staged) fence_proxy_async_smem();  // the residual may be overwritten by a later copy
      // Warp partials, then every warp of every CTA combines them in the
      // same order (r and p at xn: one owner, the rest add zeros).
      const F2 zs = warp_sum_f2(comp_value(acc));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        r_x += __shfl_xor_sync(0xffffffffu, r_x, o);
        p_x += __shfl_xor_sync(0xffffffffu, p_x, o);
      }
      const float4* e = push(make_float4(zs.hi, zs.lo, r_x, p_x), true);
      const int cnt = ncl * kMssWarps;
      const float4 e0 = lane < cnt ? e[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 e1 = lane + 32 < cnt ? e[lane + 32] : make_float4(0.f, 0.f, 0.f, 0.f);
      F2 Znew = warp_sum_f2(f2_add(F2{e0.x, e0.y}, F2{e1.x, e1.y}));
      float rxn = e0.z + e1.z, pxn = e0.w + e1.w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        rxn += __shfl_xor_sync(0xffffffffu, rxn, o);
        pxn += __shfl_xor_sync(0xffffffffu, pxn, o);
      }
      if (staged) node_of[qj] = -1;  // c's proposals are spent
      if (Znew.hi > 0.f) {  // else p = q up to rounding: keep p
        cur = nxt;
        if (staged) pb = qj;  // the residual is the distribution's row now
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
    if (staged) stage_row(u, next_child(u, u));
    row_stats(u);
  }

  pdl_trigger();  // the walk is done: let the next kernel be scheduled
  // Bonus token: smallest y with cumsum(w)[y] > u_smp[u] * sum(w), w = the
  // unnormalised current distribution.  Each thread owns a contiguous run of
  // its CTA's slice; runs and slices are in vocabulary order.
  {
    const Slice wsrc = staged ? Slice{buf(pb), lo} : (from_resid ? Slice{resid[cur], 0} : logits_of(u));
    const int64_t per_t = ((((hi - lo) + T - 1) / T) + 3) & ~int64_t(3);
    const int64_t tlo = min(hi, lo + (int64_t)tid * per_t), thi = min(hi, tlo + per_t);
    const float bscale = from_resid ? 1.f : wscale;  // staged weights to one common scale
    auto weight = [&](float a, int64_t y) {
      if (staged) return a * bscale;
      return from_resid ? a : (kept(a, y, tau, ycut) ? exp_diff(a * inv_t, m_u) : 0.f);
    };
    CompSum acc;
    int64_t last_pos = -1;
    {
      int64_t y = tlo;
      for (; y + 4 <= thi; y += 4) {
        const float4 a = wsrc.ld4(y, vec);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w = weight(at(a, e), y + e);
          acc.add(w);
          if (w > 0.0f) last_pos = y + e;
        }
      }
      for (; y < thi; ++y) {
        const float w = weight(wsrc[y], y);
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
    const float4* e = push(make_float4(cta_total.hi, cta_total.lo, __int_as_float(last_s), 0.f), false);
    F2 base{0.f, 0.f}, total{0.f, 0.f};
    int last_all = -1;
    for (int r = 0; r < ncl; ++r) {  // in rank order, identical in every CTA
      const F2 t{e[r].x, e[r].y};
      if (r < rank) base = f2_add(base, t);
      total = f2_add(total, t);
      last_all = max(last_all, __float_as_int(e[r].z));
    }
    const F2 excl = f2_add(f2_add(base, wbase), wexcl);
    const F2 target = f2_scale(total, __ldg(u_smp + off + u));
    if (mine.hi > 0.f && !f2_lt(target, excl) && f2_lt(target, f2_add(excl, mine))) {
      // This run holds the crossing; walk it in order.
      int64_t pick = -1;
      CompSum run;
      for (int64_t y = tlo; y < thi; ++y) {
        const float w = weight(wsrc[y], y);
        run.add(w);
        if (f2_lt(target, f2_add(excl, comp_value(run)))) {
          pick = y;
          break;
        }
      }
      if (pick < 0) pick = last_pos;  // rounding inside the run
      atomicMin(&pick_s, (int)pick);
    }
    drain();
    __syncthreads();
    const float4* e2 = push(make_float4(__int_as_float(pick_s), tmo ? 1.f : 0.f, 0.f, 0.f), false);
    if (rank == 0 && tid == 0) {
      int pick = INT32_MAX;
      bool timed_out = tmo;
      for (int r = 0; r < ncl; ++r) {
        pick = min(pick, __float_as_int(e2[r].x));
        timed_out = timed_out || e2[r].y != 0.f;
      }
      // No crossing (rounding left the target at the total): last positive entry.
      bonus[b] = pick != INT32_MAX ? pick : last_all;
      accept_len[b] = len - 1;
      if (n_tried) n_tried[b] = tried;
      status[b] = timed_out ? TSV_ERR_TIMEOUT : TSV_OK;
    }
    // Every push into this CTA has landed (the last wait counted them all) and
    // it reads no other CTA's memory from here on: it may leave.
  }
  if (rank == 0)
    for (int i = len + tid; i < n; i += T) path[off + i] = -1;
}

// ------------------------------------------------------------------ tree construction

// Expansion step (SpecInfer §3, expansion-based token trees): row f of the
// frontier's SSM logits gets its k largest-logit tokens as children, larger
// first, equal logits by lower token index.  A row is split over a cluster
// of CTAs when the frontier is small: for k <= 8 each CTA makes one pass over
// its slice with per-thread top-k lists and rank 0 merges the CTAs' lists;
// wider expansions use the same selection as the warped support (a CTA
// launched without a cluster is a cluster of one).
constexpr int kExpandSmallK = 8;  // widest expansion done in one pass over the row

__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Top-k of entries [lo, hi) of one row for k <= KP <= kExpandSmallK, in one
// pass: every thread keeps its KP best (value, index) sorted in registers;
// then k rounds pick the best head among the 256 lists (a block-wide argmax in
// ranking order).  Entry j of the result goes to (out_v[j], out_i[j]) (thread
// 0 writes; -inf / INT32_MAX when the slice holds fewer than k entries).
template <int KP>
__device__ void expand_small(const float* __restrict__ row, int64_t lo, int64_t hi, int k,
                             float* __restrict__ out_v, int32_t* __restrict__ out_i, float* lv, int* li,
                             float* rv, int* ri) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float bv[KP];
  int bi[KP];
#pragma unroll
  for (int i = 0; i < KP; ++i) {
    bv[i] = -INFINITY;
    bi[i] = INT32_MAX;
  }
  auto offer = [&](float v, int y) {
    if (ranks_before(v, y, bv[KP - 1], bi[KP - 1])) {
      bv[KP - 1] = v;
      bi[KP - 1] = y;
#pragma unroll
      for (int i = KP - 1; i > 0; --i) {
        if (ranks_before(bv[i], bi[i], bv[i - 1], bi[i - 1])) {
          const float tv = bv[i];
          bv[i] = bv[i - 1];
          bv[i - 1] = tv;
          const int ti = bi[i];
          bi[i] = bi[i - 1];
          bi[i - 1] = ti;
        }
      }
    }
  };
  // 16-byte loads, eight in flight per thread, when the slice is aligned
  // (lo is a multiple of 4).
  constexpr int kInFlight = 8;
  const bool vec = ((lo & 3) == 0) && ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
  const int64_t n4 = vec ? (hi - lo) / 4 : 0;
  const float4* r4 = reinterpret_cast<const float4*>(row + lo);
  for (int64_t g0 = tid; g0 < n4; g0 += kInFlight * kMssThreads) {
    float4 a[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u)
      if (g0 + u * kMssThreads < n4) a[u] = __ldg(r4 + g0 + u * kMssThreads);
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int64_t g = g0 + u * kMssThreads;
      if (g < n4) {
        const int y = (int)(lo + 4 * g);
        offer(a[u].x, y);
        offer(a[u].y, y + 1);
        offer(a[u].z, y + 2);
        offer(a[u].w, y + 3);
      }
    }
  }
  for (int64_t y = lo + 4 * n4 + tid; y < hi; y += kMssThreads) offer(__ldg(row + y), (int)y);
#pragma unroll
  for (int i = 0; i < KP; ++i) {
    lv[tid * KP + i] = bv[i];
    li[tid * KP + i] = bi[i];
  }
  __syncthreads();
  int pos = 0;
  for (int j = 0; j < k; ++j) {
    float v = pos < KP ? lv[tid * KP + pos] : -INFINITY;
    int id = pos < KP ? li[tid * KP + pos] : INT32_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, id, o);
      if (ranks_before(ov, oi, v, id)) {
        v = ov;
        id = oi;
      }
    }
    if (lane == 0) {
      rv[warp] = v;
      ri[warp] = id;
    }
    __syncthreads();
    float bvv = rv[0];
    int bid = ri[0];
    for (int ww = 1; ww < kMssWarps; ++ww)
      if (ranks_before(rv[ww], ri[ww], bvv, bid)) {
        bvv = rv[ww];
        bid = ri[ww];
      }
    if (tid == 0) {
      out_v[j] = bvv;
      out_i[j] = bid;
    }
    if (pos < KP && li[tid * KP + pos] == bid) ++pos;  // indices are unique: one list advances
    __syncthreads();
  }
}

// One frontier row per cluster of `ncl` CTAs (ncl = 1: one CTA), CTA rank r
// taking vocabulary slice r.  k <= 8: every CTA finds its slice's top-k, rank
// 0 merges the ncl lists through distributed shared memory.  Wider: the
// cluster runs the warped support's selection (maximum first, exchanged).
__global__ void __launch_bounds__(kMssThreads)
    tree_expand_kernel(const float* __restrict__ logits, int64_t V, int k, int ncl,
                       int32_t* __restrict__ tokens) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ __align__(16) float pub[2][4];
  __shared__ SelSmem sel;
  __shared__ float red[128];
  __shared__ float lv[kMssThreads * kExpandSmallK];
  __shared__ int li[kMssThreads * kExpandSmallK];
  __shared__ float rv[kMssWarps];
  __shared__ int ri[kMssWarps];
  __shared__ float top_v[kExpandSmallK];
  __shared__ int32_t top_i[kExpandSmallK];
  const int f = blockIdx.x / ncl;
  const int rank = blockIdx.x - f * ncl;  // == %cluster_ctarank for 1-D clusters of ncl
  const float* row = logits + (size_t)f * (size_t)V;
  int32_t* out = tokens + (size_t)f * k;
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t lo = min(V, (int64_t)rank * per), hi = min(V, lo + per);
  if (k <= kExpandSmallK) {
    if (k <= 1) expand_small<1>(row, lo, hi, k, top_v, top_i, lv, li, rv, ri);
    else if (k <= 2) expand_small<2>(row, lo, hi, k, top_v, top_i, lv, li, rv, ri);
    else if (k <= 4) expand_small<4>(row, lo, hi, k, top_v, top_i, lv, li, rv, ri);
    else expand_small<8>(row, lo, hi, k, top_v, top_i, lv, li, rv, ri);
    if (ncl == 1) {
      if (threadIdx.x < k) out[threadIdx.x] = top_i[threadIdx.x];
      return;
    }
    __syncthreads();
    cluster_sync_all();  // every CTA's list is in its shared memory
    if (rank == 0 && threadIdx.x < 32) {
      // The ncl lists (k entries each, at most 64 in all): lane l holds
      // entries l and l + 32; k rounds of a warp argmax in ranking order.
      const int lane = threadIdx.x, total = ncl * k;
      float v0 = -INFINITY, v1 = -INFINITY;
      int i0 = INT32_MAX, i1 = INT32_MAX;
      if (lane < total) {
        v0 = ld_dsmem_f32(mapa_shared(smem_u32(&top_v[lane % k]), (uint32_t)(lane / k)));
        i0 = ld_dsmem_s32(mapa_shared(smem_u32(&top_i[lane % k]), (uint32_t)(lane / k)));
      }
      if (lane + 32 < total) {
        v1 = ld_dsmem_f32(mapa_shared(smem_u32(&top_v[(lane + 32) % k]), (uint32_t)((lane + 32) / k)));
        i1 = ld_dsmem_s32(mapa_shared(smem_u32(&top_i[(lane + 32) % k]), (uint32_t)((lane + 32) / k)));
      }
      for (int j = 0; j < k; ++j) {
        const bool first = ranks_before(v0, i0, v1, i1) || i1 == INT32_MAX;
        float v = first ? v0 : v1;
        int id = first ? i0 : i1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, o);
          const int oi = __shfl_xor_sync(0xffffffffu, id, o);
          if (ranks_before(ov, oi, v, id)) {
            v = ov;
            id = oi;
          }
        }
        if (lane == 0) out[j] = id;
        if (i0 == id) {  // indices are unique: exactly one entry leaves
          v0 = -INFINITY;
          i0 = INT32_MAX;
        } else if (i1 == id) {
          v1 = -INFINITY;
          i1 = INT32_MAX;
        }
      }
    }
    cluster_sync_all();  // every CTA keeps its list until rank 0 has read it
    return;
  }
  float m = -INFINITY;
  for (int64_t y = lo + threadIdx.x; y < hi; y += kMssThreads) m = fmaxf(m, __ldg(row + y));
  m = block_max(m, red);
  int xk = 0;
  if (ncl > 1) {  // the row maximum over the cluster
    if (threadIdx.x == 0) pub[0][0] = m;
    cluster_sync_all();
    for (int r = 0; r < ncl; ++r) m = fmaxf(m, ld_dsmem_f32(mapa_shared(smem_u32(&pub[0][0]), (uint32_t)r)));
    ++xk;
  }
  warped_support(Slice{row, 0}, V, lo, hi, 1.0f, m, k, 1.0f, ncl, rank, xk, pub, sel);
  if (rank == 0)
    for (int j = threadIdx.x; j < k; j += kMssThreads) out[j] = sel.srt_i[j];
  if (ncl > 1) cluster_sync_all();  // peers' candidate lists were read in the selection
}

// Merge (SpecInfer §3, merge-based token trees): the input trees of request b
// share its root; a node is identified by its token path, so an input node
// maps to the union child of its parent's image that carries its token, or
// becomes a new union node.  Inputs are taken tree by tree, node by node, so
// the union is in creation order (parents first).  Warp 0 walks the nodes;
// a lookup compares 32 union nodes per ballot.
constexpr int kMergeMaxInput = kTreeMergeMaxInput;

__global__ void __launch_bounds__(256)
    tree_merge_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ tokens,
                      const int32_t* __restrict__ tree_offsets, const int32_t* __restrict__ request_trees,
                      int32_t* __restrict__ out_parent, int32_t* __restrict__ out_tokens,
                      int32_t* __restrict__ out_source, int32_t* __restrict__ out_count,
                      int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ int32_t up[TSV_MAX_NODES], ut[TSV_MAX_NODES], usrc[TSV_MAX_NODES];
  __shared__ int32_t ipar[kMergeMaxInput], itok[kMergeMaxInput], imap[kMergeMaxInput];
  __shared__ int bad, ucount_s;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int t0 = request_trees[b], t1 = request_trees[b + 1];
  const int n0 = tree_offsets[t0], total = tree_offsets[t1] - n0;
  if (tid == 0) bad = (t1 <= t0) ? TSV_ERR_BAD_TREE : (total > kMergeMaxInput ? TSV_ERR_UNSUPPORTED : 0);
  __syncthreads();
  if (!bad) {
    for (int i = tid; i < total; i += blockDim.x) {
      ipar[i] = parent[n0 + i];
      itok[i] = tokens[n0 + i];
    }
    for (int t = t0 + tid; t < t1; t += blockDim.x)
      if (tree_offsets[t + 1] <= tree_offsets[t]) atomicMax(&bad, TSV_ERR_BAD_TREE);
  }
  __syncthreads();
  if (!bad) {
    // Each input tree: a root at its first node, every other parent earlier.
    for (int t = t0; t < t1; ++t) {
      const int s = tree_offsets[t] - n0, e = tree_offsets[t + 1] - n0;
      for (int i = s + tid; i < e; i += blockDim.x) {
        const int p = ipar[i];
        if (!((i == s) ? (p == -1) : (p >= 0 && p < i - s))) atomicMax(&bad, TSV_ERR_BAD_TREE);
      }
    }
  }
  __syncthreads();
  if (!bad && tid < 32) {
    const int lane = tid;
    int ucount = 1;
    if (lane == 0) {
      up[0] = -1;
      ut[0] = itok[0];
      usrc[0] = n0;
    }
    for (int t = t0; t < t1 && ucount >= 0; ++t) {
      const int s = tree_offsets[t] - n0, e = tree_offsets[t + 1] - n0;
      if (lane == 0) imap[s] = 0;
      __syncwarp();
      for (int i = s + 1; i < e; ++i) {
        const int mp = imap[s + ipar[i]], tk = itok[i];
        int found = -1;
        for (int j0 = mp + 1; j0 < ucount; j0 += 32) {
          const int j = j0 + lane;
          const uint32_t hit = __ballot_sync(0xffffffffu, j < ucount && up[j] == mp && ut[j] == tk);
          if (hit) {
            found = j0 + __ffs(hit) - 1;
            break;
          }
        }
        if (found < 0) {
          if (ucount >= TSV_MAX_NODES) {
            ucount = -1;  // the union outgrows a verifiable tree
            break;
          }
          if (lane == 0) {
            up[ucount] = mp;
            ut[ucount] = tk;
            usrc[ucount] = n0 + i;
          }
          found = ucount++;
        }
        if (lane == 0) imap[i] = found;
        __syncwarp();
      }
    }
    if (lane == 0) {
      ucount_s = ucount;
      if (ucount < 0) bad = TSV_ERR_UNSUPPORTED;
    }
  }
  __syncthreads();
  const int cnt = bad ? 0 : ucount_s;
  for (int j = tid; j < total; j += blockDim.x) {
    out_parent[n0 + j] = j < cnt ? up[j] : -1;
    out_tokens[n0 + j] = j < cnt ? ut[j] : -1;
    if (out_source) out_source[n0 + j] = j < cnt ? usrc[j] : -1;
  }
  if (tid == 0) {
    out_count[b] = cnt;
    status[b] = bad ? bad : TSV_OK;
  }
}

// CTAs per frontier row: enough to fill the SMs when the frontier is small,
// at most 8 (one portable cluster) and slices of at least kMssMinSlice.
int expand_cluster_size(int64_t V, int32_t F, int num_sms) {
  int64_t c = num_sms / (F > 0 ? F : 1);
  const int64_t cap = (V + kMssMinSlice - 1) / kMssMinSlice;
  c = c < cap ? c : cap;
  c = c < kMssMaxCluster ? c : kMssMaxCluster;
  return (int)(c < 1 ? 1 : c);
}

cudaError_t launch_tree_expand(const float* logits, int64_t V, int32_t F, int32_t k, int32_t* tokens,
                               int num_sms, cudaStream_t st) {
  if (F == 0) return cudaSuccess;
  const int ncl = expand_cluster_size(V, F, num_sms);
  return launch_pdl(tree_expand_kernel, dim3((unsigned)(F * ncl)), dim3(kMssThreads), 0, st,
                    ncl > 1 ? (unsigned)ncl : 0u, logits, V, k, ncl, tokens);
}

cudaError_t launch_tree_merge(const int32_t* parent, const int32_t* tokens, const int32_t* tree_offsets,
                              const int32_t* request_trees, int32_t B, int32_t* out_parent,
                              int32_t* out_tokens, int32_t* out_source, int32_t* out_count,
                              int32_t* status, cudaStream_t st) {
  return launch_pdl(tree_merge_kernel, dim3(B), dim3(256), 0, st, 0u, parent, tokens, tree_offsets, request_trees,
                    out_parent, out_tokens, out_source, out_count, status);
}

int mss_cluster_size(int64_t V) {
  const int64_t c = (V + kMssMinSlice - 1) / kMssMinSlice;
  return (int)(c < 1 ? 1 : (c > kMssMaxCluster ? kMssMaxCluster : c));
}

cudaError_t mss_set_attributes(int device, size_t* staged_limit) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, mss_verify_kernel);
  if (e != cudaSuccess) return e;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  const size_t limit = (size_t)optin > fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
  e = cudaFuncSetAttribute(mss_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
  if (e != cudaSuccess) return e;
  *staged_limit = limit;
  return cudaSuccess;
}

size_t mss_staged_bytes(int64_t V) {
  const int ncl = mss_cluster_size(V);
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t per_al = (per + 31) & ~int64_t(31);
  return (size_t)(3 * per_al * 4);
}

cudaError_t launch_mss_verify(const float* llm_logits, const float* ssm_probs, int64_t V,
                              const int32_t* tokens, const int32_t* parent,
                              const int32_t* node_offsets, const float* u_acc, const float* u_smp,
                              float inv_t, int32_t top_k, float top_p, int32_t B, float* resid,
                              int32_t* path, int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                              int32_t* status, size_t staged_limit, cudaStream_t st) {
  const int ncl = mss_cluster_size(V);
  const int vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(llm_logits) |
                                    reinterpret_cast<uintptr_t>(ssm_probs) |
                                    reinterpret_cast<uintptr_t>(resid)) & 15) == 0;
  // Slices staged in shared memory when three of them fit (bulk copies want
  // the 16-byte alignment `vec` stands for).
  const size_t dyn = mss_staged_bytes(V);
  const int staged = vec && dyn <= staged_limit;
  return launch_pdl(mss_verify_kernel, dim3((unsigned)(B * ncl)), dim3(kMssThreads), staged ? dyn : 0, st,
                    (unsigned)ncl, llm_logits, ssm_probs, V, tokens, parent, node_offsets, u_acc, u_smp, inv_t,
                    top_k, top_p, ncl, vec, staged, resid, path, accept_len, bonus, n_tried, status);
}

}  // namespace tsv
