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

#include <type_traits>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

namespace {

constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxInFlight = 4;
constexpr int kMinSlice = 2048;  // vocab entries per CTA at least
constexpr int64_t kMaxSlice = 16384;  // vocab entries per CTA at most
// Largest slice pulled into L2 at the start (every slice: a 64 KB slice is
// four rounds of the threads' loads, which the bulk prefetch overlaps).
constexpr uint32_t kArgmaxPrefetchMax = (uint32_t)kMaxSlice * 4;

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

// Order-preserving 32-bit key of a float (-0 counts as +0): larger logit,
// larger key.
__device__ __forceinline__ uint32_t order_key(float l) {
  const uint32_t u = __float_as_uint(l + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value, index) as one word whose unsigned order is the argmax order:
// larger value first, equal values by lower index.
__device__ __forceinline__ unsigned long long argmax_word(ArgMax a) {
  return ((unsigned long long)order_key(a.v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)a.i);
}

__device__ __forceinline__ int32_t argmax_word_index(unsigned long long w) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)w);
}

}  // namespace

// Argmax (lowest index on ties) of vocab slice s of logits row `row`, reduced
// over the CTA; the result is valid in thread 0.  Every thread issues all of
// its loads (up to kArgmaxInFlight 16-byte loads) before using any, so a
// slice of up to kArgmaxInFlight * 4 * kArgmaxThreads entries costs one
// memory round trip.  `red` holds one entry per warp.
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
    for (int64_t k = lo4 + threadIdx.x; k < hi4; k += kArgmaxInFlight * kArgmaxThreads) {
      float4 a[kArgmaxInFlight];
#pragma unroll
      for (int u = 0; u < kArgmaxInFlight; ++u)
        if (k + u * kArgmaxThreads < hi4) a[u] = __ldcs(x4 + k + u * kArgmaxThreads);
#pragma unroll
      for (int u = 0; u < kArgmaxInFlight; ++u) {
        if (k + u * kArgmaxThreads < hi4) {
          const int32_t base = (int32_t)((k + u * kArgmaxThreads) << 2);
          best = better(best, ArgMax{a[u].x, base});
          best = better(best, ArgMax{a[u].y, base + 1});
          best = better(best, ArgMax{a[u].z, base + 2});
          best = better(best, ArgMax{a[u].w, base + 3});
        }
      }
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
// per-node results.
struct WalkSmem {
  int32_t par[TSV_MAX_NODES];
  int32_t tok[TSV_MAX_NODES];
  int32_t am[TSV_MAX_NODES];
  int32_t nxt[TSV_MAX_NODES];
};

// The greedy walk of request b from its rows' argmax words: every child c
// whose token equals argmax(parent(c)) proposes itself to its parent with
// atomicMin (lowest index wins), then the chain is followed from the root.
// Run by one whole CTA of kArgmaxThreads threads; thread i holds node i's
// parent pv and token tv (read before, while the argmax words were
// completing).  The words are read and reset to zero (the workspace is left
// as it was found), then three barriers: every node's argmax known and the
// tree checked; proposals made; warp 0 follows the chain and writes the path.
__device__ void greedy_walk_request(int b, int off, int n, unsigned long long* rowbest, int pv, int tv,
                                    int32_t* path, int32_t* accept_len, int32_t* bonus, int32_t* status,
                                    WalkSmem& w) {
  const int T = blockDim.x;
  const int i = threadIdx.x;
  static_assert(TSV_MAX_NODES <= kArgmaxThreads, "one node per thread");
  for (int r = i; r < n; r += T) {
    const unsigned long long word = __ldcg(rowbest + off + r);
    rowbest[off + r] = 0ull;
    if (r < TSV_MAX_NODES) w.am[r] = argmax_word_index(word);
  }
  const int size_code = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
  if (size_code) {  // uniform: n is the same for every thread
    fail_request(path + off, n, accept_len + b, bonus + b, nullptr, status + b, size_code);
    return;
  }
  bool bad = false;
  if (i < n) {
    w.par[i] = pv;
    w.tok[i] = tv;
    w.nxt[i] = INT32_MAX;
    bad = !((i == 0) ? (pv == -1) : (pv >= 0 && pv < i));
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

// Walk-only kernel: one CTA per request (used when N == 0, where no argmax
// CTA exists; every request then has no node and is reported as a bad tree).
__global__ void __launch_bounds__(kArgmaxThreads)
    greedy_walk_kernel(unsigned long long* __restrict__ rowbest, const int32_t* __restrict__ tokens,
                       const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                       int32_t* __restrict__ path, int32_t* __restrict__ accept_len,
                       int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ WalkSmem w;
  const int b = blockIdx.x;
  const int off = node_offsets[b], n = node_offsets[b + 1] - off;
  const int i = threadIdx.x;
  const int pv = i < n ? parent[off + i] : 0, tv = i < n ? tokens[off + i] : 0;
  greedy_walk_request(b, off, n, rowbest, pv, tv, path, accept_len, bonus, status, w);
}

// Fused greedy verification: grid (splits, N).  Each CTA reduces one vocab
// slice of one row and folds its (maximum, lowest index) into the row's
// argmax word with one 64-bit atomicMax; the last CTA to finish among a
// request's rows x slices (an acquire-release counter, no waiting) walks that
// request's tree.  CTA (0, 0) also reports requests that own no rows.  Words
// and counters start at zero and are left at zero.  `beside`: the inputs were
// complete before the preceding kernel on the stream began, so the CTAs start
// while it runs; each walker waits for it before leaving, so this grid still
// completes after it.
// At most 32 registers a thread (8192 a CTA) and under 5 KB of shared memory:
// a CTA fits on an SM beside a running keys-on-lanes attention CTA, so
// verification launched on another stream reads its logits during attention.
__global__ void __launch_bounds__(kArgmaxThreads, 8)
    greedy_verify_kernel(const float* __restrict__ logits, int64_t V, int splits,
                         const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
                         const int32_t* __restrict__ node_offsets, int B,
                         unsigned long long* __restrict__ rowbest, int32_t* __restrict__ counters,
                         int32_t* __restrict__ path, int32_t* __restrict__ accept_len,
                         int32_t* __restrict__ bonus, int32_t* __restrict__ status, int beside) {
  // The slice is pulled into L2 while the previous kernel finishes (or, beside
  // it, while the threads' first loads are in flight): a prefetch reads no
  // value, so it may run ahead of that kernel's writes.
  if (threadIdx.x == 0 && (V & 3) == 0) {
    const int64_t per = slice_len(V, splits);
    const int64_t lo = min(V, (int64_t)blockIdx.x * per), hi = min(V, lo + per);
    const float* src = logits + (size_t)blockIdx.y * (size_t)V + lo;
    const uint32_t bytes = (uint32_t)((hi - lo) * 4);
    if (bytes > 0 && bytes <= kArgmaxPrefetchMax && (reinterpret_cast<uintptr_t>(src) & 15) == 0)
      bulk_prefetch_l2(src, bytes);
  }
  if (beside) pdl_trigger();  // the next kernel may start beside this one too
  else pdl_wait();            // the previous kernel's results are visible from here on
  __shared__ int32_t offs[TSV_MAX_BATCH + 1];
  __shared__ WalkSmem w;
  __shared__ ArgMax red[kArgmaxThreads / 32];
  __shared__ int last;
  const int row = blockIdx.y, s = blockIdx.x;
  // The offsets travel with the first logits loads: stored after the slice.
  static_assert(TSV_MAX_BATCH < kArgmaxThreads, "one offset per thread");
  const int my_off = threadIdx.x <= B ? node_offsets[threadIdx.x] : 0;
  const ArgMax best = slice_argmax(logits, V, splits, row, s, red);
  if (!beside) pdl_trigger();  // this CTA's share of the logits is read: let the next kernel be scheduled
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
  // The request's tree, read by every CTA while its atomics complete: the
  // one that finishes last walks it without another memory round trip.
  const int i = threadIdx.x;
  const int pv = i < n ? __ldg(parent + off + i) : 0, tv = i < n ? __ldg(tokens + off + i) : 0;
  if (threadIdx.x == 0) {
    atomicMax(rowbest + row, argmax_word(best));
    last = atom_add_acq_rel_gpu(counters + b, 1) == n * splits - 1;
  }
  __syncthreads();
  if (!last) return;
  greedy_walk_request(b, off, n, rowbest, pv, tv, path, accept_len, bonus, status, w);
  if (threadIdx.x == 0) counters[b] = 0;
  if (beside && threadIdx.x == 0) pdl_wait();
}

// Slices per row: at least one CTA per SM (a short row is then read in one
// round trip, and few CTAs share a request's counter) and slices of at most
// kMaxSlice entries (long rows: more CTAs, more loads in flight), of at
// least kMinSlice.
int greedy_splits(int64_t V, int32_t N, int num_sms) {
  int64_t s = ((int64_t)num_sms + N - 1) / (N > 0 ? N : 1);
  s = s > (V + kMaxSlice - 1) / kMaxSlice ? s : (V + kMaxSlice - 1) / kMaxSlice;
  const int64_t cap = (V + kMinSlice - 1) / kMinSlice;
  s = s < cap ? s : cap;
  return (int)(s < 1 ? 1 : s);
}

cudaError_t launch_greedy_verify(const float* logits, int64_t V, int32_t N, int splits,
                                 const int32_t* tokens, const int32_t* parent,
                                 const int32_t* node_offsets, int32_t B, unsigned long long* rowbest,
                                 int32_t* counters, int32_t* path, int32_t* accept_len, int32_t* bonus,
                                 int32_t* status, int beside, cudaStream_t st) {
  dim3 grid(splits, N);
  return launch_pdl(greedy_verify_kernel, grid, dim3(kArgmaxThreads), 0, st, 0u, logits, V, splits, tokens, parent,
                    node_offsets, B, rowbest, counters, path, accept_len, bonus, status, beside);
}

cudaError_t launch_greedy_walk(unsigned long long* rowbest, const int32_t* tokens, const int32_t* parent,
                               const int32_t* node_offsets, int32_t B, int32_t* path,
                               int32_t* accept_len, int32_t* bonus, int32_t* status,
                               cudaStream_t st) {
  return launch_pdl(greedy_walk_kernel, dim3(B), dim3(kArgmaxThreads), 0, st, 0u, rowbest, tokens, parent,
                    node_offsets, path, accept_len, bonus, status);
}

// ------------------------------------------------------------------ stochastic

namespace {

constexpr int kMssThreads = 512;  // stochastic verification CTAs: 16 warps, one CTA per SM
constexpr int kMssCompactWarps = 2;  // compact CTAs (leader and one worker) that run beside attention
// Registers a thread: 128 fill an SM's 65536 with 512 threads; the form that
// leaves room for greedy verification beside it takes 112 (8192 left).
constexpr int kMssRegs = 128, kMssRoomRegs = 112;
constexpr int kMssWarps = kMssThreads / 32;
constexpr int kSelThreads = 256;  // tree-expansion CTAs
constexpr int kSelWarps = kSelThreads / 32;
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

template <int kWarps>
__device__ float block_max(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) v = fmaxf(v, red[w]);
  return v;
}

__device__ __forceinline__ F2 shfl_f2(F2 v, int src) {
  return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

__device__ __forceinline__ F2 shfl_up_f2(F2 v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}

// Inclusive prefix sum over the warp's lanes (lane l: lanes 0..l).
__device__ __forceinline__ F2 warp_scan_f2(F2 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const F2 t = shfl_up_f2(v, o);
    if (lane >= o) v = f2_add(t, v);
  }
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

// Shared scratch of the warped support (CTAs of up to kMssThreads threads).
struct SelSmem {
  int hist[2][256];  // per-CTA digit histograms, alternating with the exchanges
  int wsum[kMssWarps];
  int ints[8];
  float cand_v[kMaxTopK];
  int cand_i[kMaxTopK];
  float srt_v[kMaxTopK];
  int srt_i[kMaxTopK];
  F2 tsum[kMssWarps];
  F2 s_cut;
};
static_assert(kSelThreads >= 256 && kMssThreads >= 256, "one histogram bin per thread of the first 256");

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
// cluster runs it in lockstep; `xk` counts the exchanges.  kT threads per CTA.
template <int kT>
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
      if (tid < 256) h[tid] = 0;
      __syncthreads();
      for (int64_t y = lo + tid; y < hi; y += kT) {
        const uint32_t k = order_key(lrow[y]);
        if (pass == 0 || (k >> (shift + 8)) == prefix) atomicAdd(&h[(k >> shift) & 255], 1);
      }
      __syncthreads();
      cluster_sync_all();
      int cnt = 0;  // bin tid's count over the cluster (threads past the 256 bins: none)
      if (tid < 256)
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
      for (int ww = warp + 1; ww < kT / 32; ++ww) sfx += w.wsum[ww];
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
      for (int64_t y = lo + tid; y < hi; y += kT) c += order_key(lrow[y]) == prefix;
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
  for (int64_t y = lo + tid; y < hi; y += kT) {
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
  for (int j = tid; j < P2; j += kT) {
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
      for (int i = tid; i < P2; i += kT) {
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
  const int per = (K + kT - 1) / kT;
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
  for (int ww = 0; ww < kT / 32; ++ww) {
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
// other's shared memory), and p at the next child's token, which the thread
// owning that token publishes with the sums.  A CTA reads only its own slice
// of the logits, proposals and residual rows.
//
// Within a CTA, warp 0 (the leader) runs the walk: it waits for exchanges,
// combines them, takes the accept decisions, keeps the buffer bookkeeping and
// issues the copies.  It hands each vocabulary-wide step to the other warps
// through a descriptor in shared memory and one barrier: the row statistics
// and residual passes to the 15 worker warps, the statistics of a warped row
// and the bonus draw to all 16.  While the workers run a pass, the leader
// prepares the next decision (the next child, its sibling, the owner of the
// sibling's token, the proposal copies), so only the exchange, its combine
// and the accept test lie between two passes.
//
// Exchanges: each CTA (or each worker warp of each CTA) stores its 16-byte
// partial into a slot of every CTA of the cluster with st.async, which
// completes the receiver's mbarrier transaction count; the receiver's leader
// waits on its own mbarrier and reads the slots locally.  Two slot sets
// alternate: a CTA pushes exchange k + 2 only after exchange k + 1 completed,
// that is after every CTA pushed k + 1, which each does only after its
// leader has read exchange k (a step barrier lies between).  The last
// exchange (the bonus token's position) goes to rank 0 alone.
//
// Staged (kStaged, when the slices fit): each CTA holds three slice buffers
// in shared memory.  One holds the row the current distribution comes from
// (the logits of the node being expanded, or the last residual); the others
// hold the proposals of the child being tested and of its next sibling,
// fetched ahead.  A rejection writes the residual max(0, p - q) over the
// tested child's proposals, which are not needed again, and that buffer
// becomes the distribution's row; the old row's buffer is free.  Slices move
// by bulk asynchronous copies counted on one mbarrier per buffer, issued and
// waited for by the leader before the step that reads them; the logits rows
// of a node's first two children are pulled into L2 meanwhile.  Otherwise the
// slices are read from global memory and the residual rows live in the
// workspace.
struct MssStep {
  int kind;        // kStepRow, kStepPass or kStepBonus
  int u;           // the node being expanded
  int src;         // staged: buffer of the distribution's row; else -1 (logits of u) or a residual row
  int qj;          // residual pass, staged: buffer of the proposals, overwritten by the residual
  int c;           // residual pass: the rejected child
  int nxt;         // residual pass, unstaged: the residual row written
  int xs;          // slot set of the step's exchange
  int xn;          // residual pass: the next child's token (-1: none)
  int ycut, len;
  float pscale;    // p(y) = source(y) * pscale (staged or residual rows)
  float m_u, inv_s, tau;  // unstaged logits rows: p(y) from the logit
  float bscale, us;       // bonus: weight scale, sampling uniform
};
constexpr int kStepNone = 0, kStepRow = 1, kStepPass = 2, kStepBonus = 3;

template <bool kStaged, int kWarps, int kRegs>
__global__ void __maxnreg__(kRegs)
    mss_verify_kernel(const float* __restrict__ llm_logits, const float* __restrict__ ssm_probs,
                      int64_t V, const int32_t* __restrict__ tokens,
                      const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offsets,
                      const float* __restrict__ u_acc, const float* __restrict__ u_smp, float inv_t,
                      int top_k, float top_p, int ncl, int vec_in, int beside,
                      float* __restrict__ resid_all, int32_t* __restrict__ path,
                      int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                      int32_t* __restrict__ n_tried, int32_t* __restrict__ status) {
  // The request's offsets are pulled into L2 while the previous kernel
  // finishes (a prefetch reads no value, so it may run ahead of its writes).
  if (threadIdx.x == 0) prefetch_l2(node_offsets + blockIdx.x / ncl);
  // `beside`: the inputs were complete before the preceding kernel on the
  // stream began, so the walk runs alongside that kernel; every CTA's thread
  // 0 waits for it before leaving instead, so this grid still completes
  // after it (the stream order every later kernel relies on).
  if (!beside) pdl_wait();  // the previous kernel's results are visible from here on
  // The next kernel may be scheduled now: it waits for this one's completion
  // itself, and it is launched only once every CTA of this grid has started,
  // so its CTAs never hold SMs this grid still needs.
  pdl_trigger();
  __shared__ int32_t tok_s[TSV_MAX_NODES], par_s[TSV_MAX_NODES];
  __shared__ float ua_s[TSV_MAX_NODES], us_s[TSV_MAX_NODES], qx_s[TSV_MAX_NODES], lx_s[TSV_MAX_NODES];
  constexpr int T = kWarps * 32;
  constexpr int kWorkerWarps = kWarps - 1;     // warps 1..kWarps-1
  constexpr int TW = kWorkerWarps * 32;        // threads of the row statistics and residual passes
  constexpr int kSlots = kMssMaxCluster * kWorkerWarps;
  constexpr bool kWarpedOK = kWarps == kMssWarps;  // the warped support runs on full CTAs only
  static_assert(kWorkerWarps >= 1 && kSlots >= kMssMaxCluster, "a leader and at least one worker");
  __shared__ float red[kWarps];
  __shared__ F2 scan_s[kWarps], wpre_s[kWarps], target_s;
  __shared__ float mx_s;
  __shared__ __align__(16) float pub[2][4];  // exchange slots of the warped support, alternating
  __shared__ int bad, bad_tok, tmo_s, pick_s, last_s;
  __shared__ __align__(8) uint64_t cbar[3];  // staged copies: one barrier per slice buffer
  __shared__ __align__(8) uint64_t xbar[2];  // exchanges, alternating
  __shared__ __align__(16) float4 xslot[2][kSlots];
  __shared__ MssStep dsc[2];                 // step descriptors, alternating
  __shared__ typename std::conditional<kWarpedOK, SelSmem, int>::type sel;
  extern __shared__ __align__(128) float mss_dyn[];
  // 4-float groups in flight per worker: shared memory 3 (2 in the form with
  // fewer registers, which would spill at 3), global memory kMssGroups.
  constexpr int G = kStaged ? (kRegs >= kMssRegs ? 3 : 2) : kMssGroups;
  const bool vec = kStaged || vec_in != 0;     // staged slices are always 16-byte aligned
  const bool warped = top_k > 0 || top_p < 1.0f;
  const int b = blockIdx.x / ncl;
  const int rank = blockIdx.x - b * ncl;  // == %cluster_ctarank for 1-D clusters of ncl
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const bool leader = warp == 0;
  const int wid = tid - 32;  // worker index (warps 1..15)
  const int off = node_offsets[b];
  const int n = node_offsets[b + 1] - off;
  if (tid == 0) {
    pick_s = INT32_MAX;
    last_s = -1;
    tmo_s = 0;
    bad = (n < 1) ? TSV_ERR_BAD_TREE : (n > TSV_MAX_NODES ? TSV_ERR_UNSUPPORTED : 0);
    bad_tok = 0;
    if (kStaged)
      for (int i = 0; i < 3; ++i) mbar_init(&cbar[i], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_fence_init();
  }

  // This CTA's slice (a multiple of 4 long, so 16-byte aligned rows stay aligned).
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t lo = min(V, (int64_t)rank * per), hi = min(V, lo + per);
  const int64_t n4 = (hi - lo) >> 2;  // full groups
  const int64_t per_al = (per + 31) & ~int64_t(31);
  const uint32_t slice_bytes = (uint32_t)((hi - lo) * 4);  // a multiple of 16 when staged
  auto buf = [&](int j) { return mss_dyn + (size_t)j * (size_t)per_al; };
  // Staged bookkeeping, the leader's (identical in its lanes, held in
  // registers): buffer pb holds the distribution's row; 10-bit field j of
  // `nodes` is one more than the child whose proposals buffer j holds or
  // receives (0: none); bit j of `pend`: a copy into j not yet waited for;
  // bit j of `par`: parity of the next phase of j's barrier.  Only lane 0 of
  // the leader waits on these barriers, and the step barrier orders every
  // other thread's reads after its wait.
  int pb = 0;
  uint32_t nodes = 0u, pend = 0u, par = 0u;
  auto node_of = [&](int j) { return (int)((nodes >> (10 * j)) & 1023u) - 1; };
  auto set_node = [&](int j, int c) {
    nodes = (nodes & ~(1023u << (10 * j))) | ((uint32_t)(c + 1) << (10 * j));
  };
  auto land = [&](int j) {  // the copy into buffer j (if any) has landed
    if ((pend >> j) & 1u) {
      if (lane == 0 && !mbar_wait(&cbar[j], (par >> j) & 1u, nullptr)) tmo_s = 1;
      par ^= 1u << j;
      pend &= ~(1u << j);
    }
  };
  // This CTA's slice of a global row into buffer j, which no thread reads any
  // more (an exchange or a barrier since its last use); a copy into j that
  // nobody waited for lands first.
  auto issue_copy = [&](int j, const float* row) {
    land(j);
    if (lane == 0) {
      mbar_arrive_expect_tx(&cbar[j], slice_bytes);
      for (uint32_t o = 0; o < slice_bytes; o += kBulkChunk)
        bulk_copy_g2s(buf(j) + o / 4, row + lo + o / 4, min(kBulkChunk, slice_bytes - o), &cbar[j]);
    }
    pend |= 1u << j;
  };
  auto q_buffer_of = [&](int c) {
    int r = -1;
#pragma unroll
    for (int j = 2; j >= 0; --j)
      if (j != pb && node_of(j) == c) r = j;
    return r;
  };
  // A buffer other than pb, preferring one with no copy in flight.
  auto free_buffer = [&]() {
    int pick = -1;
#pragma unroll
    for (int j = 0; j < 3; ++j)
      if (j != pb && (pick < 0 || (((pend >> pick) & 1u) && !((pend >> j) & 1u)))) pick = j;
    return pick;
  };
  auto q_issue = [&](int j, int c) {
    issue_copy(j, ssm_probs + (size_t)(off + c) * (size_t)V);
    set_node(j, c);
  };
  // Row of node u into buffer pb, and the proposals of its first child c.
  auto stage_row = [&](int u, int c) {
    issue_copy(pb, llm_logits + (size_t)(off + u) * (size_t)V);
    set_node(pb, -1);
    if (c >= 0 && q_buffer_of(c) < 0) q_issue(free_buffer(), c);
  };
  auto drain = [&]() {  // leader: no copy may be in flight when the CTA leaves
    if (kStaged)
      for (int j = 0; j < 3; ++j) land(j);
  };
  __syncthreads();  // barriers initialised ...
  cluster_arrive_release();  // ... and every CTA waits for the others' before its first push
  // Node 0 is the root and node 1 (if any) its first child in every valid
  // tree: their slices travel while the tree is read and checked.
  if (kStaged && leader && n >= 1) stage_row(0, n >= 2 ? 1 : -1);

  // One parallel step reads every node's parent, token and uniforms, and
  // checks them: a single root at node 0, every other parent earlier in the
  // order (else TSV_ERR_BAD_TREE), tokens in [0, V) (else TSV_ERR_INVALID_ARG;
  // tree errors take precedence).
  for (int i = tid; bad == 0 && i < n; i += T) {
    const int p = parent[off + i];
    const int x = i > 0 ? tokens[off + i] : 0;
    const float ua = i > 0 ? u_acc[off + i] : 0.f;
    const float us = u_smp[off + i];
    par_s[i] = p;
    us_s[i] = us;
    if (!((i == 0) ? (p == -1) : (p >= 0 && p < i))) atomicMax(&bad, TSV_ERR_BAD_TREE);
    if (i > 0) {
      tok_s[i] = x;
      ua_s[i] = ua;
      if (x < 0 || (int64_t)x >= V) bad_tok = TSV_ERR_INVALID_ARG;
    }
  }
  __syncthreads();
  const int code = bad ? bad : bad_tok;
  cluster_wait_acquire();
  if (code) {  // uniform over the cluster: every CTA sees the same tree
    if (leader) drain();
    if (rank == 0)
      fail_request(path + off, n, accept_len + b, bonus + b, n_tried ? n_tried + b : nullptr,
                   status + b, code);
    if (beside && tid == 0) pdl_wait();
    return;
  }
  // The lowest-index child of p after node `from` (children follow their
  // parent in the order), or -1: a ballot scan by the calling warp.
  auto next_child = [&](int p, int from) {
    for (int base = from + 1; base < n; base += 32) {
      const int c = base + lane;
      const uint32_t bal = __ballot_sync(0xffffffffu, c < n && par_s[c] == p);
      if (bal) return base + __ffs(bal) - 1;
    }
    return -1;
  };
  // The logits rows of u's first two children (the next row the walk reads
  // if one of them is accepted) into L2; called by one warp.
  auto prefetch_children = [&](int u) {
    if (!kStaged || slice_bytes == 0) return;
    const int c1 = next_child(u, u);
    const int c2 = c1 >= 0 ? next_child(u, c1) : -1;
    const int c = lane == 0 ? c1 : c2;
    if (lane < 2 && c >= 0)
      for (uint32_t o = 0; o < slice_bytes; o += kBulkChunk)
        bulk_prefetch_l2(llm_logits + (size_t)(off + c) * (size_t)V + lo + o / 4, min(kBulkChunk, slice_bytes - o));
  };

  float* const resid0 = resid_all + (size_t)b * 2 * (size_t)V;  // unstaged residual rows 0 and 1
  auto resid_row = [&](int r) { return resid0 + (size_t)r * (size_t)V; };
  int xk = 0;  // exchanges of the warped support so far (the same count in every thread)
  int xp = 0;  // leader: pushed exchanges so far (the same count in every CTA)
  uint32_t xpar = 0u;  // leader: bit s, parity of the next phase of xbar[s]
  // Exchange of one float4 per CTA into slot set xs (slot = rank, sent by
  // threads 0..ncl-1, every thread of the leader calling).
  auto push_cta = [&](float4 v, int xs) {
    if (tid == 0) mbar_arrive_expect_tx(&xbar[xs], (uint32_t)ncl * 16u);
    if (tid < ncl)
      st_async_v4(mapa_shared(smem_u32(&xslot[xs][rank]), (uint32_t)tid), v,
                  mapa_shared(smem_u32(&xbar[xs]), (uint32_t)tid));
  };
  // Exchange of one float4 per worker warp (slot = rank * 15 + warp - 1, sent
  // by lanes 0..ncl-1; v uniform over the warp).  The leader expects the
  // bytes when it releases the step.
  auto push_warp = [&](float4 v, int xs) {
    if (lane < ncl)
      st_async_v4(mapa_shared(smem_u32(&xslot[xs][rank * kWorkerWarps + warp - 1]), (uint32_t)lane), v,
                  mapa_shared(smem_u32(&xbar[xs]), (uint32_t)lane));
  };
  // Leader: waits for the exchange in flight and returns its slots.
  auto push_wait = [&]() -> const float4* {
    const int s = xp & 1;
    if (!mbar_wait(&xbar[s], (xpar >> s) & 1u, nullptr)) tmo_s = 1;
    xpar ^= 1u << s;
    ++xp;
    return xslot[s];
  };

  // The walk's state (the leader's; the statistics of a warped row are
  // computed by every thread).
  int u = 0, len = 1, cur = 0, tried = 0, qj = -1, last = kStepNone;
  int tc = -1, tn = -1, txn = -1, t_oslot = -1;  // next child to test, its next sibling, the sibling's token, owner slot
  int o_slot = -1;          // owner slot of the running residual pass (-1: none)
  bool last_loads = true;   // the children's q_c(x_c) and l(x_c) are still to be read
  bool from_resid = false;  // false: p = softmax(row u); true: p = residual / Z
  bool px_known = false;    // p at the child to test came with the last exchange
  float px_next = 0.f;
  F2 Z{0.f, 0.f};
  // Row statistics of the node being expanded: m_u = max(l / T), inv_s =
  // 1 / sum exp(l / T - m_u) over the kept tokens (all unless warped), the
  // boundary (tau, ycut) of the kept set, and wscale: p(y) = w(y) * wscale
  // for the staged weights w(y) = exp(l / T - m_cta) (m_cta: this CTA's
  // maximum; with warping, M itself).
  float m_u = 0.f, inv_s = 0.f, tau = -INFINITY, wscale = 0.f;
  int ycut = INT32_MAX;

  // Leader, while the step `d` runs: the child to test after it, that
  // child's next sibling and the owner of the sibling's token (its slot in a
  // residual exchange), and the proposal copies of both when a buffer is free
  // (not the distribution's row, not the one the step writes, not one
  // holding either child's proposals).
  auto leader_prep = [&](const MssStep& d) {
    if (last_loads) {  // first step: q_c(x_c) and the parent row's logit at x_c of every child c
      for (int i = 1 + lane; i < n; i += 32) {
        qx_s[i] = __ldg(ssm_probs + (size_t)(off + i) * (size_t)V + tok_s[i]);
        lx_s[i] = __ldg(llm_logits + (size_t)(off + par_s[i]) * (size_t)V + tok_s[i]);
      }
      __syncwarp();
      last_loads = false;
    }
    tc = d.kind == kStepRow ? next_child(u, u) : tn;
    tn = tc >= 0 ? next_child(u, tc) : -1;
    txn = tn >= 0 ? tok_s[tn] : -1;
    t_oslot = -1;
    if (txn >= 0) {  // rank xn / per; there, group (xn - lo') / 4 goes to worker group % TW,
      const int p32 = (int)per, v32 = (int)V;  // a tail element to worker (index past the groups) % TW
      const int orank = txn / p32;
      const int olo = orank * p32, ohi = min(v32, olo + p32), on4 = (ohi - olo) >> 2;
      const int rel = txn - olo;
      const int own = rel < 4 * on4 ? (rel >> 2) % TW : (rel - 4 * on4) % TW;
      t_oslot = orank * kWorkerWarps + (own >> 5);
    }
    if (kStaged) {
      const int busy = d.kind == kStepPass ? d.qj : pb;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int x = k == 0 ? tc : tn;
        if (x < 0 || q_buffer_of(x) >= 0) continue;
        int j = -1;
#pragma unroll
        for (int jj = 0; jj < 3; ++jj) {
          const int nd = node_of(jj);
          if (jj == pb || jj == busy || (nd >= 0 && (nd == tc || nd == tn))) continue;
          if (j < 0 || (((pend >> j) & 1u) && !((pend >> jj) & 1u))) j = jj;
        }
        if (j < 0) break;  // no room now: issued when the child is tested
        q_issue(j, x);
      }
    }
  };

  // Leader: the exchange of the step `d` (unwarped row statistics or a
  // residual pass), combined.
  auto leader_consume = [&](const MssStep& d) {
    const float4* e = push_wait();
    const int cnt = ncl * kWorkerWarps;
    if (d.kind == kStepRow) {
      // M = max m_r, S = sum_r e^(m_r - M) sum_w s_rw: every warp partial of
      // rank r shares its m_r.  Lanes 4r..4r+3 take rank r's slots (warps
      // 4k + lane % 4), sum them, scale once and sum over the ranks.
      static_assert(kMssMaxCluster * 4 == 32 && kWorkerWarps <= 16, "four lanes per rank");
      const int r = lane >> 2;
      float mr = -INFINITY;
      F2 S{0.f, 0.f};
      if (r < ncl) {
        mr = e[r * kWorkerWarps].x;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int w = (lane & 3) + 4 * k;
          if (w < kWorkerWarps) {
            const float4 ev = e[r * kWorkerWarps + w];
            S = f2_add(S, F2{ev.y, ev.z});
          }
        }
      }
      S = f2_add(S, shfl_xor_f2(S, 1));
      S = f2_add(S, shfl_xor_f2(S, 2));
      float M = mr;
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      S = mr != -INFINITY ? f2_scale(S, exp_diff(mr, M)) : F2{0.f, 0.f};
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) S = f2_add(S, shfl_xor_f2(S, o));
      const float m_cta = e[rank * kWorkerWarps].x;
      const float own = m_cta != -INFINITY ? exp_diff(m_cta, M) : 0.f;  // e^(m - M) of this CTA
      m_u = M;
      inv_s = f2_inv(S);
      wscale = own * inv_s;
      tau = -INFINITY;
      ycut = INT32_MAX;
      return;
    }
    // Z = sum of the residual partials (the same order in every CTA); r and
    // p at the next child's token from its owner's slot.
    F2 Zp{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kSlots / 32 + 1; ++k)
      if (lane + 32 * k < cnt) Zp = f2_add(Zp, F2{e[lane + 32 * k].x, e[lane + 32 * k].y});
    const F2 Znew = warp_sum_f2(Zp);
    float rxn = 0.f, pxn = 0.f;
    if (o_slot >= 0) {
      const float4 eo = e[o_slot];
      rxn = eo.z;
      pxn = eo.w;
    }
    if (kStaged) set_node(qj, -1);  // the rejected child's proposals are spent
    if (Znew.hi > 0.f) {  // else p = q up to rounding: keep p
      cur ^= 1;
      if (kStaged) pb = qj;  // the residual is the distribution's row now
      Z = Znew;
      from_resid = true;
      px_next = rxn * f2_inv(Znew);
    } else {
      px_next = pxn;
    }
    px_known = true;
  };

  // Leader: the accept test of child tc (if any) and the next step.
  auto leader_decide = [&](MssStep& d) {
    int kind = kStepRow;  // first: the root's statistics
    if (last != kStepNone) {
      if (tc < 0) {
        kind = kStepBonus;
      } else {
        // p(x) of the current distribution (fp32, ~2 ulp); the test is exact.
        const float px = px_known ? px_next
                                  : (kept(lx_s[tc], tok_s[tc], tau, ycut) ? exp_diff(lx_s[tc] * inv_t, m_u) * inv_s
                                                                           : 0.f);
        ++tried;
        if (accept_test(ua_s[tc], qx_s[tc], px)) {
          u = tc;
          if (rank == 0 && lane == 0) path[off + len] = u;
          ++len;
          from_resid = false;
          px_known = false;
          if (kStaged) stage_row(u, next_child(u, u));
          kind = kStepRow;
        } else {
          kind = kStepPass;
        }
      }
    }
    d.kind = kind;
    d.u = u;
    d.xs = xp & 1;
    d.m_u = m_u;
    d.inv_s = inv_s;
    d.tau = tau;
    d.ycut = ycut;
    d.len = len;
    if (kind == kStepRow) {
      if (kStaged) land(pb);
      d.src = pb;
    } else if (kind == kStepPass) {
      // Rejected: residual pass r = max(0, p - q) over the slice.  p(y) =
      // source(y) * pscale, except on a logits row read from global memory,
      // where it is exponentiated in the pass.
      d.pscale = from_resid ? f2_inv(Z) : wscale;
      d.c = tc;
      d.xn = txn;
      o_slot = t_oslot;
      if (kStaged) {
        qj = q_buffer_of(tc);
        if (qj < 0) {  // not fetched ahead
          qj = free_buffer();
          q_issue(qj, tc);
        }
        land(qj);
        d.src = pb;
        d.qj = qj;
      } else {
        d.src = from_resid ? cur : -1;
        d.nxt = cur ^ 1;
      }
    } else {
      d.src = kStaged ? pb : (from_resid ? cur : -1);
      d.bscale = from_resid ? 1.f : wscale;  // staged weights to one common scale
      d.us = us_s[u];
    }
    last = kind;
  };

  // Row statistics of an unwarped row (workers): the maximum, the weights
  // exp(l / T - m) (staged: stored over the logits) and their warp partial
  // sums, pushed for the leaders.  When the slice is at most G groups per
  // worker, its values stay in registers between the two.
  auto row_step = [&](const MssStep& d) {
    const Slice lrow = kStaged ? Slice{buf(d.src), lo} : Slice{llm_logits + (size_t)(off + d.u) * (size_t)V, 0};
    const bool one = n4 <= (int64_t)TW * G;
    float4 v[G];
    float m = -INFINITY;
    for (int64_t g0 = wid; g0 < n4; g0 += (int64_t)TW * G) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int64_t g = g0 + (int64_t)k * TW;
        if (g < n4) v[k] = lrow.ld4(lo + 4 * g, vec);
      }
#pragma unroll
      for (int k = 0; k < G; ++k)
        if (g0 + (int64_t)k * TW < n4)
          m = fmaxf(m, fmaxf(fmaxf(v[k].x * inv_t, v[k].y * inv_t), fmaxf(v[k].z * inv_t, v[k].w * inv_t)));
    }
    for (int64_t y = lo + 4 * n4 + wid; y < hi; y += TW) m = fmaxf(m, lrow[y] * inv_t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    named_bar_sync(1, TW);
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, red[w]);
    CompSum acc;
    auto weigh = [&](float4 x, int64_t g) {  // exp(l / T - m) of group g, summed (and staged: stored)
      float4 w;
      w.x = exp_diff(x.x * inv_t, m);
      w.y = exp_diff(x.y * inv_t, m);
      w.z = exp_diff(x.z * inv_t, m);
      w.w = exp_diff(x.w * inv_t, m);
      acc.add(w.x);
      acc.add(w.y);
      acc.add(w.z);
      acc.add(w.w);
      if (kStaged) *reinterpret_cast<float4*>(buf(d.src) + 4 * g) = w;
    };
    if (one) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int64_t g = wid + (int64_t)k * TW;
        if (g < n4) weigh(v[k], g);
      }
    } else {
      for (int64_t g0 = wid; g0 < n4; g0 += (int64_t)TW * G) {
#pragma unroll
        for (int k = 0; k < G; ++k) {
          const int64_t g = g0 + (int64_t)k * TW;
          if (g < n4) v[k] = lrow.ld4(lo + 4 * g, vec);
        }
#pragma unroll
        for (int k = 0; k < G; ++k) {
          const int64_t g = g0 + (int64_t)k * TW;
          if (g < n4) weigh(v[k], g);
        }
      }
    }
    for (int64_t y = lo + 4 * n4 + wid; y < hi; y += TW) {
      const float w = exp_diff(lrow[y] * inv_t, m);
      acc.add(w);
      if (kStaged) buf(d.src)[y - lo] = w;
    }
    if (kStaged) fence_proxy_async_smem();  // the slice may be overwritten by a later copy
    const F2 s = warp_sum_f2(comp_value(acc));
    push_warp(make_float4(m, s.hi, s.lo, 0.f), d.xs);
    if (warp == kWarps - 1) prefetch_children(d.u);
  };

  // Row statistics of a warped row (every thread): the maximum exchanged,
  // then the warped support found by the cluster; staged, the slice is left
  // holding the weights exp(l / T - M) of the kept tokens.
  auto row_step_warped = [&](const MssStep& d) {
    if constexpr (kWarpedOK) {
      const Slice lrow = kStaged ? Slice{buf(d.src), lo} : Slice{llm_logits + (size_t)(off + d.u) * (size_t)V, 0};
      float m = -INFINITY;
      for (int64_t y = lo + tid; y < hi; y += T) m = fmaxf(m, lrow[y] * inv_t);
      m = block_max<kWarps>(m, red);
      push_cta(make_float4(m, 0.f, 0.f, 0.f), d.xs);
      if (warp == kWarps - 1) prefetch_children(d.u);
      if (leader) {
        const float4* e = push_wait();
        float M = -INFINITY;
        for (int r = 0; r < ncl; ++r) M = fmaxf(M, e[r].x);
        if (lane == 0) mx_s = M;
      }
      __syncthreads();
      const float M = mx_s;
      const Support sp = warped_support<T>(lrow, V, lo, hi, inv_t, M, top_k, top_p, ncl, rank, xk,
                                                     pub, sel);
      m_u = M;
      inv_s = f2_inv(sp.S);
      tau = sp.tau;
      ycut = sp.ycut;
      if (kStaged) {  // weights relative to the row maximum M
        float* w = buf(d.src);
        for (int64_t y = lo + tid; y < hi; y += T) {
          const float l = w[y - lo];
          w[y - lo] = kept(l, y, tau, ycut) ? exp_diff(l * inv_t, M) : 0.f;
        }
        wscale = inv_s;
        fence_proxy_async_smem();  // the slice may be overwritten by a later copy
        __syncthreads();
      }
    }
  };

  // Residual pass (workers): r = max(0, p - q) over the slice, its warp
  // partial sums pushed for the leaders with r and p at the next child's
  // token, which its owner reads back from its own writes.
  auto pass_step = [&](const MssStep& d) {
    const bool direct = kStaged || d.src >= 0;  // p = source * pscale
    const Slice src = kStaged ? Slice{buf(d.src), lo}
                              : (d.src >= 0 ? Slice{resid_row(d.src), 0}
                                            : Slice{llm_logits + (size_t)(off + d.u) * (size_t)V, 0});
    const Slice q = kStaged ? Slice{buf(d.qj), lo} : Slice{ssm_probs + (size_t)(off + d.c) * (size_t)V, 0};
    float* const rout = kStaged ? buf(d.qj) : resid_row(d.nxt);  // staged: over q, element by element
    const int64_t rout_off = kStaged ? lo : 0;
    const float pscale = d.pscale;
    auto p_of = [&](float a, int64_t y) {
      return direct ? a * pscale : (kept(a, y, d.tau, d.ycut) ? exp_diff(a * inv_t, d.m_u) * d.inv_s : 0.f);
    };
    CompSum acc;
    for (int64_t g0 = wid; g0 < n4; g0 += (int64_t)TW * G) {
      float4 a[G], qq[G];
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int64_t g = g0 + (int64_t)k * TW;
        if (g < n4) {
          a[k] = src.ld4(lo + 4 * g, vec);
          qq[k] = q.ld4(lo + 4 * g, vec);
        }
      }
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int64_t g = g0 + (int64_t)k * TW;
        if (g < n4) {
          const int64_t y = lo + 4 * g;
          float4 r;
          r.x = fmaxf(p_of(a[k].x, y) - qq[k].x, 0.0f);
          r.y = fmaxf(p_of(a[k].y, y + 1) - qq[k].y, 0.0f);
          r.z = fmaxf(p_of(a[k].z, y + 2) - qq[k].z, 0.0f);
          r.w = fmaxf(p_of(a[k].w, y + 3) - qq[k].w, 0.0f);
          acc.add(r.x);
          acc.add(r.y);
          acc.add(r.z);
          acc.add(r.w);
          float* o = rout + (y - rout_off);
          if (vec) {
            *reinterpret_cast<float4*>(o) = r;
          } else {
            o[0] = r.x;
            o[1] = r.y;
            o[2] = r.z;
            o[3] = r.w;
          }
        }
      }
    }
    for (int64_t y = lo + 4 * n4 + wid; y < hi; y += TW) {
      const float r = fmaxf(p_of(src[y], y) - q[y], 0.0f);
      rout[y - rout_off] = r;
      acc.add(r);
    }
    if (kStaged) fence_proxy_async_smem();  // the residual may be overwritten by a later copy
    // The owner of xn in this CTA: group (xn - lo) / 4 goes to worker
    // group % TW, a tail element to worker (index past the groups) % TW.
    int own = -1;
    if (d.xn >= lo && d.xn < hi) {
      const int64_t rel = d.xn - lo;
      own = (int)(rel < 4 * n4 ? (rel >> 2) % TW : (rel - 4 * n4) % TW);
    }
    float r_x = 0.f, p_x = 0.f;
    if (own == wid) {  // its own writes, read back
      p_x = p_of(src[d.xn], d.xn);
      r_x = rout[d.xn - rout_off];
    }
    const F2 zs = warp_sum_f2(comp_value(acc));
    if (own >= 0 && (own >> 5) == warp - 1) {  // uniform over the warp for the push
      r_x = __shfl_sync(0xffffffffu, r_x, own & 31);
      p_x = __shfl_sync(0xffffffffu, p_x, own & 31);
    }
    push_warp(make_float4(zs.hi, zs.lo, r_x, p_x), d.xs);
  };

  if (rank == 0 && tid == 0) path[off] = 0;
  MssStep d;
  for (int st = 0;; ++st) {
    if (leader) {
      leader_decide(d);
      if (lane == 0) {
        dsc[st & 1] = d;
        if (d.kind == kStepPass || (d.kind == kStepRow && !warped))  // the workers' partials
          mbar_arrive_expect_tx(&xbar[d.xs], (uint32_t)(ncl * kWorkerWarps) * 16u);
      }
    }
    __syncthreads();  // the step is described and its input has landed
    d = dsc[st & 1];
    if (d.kind == kStepBonus) break;
    if (d.kind == kStepRow && warped) {
      row_step_warped(d);
      if (leader) leader_prep(d);
    } else if (leader) {
      leader_prep(d);
      leader_consume(d);
    } else if (d.kind == kStepRow) {
      row_step(d);
    } else {
      pass_step(d);
    }
  }

  if (rank == 0)
    for (int i = d.len + tid; i < n; i += T) path[off + i] = -1;
  if (leader) drain();  // no copy may be in flight when the CTA leaves
  // Bonus token: smallest y with cumsum(w)[y] > u_smp[u] * sum(w), w = the
  // unnormalised current distribution.  Each thread owns a contiguous run of
  // its CTA's slice; runs and slices are in vocabulary order.  The CTA totals
  // are exchanged; from their prefix sums every CTA finds the same rank whose
  // interval holds the target, and only that CTA searches its runs and
  // writes the token.
  const Slice wsrc = kStaged ? Slice{buf(d.src), lo}
                             : (d.src >= 0 ? Slice{resid_row(d.src), 0}
                                           : Slice{llm_logits + (size_t)(off + d.u) * (size_t)V, 0});
  const int64_t per_t = ((((hi - lo) + T - 1) / T) + 3) & ~int64_t(3);
  const int64_t tlo = min(hi, lo + (int64_t)tid * per_t), thi = min(hi, tlo + per_t);
  auto weight = [&](float a, int64_t y) {
    if (kStaged) return a * d.bscale;
    return d.src >= 0 ? a : (kept(a, y, d.tau, d.ycut) ? exp_diff(a * inv_t, d.m_u) : 0.f);
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
  // Exclusive prefix over the CTA's threads: a warp scan here; the leader
  // scans the warp totals and the CTA totals.
  const F2 incl = warp_scan_f2(mine);
  F2 wexcl = shfl_up_f2(incl, 1);
  if (lane == 0) wexcl = F2{0.f, 0.f};
  if (lane == 31) scan_s[warp] = incl;
  if (last_pos >= 0) atomicMax(&last_s, (int)last_pos);
  __syncthreads();
  if (leader) {
    F2 wt = lane < kWarps ? scan_s[lane] : F2{0.f, 0.f};
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const F2 t = shfl_up_f2(wt, o);
      if (lane >= o) wt = f2_add(t, wt);
    }
    const F2 cta_total = shfl_f2(wt, kWarps - 1);
    F2 wex = shfl_up_f2(wt, 1);
    if (lane == 0) wex = F2{0.f, 0.f};
    push_cta(make_float4(cta_total.hi, cta_total.lo, __int_as_float(last_s), tmo_s ? 1.f : 0.f), xp & 1);
    const float4* e = push_wait();
    // The CTA totals in rank order, scanned by lanes 0..ncl-1 (identical in
    // every CTA); the crossing rank is the first whose inclusive prefix
    // exceeds the target.
    F2 ct = lane < ncl ? F2{e[lane].x, e[lane].y} : F2{0.f, 0.f};
    int last_all = lane < ncl ? __float_as_int(e[lane].z) : -1;
    const bool timed_out = __ballot_sync(0xffffffffu, lane < ncl && e[lane].w != 0.f) != 0u;
#pragma unroll
    for (int o = 1; o < kMssMaxCluster; o <<= 1) {
      const F2 t = shfl_up_f2(ct, o);
      if (lane >= o) ct = f2_add(t, ct);
      last_all = max(last_all, __shfl_xor_sync(0xffffffffu, last_all, o));
    }
    const F2 total = shfl_f2(ct, ncl - 1);
    F2 base = shfl_f2(ct, rank > 0 ? rank - 1 : 0);
    if (rank == 0) base = F2{0.f, 0.f};
    const F2 target = f2_scale(total, d.us);
    const uint32_t over = __ballot_sync(0xffffffffu, lane < ncl && f2_lt(target, ct));
    const int rc = over ? __ffs(over) - 1 : -1;
    if (lane < kWarps) wpre_s[lane] = f2_add(base, wex);
    if (lane == 0) {
      target_s = target;
      pick_s = rc;
      if (rank == 0) {
        // No crossing (rounding left the target at the total): last positive entry.
        if (rc < 0) bonus[b] = last_all;
        accept_len[b] = d.len - 1;
        if (n_tried) n_tried[b] = tried;
        status[b] = timed_out ? TSV_ERR_TIMEOUT : TSV_OK;
      }
    }
  }
  __syncthreads();
  if (pick_s != rank) {  // uniform over the CTA
    if (beside && tid == 0) pdl_wait();
    return;
  }
  __syncthreads();  // every thread has read pick_s
  if (tid == 0) pick_s = INT32_MAX;
  __syncthreads();
  const F2 excl = f2_add(wpre_s[warp], wexcl);
  const F2 target = target_s;
  // The run holding the crossing is walked by its whole warp, 32 entries at
  // a time (an inclusive scan per chunk).
  const bool cross = mine.hi > 0.f && !f2_lt(target, excl) && f2_lt(target, f2_add(excl, mine));
  const uint32_t cb = __ballot_sync(0xffffffffu, cross);
  if (cb) {
    const int sl = __ffs(cb) - 1;
    const int64_t rlo = __shfl_sync(0xffffffffu, tlo, sl), rhi = __shfl_sync(0xffffffffu, thi, sl);
    F2 run = shfl_f2(excl, sl);
    int64_t pick = -1;
    for (int64_t base_y = rlo; base_y < rhi && pick < 0; base_y += 32) {
      const int64_t y = base_y + lane;
      const float w = y < rhi ? weight(wsrc[y], y) : 0.f;
      const F2 inc = warp_scan_f2(F2{w, 0.f});
      const uint32_t hit = __ballot_sync(0xffffffffu, w > 0.f && f2_lt(target, f2_add(run, inc)));
      if (hit) pick = base_y + __ffs(hit) - 1;
      run = f2_add(run, shfl_f2(inc, 31));
    }
    if (pick < 0) pick = __shfl_sync(0xffffffffu, last_pos, sl);  // rounding inside the run
    if (lane == 0) atomicMin(&pick_s, (int)pick);
  }
  __syncthreads();
  // No run holds it (rounding at the slice's end): the slice's last positive entry.
  if (tid == 0) bonus[b] = pick_s != INT32_MAX ? pick_s : last_s;
  if (beside && tid == 0) pdl_wait();
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
  for (int64_t g0 = tid; g0 < n4; g0 += kInFlight * kSelThreads) {
    float4 a[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u)
      if (g0 + u * kSelThreads < n4) a[u] = __ldg(r4 + g0 + u * kSelThreads);
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int64_t g = g0 + u * kSelThreads;
      if (g < n4) {
        const int y = (int)(lo + 4 * g);
        offer(a[u].x, y);
        offer(a[u].y, y + 1);
        offer(a[u].z, y + 2);
        offer(a[u].w, y + 3);
      }
    }
  }
  for (int64_t y = lo + 4 * n4 + tid; y < hi; y += kSelThreads) offer(__ldg(row + y), (int)y);
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
    for (int ww = 1; ww < kSelWarps; ++ww)
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
__global__ void __launch_bounds__(kSelThreads)
    tree_expand_kernel(const float* __restrict__ logits, int64_t V, int k, int ncl,
                       int32_t* __restrict__ tokens) {
  pdl_trigger();
  pdl_wait();  // the previous kernel's results are visible from here on
  __shared__ __align__(16) float pub[2][4];
  __shared__ SelSmem sel;
  __shared__ float red[128];
  __shared__ float lv[kSelThreads * kExpandSmallK];
  __shared__ int li[kSelThreads * kExpandSmallK];
  __shared__ float rv[kSelWarps];
  __shared__ int ri[kSelWarps];
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
  for (int64_t y = lo + threadIdx.x; y < hi; y += kSelThreads) m = fmaxf(m, __ldg(row + y));
  m = block_max<kSelWarps>(m, red);
  int xk = 0;
  if (ncl > 1) {  // the row maximum over the cluster
    if (threadIdx.x == 0) pub[0][0] = m;
    cluster_sync_all();
    for (int r = 0; r < ncl; ++r) m = fmaxf(m, ld_dsmem_f32(mapa_shared(smem_u32(&pub[0][0]), (uint32_t)r)));
    ++xk;
  }
  warped_support<kSelThreads>(Slice{row, 0}, V, lo, hi, 1.0f, m, k, 1.0f, ncl, rank, xk, pub, sel);
  if (rank == 0)
    for (int j = threadIdx.x; j < k; j += kSelThreads) out[j] = sel.srt_i[j];
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
  return launch_pdl(tree_expand_kernel, dim3((unsigned)(F * ncl)), dim3(kSelThreads), 0, st,
                    ncl > 1 ? (unsigned)ncl : 0u, logits, V, k, ncl, tokens);
}

cudaError_t launch_tree_merge(const int32_t* parent, const int32_t* tokens, const int32_t* tree_offsets,
                              const int32_t* request_trees, int32_t B, int32_t* out_parent,
                              int32_t* out_tokens, int32_t* out_source, int32_t* out_count,
                              int32_t* status, cudaStream_t st) {
  return launch_pdl(tree_merge_kernel, dim3(B), dim3(256), 0, st, 0u, parent, tokens, tree_offsets, request_trees,
                    out_parent, out_tokens, out_source, out_count, status);
}

// CTAs per request: slices of at least kMssMinSlice entries, at most 8 (one
// portable cluster), and no more than lets every request's cluster be
// resident at once (max_clusters[c]: clusters of c CTAs the device holds at
// once; the kernel runs one CTA per SM).
int mss_cluster_size(int64_t V, int32_t B, const int* max_clusters, int cap) {
  int64_t c = (V + kMssMinSlice - 1) / kMssMinSlice;
  c = c < 1 ? 1 : (c > cap ? cap : c);
  if (max_clusters != nullptr)
    while (c > 1 && max_clusters[c] < B) --c;
  return (int)c;
}

cudaError_t mss_set_attributes(int device, size_t* staged_limit, int* max_clusters) {
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  size_t limit = (size_t)optin;
  void (*kernels[3])(const float*, const float*, int64_t, const int32_t*, const int32_t*, const int32_t*,
                     const float*, const float*, float, int, float, int, int, int, float*, int32_t*, int32_t*,
                     int32_t*, int32_t*, int32_t*) = {mss_verify_kernel<true, kMssWarps, kMssRegs>,
                                                     mss_verify_kernel<true, kMssWarps, kMssRoomRegs>,
                                                     mss_verify_kernel<false, kMssWarps, kMssRegs>};
  for (auto* k : kernels) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, k);
    if (e != cudaSuccess) return e;
    const size_t l = (size_t)optin > fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l);
    if (e != cudaSuccess) return e;
    if (k == kernels[0]) limit = l;
  }
  *staged_limit = limit;
  // Resident clusters per size, for the staged kernel at its largest slice
  // set (one CTA per SM either way: its threads and registers fill an SM).
  max_clusters[0] = 0;
  for (int c = 1; c <= kMssMaxCluster; ++c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c);
    cfg.blockDim = dim3(kMssThreads);
    cfg.dynamicSmemBytes = limit;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)c;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, mss_verify_kernel<true, kMssWarps, kMssRegs>, &cfg);
    if (e != cudaSuccess) return e;
    max_clusters[c] = nc;
  }
  return cudaSuccess;
}

size_t mss_staged_bytes(int64_t V, int ncl) {
  const int64_t per = (((V + ncl - 1) / ncl) + 3) & ~int64_t(3);
  const int64_t per_al = (per + 31) & ~int64_t(31);
  return (size_t)(3 * per_al * 4);
}

cudaError_t launch_mss_verify(const float* llm_logits, const float* ssm_probs, int64_t V,
                              const int32_t* tokens, const int32_t* parent,
                              const int32_t* node_offsets, const float* u_acc, const float* u_smp,
                              float inv_t, int32_t top_k, float top_p, int32_t B, float* resid,
                              int32_t* path, int32_t* accept_len, int32_t* bonus, int32_t* n_tried,
                              int32_t* status, size_t staged_limit, const int* max_clusters,
                              int beside, int room, cudaStream_t st) {
  const int ncl = mss_cluster_size(V, B, max_clusters, beside == kMssBesideFull ? kMssBesideMaxCluster : kMssMaxCluster);
  const int vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(llm_logits) |
                                    reinterpret_cast<uintptr_t>(ssm_probs) |
                                    reinterpret_cast<uintptr_t>(resid)) & 15) == 0;
  // Slices staged in shared memory when three of them fit (bulk copies want
  // the 16-byte alignment `vec` stands for).
  const size_t dyn = mss_staged_bytes(V, ncl);
  const bool warped = top_k > 0 || top_p < 1.0f;
  // The full-size forms start beside the previous kernel only in the full
  // overlap mode; a warped call in the compact mode takes them and waits (the
  // warped support needs every warp).
  const int full = beside == kMssBesideFull ? 1 : 0;
  if (beside == kMssBesideCompact && !warped)  // two warps, slices from global memory: fits beside an attention CTA
    return launch_pdl(mss_verify_kernel<false, kMssCompactWarps, kMssRegs>, dim3((unsigned)(B * ncl)),
                      dim3(kMssCompactWarps * 32), 0, st, (unsigned)ncl, llm_logits, ssm_probs, V, tokens, parent,
                      node_offsets, u_acc, u_smp, inv_t, top_k, top_p, ncl, vec, 1, resid, path, accept_len, bonus,
                      n_tried, status);
  if (vec && dyn <= staged_limit)  // `room`: leave registers for a greedy CTA beside each CTA
    return launch_pdl(room ? mss_verify_kernel<true, kMssWarps, kMssRoomRegs>
                           : mss_verify_kernel<true, kMssWarps, kMssRegs>,
                      dim3((unsigned)(B * ncl)), dim3(kMssThreads), dyn, st,
                      (unsigned)ncl, llm_logits, ssm_probs, V, tokens, parent, node_offsets, u_acc, u_smp,
                      inv_t, top_k, top_p, ncl, vec, full, resid, path, accept_len, bonus, n_tried, status);
  return launch_pdl(mss_verify_kernel<false, kMssWarps, kMssRegs>, dim3((unsigned)(B * ncl)), dim3(kMssThreads), 0, st,
                    (unsigned)ncl, llm_logits, ssm_probs, V, tokens, parent, node_offsets, u_acc, u_smp, inv_t,
                    top_k, top_p, ncl, vec, full, resid, path, accept_len, bonus, n_tried, status);
}

}  // namespace tsv
