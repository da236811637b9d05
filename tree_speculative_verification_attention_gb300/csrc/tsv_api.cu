// tsv_api.cu — the C ABI declared in include/tsv.h: argument checks, work
// planning, tensor-map encoding and kernel launches.  No allocation happens
// here: every buffer, scratch included, belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "tsv_internal.h"

using namespace tsv;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct tsv_handle_s {
  int device;
  int num_sms;
  EncodeTiledFn encode;
  bool tc_attr_set[2];    // rows-on-lanes kernel (tile pairs), D = 64, 128
  bool tc1_attr_set[2];   // rows-on-lanes kernel (one tile), D = 64, 128
  bool keys_attr_set[2];  // keys-on-lanes kernel, D = 64, 128
  bool mss_attr_set;      // MSS kernel's shared-memory limit
  size_t mss_staged_limit;
  int mss_max_clusters[kMssClusterSizes];  // resident MSS clusters of each size
  uint32_t verify_overlap;  // tsv_set_verify_overlap: TSV_OVERLAP_* flags
};

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Checks the host copies of the batch layout.
tsv_status check_batch(int32_t B, const int32_t* prefix_len, const int32_t* node_offsets) {
  if (B < 1 || B > TSV_MAX_BATCH || !prefix_len || !node_offsets) return TSV_ERR_INVALID_ARG;
  if (node_offsets[0] != 0) return TSV_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int64_t n = (int64_t)node_offsets[b + 1] - node_offsets[b];
    if (n < 0 || prefix_len[b] < 0) return TSV_ERR_INVALID_ARG;
    if (n > TSV_MAX_NODES) return TSV_ERR_UNSUPPORTED;
    if ((int64_t)prefix_len[b] + n > INT32_MAX - 2 * kBN) return TSV_ERR_UNSUPPORTED;
  }
  return TSV_OK;
}

// Slot order of the requests: longest key range (prefix + nodes) first, ties
// by request index.
void order_slots(AttnPlan& p) {
  for (int s = 0; s < p.B; ++s) p.slot_req[s] = s;
  std::stable_sort(p.slot_req, p.slot_req + p.B, [&](int32_t a, int32_t b) {
    return (int64_t)p.prefix[a] + p.nodes[a] > (int64_t)p.prefix[b] + p.nodes[b];
  });
}

// CTAs of the rows-on-lanes kernel per (KV head, key chunk): two 128-row
// query tiles each when the plan pairs tiles, else one.
inline int64_t tc_units(const AttnPlan& p, int32_t mtiles) {
  return p.tc_tile_pairs ? (mtiles + 1) / 2 : mtiles;
}

// Splits every request's keys into chunks of one common length (a multiple of
// the 128-key block), over the chunk counts that cut the longest request into
// 1 .. 64 pieces.
void build_plan(AttnPlan& p, int num_sms, int32_t B, const int32_t* prefix_len,
                const int32_t* node_offsets, int32_t Hq, int32_t Hkv, int32_t D, float scale) {
  memset(&p, 0, sizeof(p));
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = D;
  p.scale_log2 = scale * 1.4426950408889634f;
  int64_t lmax = 1;
  for (int b = 0; b < B; ++b) {
    p.prefix[b] = prefix_len[b];
    p.node_off[b] = node_offsets[b];
    p.nodes[b] = node_offsets[b + 1] - node_offsets[b];
    p.mtiles[b] = (int32_t)cdiv((int64_t)p.nodes[b] * p.G, kBM);
    lmax = std::max<int64_t>(lmax, (int64_t)p.prefix[b] + p.nodes[b]);
    if (p.mtiles[b] >= 2) p.tc_tile_pairs = 1;  // some request has two tiles or more
  }
  // Tile pairs: the fewest chunks whose CTAs fill at least 3/4 of the SMs in
  // one wave (every extra chunk adds partial rows to write and to merge, and
  // the merge of a group runs in its last CTA).  Otherwise, or failing that,
  // the least estimated makespan waves * (chunk + per-CTA overhead).
  const int64_t overhead = 2 * kBN;
  int64_t best_cost = INT64_MAX, best_chunk = cdiv(lmax, kBN) * kBN, one_wave_chunk = 0;
  for (int pieces = 1; pieces <= 64; ++pieces) {
    const int64_t chunk = cdiv(cdiv(lmax, pieces), kBN) * kBN;
    int64_t units = 0;
    for (int b = 0; b < B; ++b)
      units += (int64_t)Hkv * tc_units(p, p.mtiles[b]) * cdiv((int64_t)p.prefix[b] + p.nodes[b], chunk);
    if (one_wave_chunk == 0 && units <= num_sms && 4 * units >= 3 * (int64_t)num_sms) one_wave_chunk = chunk;
    const int64_t waves = cdiv(units, num_sms);
    const int64_t cost = waves * (chunk + overhead);
    if (cost < best_cost || (cost == best_cost && chunk > best_chunk)) {
      best_cost = cost;
      best_chunk = chunk;
    }
    if (chunk == kBN) break;
  }
  if (p.tc_tile_pairs && one_wave_chunk > 0) best_chunk = one_wave_chunk;
  p.chunk_keys = (int32_t)best_chunk;
  order_slots(p);
  int64_t units = 0, rows = 0, ctrs = 0;
  for (int s = 0; s < B; ++s) {
    const int b = p.slot_req[s];
    const int64_t L = (int64_t)p.prefix[b] + p.nodes[b];
    p.n_chunks[b] = p.mtiles[b] > 0 ? (int32_t)cdiv(L, best_chunk) : 0;
    p.unit_start[s] = (int32_t)units;
    units += (int64_t)Hkv * tc_units(p, p.mtiles[b]) * p.n_chunks[b];
    p.ctr_base[b] = (int32_t)ctrs;
    ctrs += (int64_t)Hkv * p.mtiles[b];
    if (p.n_chunks[b] > 1) {
      p.part_row[b] = rows;
      rows += (int64_t)Hkv * p.n_chunks[b] * p.nodes[b] * p.G;
    } else {
      p.part_row[b] = -1;
    }
  }
  p.unit_start[B] = (int32_t)units;
  p.n_units = (int32_t)units;
  p.part_rows_total = rows;
  p.n_counters = (int32_t)ctrs;
  // Tile pairs with the same chunk count K (2 .. 8) in every request: the K
  // chunk CTAs of a group form a cluster and merge through distributed shared
  // memory instead of global partials and a last-CTA merge.
  int K = 0;
  bool uniform = true;
  for (int b = 0; b < B; ++b) {
    if (p.mtiles[b] == 0) continue;
    if (K == 0) K = p.n_chunks[b];
    else if (p.n_chunks[b] != K) uniform = false;
  }
  p.cluster = (p.tc_tile_pairs && uniform && K >= 2 && K <= 8) ? K : 0;
}

// Plan of the keys-on-lanes kernel (every request at most 64 query rows per
// KV head): each request's keys are cut into the same number K of chunks (K in
// 1 .. 8, the cluster size), chunk length ceil(L_b / K) rounded up to the
// 128-key block.  K minimises the estimated makespan max(waves x longest unit,
// total work / SMs), in keys plus a per-unit overhead of two blocks; ties go to
// the smaller cluster.
void build_plan_keys(AttnPlan& p, int num_sms, int32_t B, const int32_t* prefix_len,
                     const int32_t* node_offsets, int32_t Hq, int32_t Hkv, int32_t D, float scale) {
  memset(&p, 0, sizeof(p));
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.D = D;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.keys_kernel = 1;
  for (int b = 0; b < B; ++b) {
    p.prefix[b] = prefix_len[b];
    p.node_off[b] = node_offsets[b];
    p.nodes[b] = node_offsets[b + 1] - node_offsets[b];
    p.mtiles[b] = (int32_t)cdiv((int64_t)p.nodes[b] * p.G, kKeysTileRows);
  }
  const int64_t overhead = 2 * kKeysBlockKeys;
  int best_k = 1;
  double best_est = 1e300;
  for (int K = 1; K <= 8; ++K) {
    double total = 0, longest = 0;
    int64_t units = 0;
    for (int b = 0; b < B; ++b) {
      if (p.mtiles[b] == 0) continue;
      const int64_t L = (int64_t)p.prefix[b] + p.nodes[b];
      const int64_t clen = cdiv(cdiv(L, K), kKeysBlockKeys) * kKeysBlockKeys;
      const double unit_cost = (double)(clen + overhead);
      units += (int64_t)Hkv * p.mtiles[b] * K;
      total += unit_cost * (double)Hkv * p.mtiles[b] * K;
      longest = std::max(longest, unit_cost);
    }
    const double est = std::max((double)cdiv(units, num_sms) * longest, total / num_sms);
    if (est < best_est) {
      best_est = est;
      best_k = K;
    }
  }
  p.cluster = best_k;
  order_slots(p);
  int64_t units = 0;
  for (int s = 0; s < B; ++s) {
    const int b = p.slot_req[s];
    const int64_t L = (int64_t)p.prefix[b] + p.nodes[b];
    p.chunk_len[b] = (int32_t)(cdiv(cdiv(L, best_k), kKeysBlockKeys) * kKeysBlockKeys);
    p.n_chunks[b] = p.mtiles[b] > 0 ? best_k : 0;
    p.unit_start[s] = (int32_t)units;
    units += (int64_t)Hkv * p.mtiles[b] * p.n_chunks[b];
    p.part_row[b] = -1;
  }
  p.unit_start[B] = (int32_t)units;
  p.n_units = (int32_t)units;
  p.prefetch_l2 = units <= num_sms ? 1 : 0;
  p.persistent = (best_k == 1 && units > num_sms && units <= (int64_t)kKeysMaxUnitsPerCta * num_sms) ? 1 : 0;
  p.grid = p.persistent ? num_sms : (int32_t)units;
}

// The keys-on-lanes kernel serves batches whose requests all have at most 64
// query rows per KV head (GQA group dividing 64).
bool use_keys_kernel(int32_t B, const int32_t* node_offsets, int32_t Hq, int32_t Hkv) {
  const int32_t G = Hq / Hkv;
  if (kKeysTileRows % G != 0) return false;
  for (int b = 0; b < B; ++b)
    if ((int64_t)(node_offsets[b + 1] - node_offsets[b]) * G > kKeysTileRows) return false;
  return true;
}

// Workspace of one attention call.  Tensor-core path: merge counters first
// (they must be zero before the first call on a workspace; every completed
// call leaves them zero), then the split partials.  CUDA-core path without
// prepared bitsets: the bitsets.
struct AttnLayout {
  size_t ctr_off, anc_off, part_o_off, part_lse_off, total;
};

AttnLayout attention_layout(const AttnPlan& p, int64_t N, bool anc_given, bool use_tc) {
  AttnLayout a{};
  size_t off = 0;
  a.ctr_off = off;
  if (use_tc && p.part_rows_total > 0) off += round256((size_t)p.n_counters * sizeof(int32_t));
  a.anc_off = off;
  if (!anc_given && !use_tc) off += round256((size_t)N * TSV_ANC_WORDS * sizeof(uint32_t));
  a.part_o_off = off;
  if (use_tc) off += round256((size_t)p.part_rows_total * p.D * sizeof(float));
  a.part_lse_off = off;
  if (use_tc) off += round256((size_t)p.part_rows_total * sizeof(float));
  a.total = off;
  return a;
}

tsv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TSV_OK : TSV_ERR_CUDA; }

tsv_status encode_kv_map(tsv_handle h, CUtensorMap* map, const void* base, int64_t sb, int64_t sl,
                         int64_t sh, int32_t B, int64_t L, int32_t Hkv, int32_t D, int box_rows) {
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)L, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)sh * 2, (cuuint64_t)sl * 2, (cuuint64_t)sb * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TSV_OK : TSV_ERR_INVALID_ARG;
}

// Q [N, Hq, D] as a 3-D map (D, Hq, N); a box of (64, G, tile_rows/G) is one
// tile whose row r is (node r / G, head-in-group r % G).
tsv_status encode_q_map(tsv_handle h, CUtensorMap* map, const void* q, int64_t N, int32_t Hq,
                        int32_t G, int32_t D, int tile_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)N};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(tile_rows / G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TSV_OK : TSV_ERR_INVALID_ARG;
}

bool attention_uses_tc(tsv_dtype dtype, uint32_t flags) {
  return dtype == TSV_BF16 && !(flags & TSV_ATTN_SIMT);
}

}  // namespace

extern "C" {

const char* tsv_status_string(int status) {
  switch (status) {
    case TSV_OK: return "ok";
    case TSV_ERR_INVALID_ARG: return "invalid argument";
    case TSV_ERR_BAD_TREE: return "bad tree (parent array breaks the topological convention)";
    case TSV_ERR_UNSUPPORTED: return "unsupported shape";
    case TSV_ERR_CUDA: return "CUDA error";
    case TSV_ERR_TIMEOUT: return "device-side wait timed out";
    case TSV_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int tsv_version(void) { return 100; }

tsv_status tsv_create(tsv_handle* out, int device) {
  if (!out) return TSV_ERR_INVALID_ARG;
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
    cudaGetLastError();
    return TSV_ERR_CUDA;
  }
  if (cudaSetDevice(device) != cudaSuccess) return TSV_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return TSV_ERR_CUDA;
  if (major != 10 || minor != 3) return TSV_ERR_UNSUPPORTED;  // kernels are built for sm_103a
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return TSV_ERR_CUDA;
  tsv_handle h = new (std::nothrow) tsv_handle_s;
  if (!h) return TSV_ERR_CUDA;
  h->device = device;
  h->num_sms = sms;
  h->encode = reinterpret_cast<EncodeTiledFn>(fn);
  h->tc_attr_set[0] = h->tc_attr_set[1] = false;
  h->tc1_attr_set[0] = h->tc1_attr_set[1] = false;
  h->keys_attr_set[0] = h->keys_attr_set[1] = false;
  h->mss_attr_set = false;
  h->mss_staged_limit = 0;
  h->verify_overlap = 0u;
  *out = h;
  return TSV_OK;
}

tsv_status tsv_set_verify_overlap(tsv_handle h, uint32_t kinds) {
  if (!h || (kinds & ~(TSV_OVERLAP_GREEDY | TSV_OVERLAP_STOCHASTIC | TSV_OVERLAP_STOCHASTIC_FULL)) != 0u)
    return TSV_ERR_INVALID_ARG;
  h->verify_overlap = kinds;
  return TSV_OK;
}

tsv_status tsv_destroy(tsv_handle h) {
  if (!h) return TSV_ERR_INVALID_ARG;
  delete h;
  return TSV_OK;
}

tsv_status tsv_tree_prepare(tsv_handle h, const int32_t* parent_d, const int32_t* node_offsets_d,
                            int32_t B, uint32_t* anc_d, int32_t* depth_d, int32_t* status_d,
                            void* stream) {
  if (!h || !parent_d || !node_offsets_d || !anc_d || !status_d) return TSV_ERR_INVALID_ARG;
  if (B < 1 || B > TSV_MAX_BATCH) return TSV_ERR_INVALID_ARG;
  return cuda_status(launch_tree_prepare(parent_d, node_offsets_d, B, anc_d, depth_d, status_d,
                                         static_cast<cudaStream_t>(stream)));
}

tsv_status tsv_tree_attention_workspace_size(tsv_handle h, tsv_dtype dtype, int32_t B,
                                             const int32_t* prefix_len_host,
                                             const int32_t* node_offsets_host, int32_t Hq,
                                             int32_t Hkv, int32_t D, int anc_given,
                                             uint32_t flags, size_t* bytes) {
  if (!h || !bytes) return TSV_ERR_INVALID_ARG;
  if (dtype != TSV_F32 && dtype != TSV_BF16) return TSV_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return TSV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TSV_ERR_UNSUPPORTED;
  tsv_status st = check_batch(B, prefix_len_host, node_offsets_host);
  if (st != TSV_OK) return st;
  AttnPlan plan;
  const bool use_tc = attention_uses_tc(dtype, flags);
  if (use_tc && use_keys_kernel(B, node_offsets_host, Hq, Hkv))
    build_plan_keys(plan, h->num_sms, B, prefix_len_host, node_offsets_host, Hq, Hkv, D, 1.f);
  else
    build_plan(plan, h->num_sms, B, prefix_len_host, node_offsets_host, Hq, Hkv, D, 1.f);
  *bytes = attention_layout(plan, node_offsets_host[B], anc_given != 0, use_tc).total;
  return TSV_OK;
}

tsv_status tsv_tree_attention(tsv_handle h, tsv_dtype dtype, const void* q_d, const void* k_cache_d,
                              const void* v_cache_d, int64_t kv_stride_b, int64_t kv_stride_l,
                              int64_t kv_stride_h, void* out_d, const int32_t* prefix_len_host,
                              const int32_t* node_offsets_host, const int32_t* prefix_len_d,
                              const int32_t* node_offsets_d, const int32_t* parent_d,
                              const uint32_t* anc_d, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                              float scale, void* workspace_d, size_t workspace_bytes,
                              int32_t* status_d, uint32_t flags, void* stream) {
  if (!h || !q_d || !k_cache_d || !v_cache_d || !out_d || !prefix_len_d || !node_offsets_d ||
      !status_d)
    return TSV_ERR_INVALID_ARG;
  if (dtype != TSV_F32 && dtype != TSV_BF16) return TSV_ERR_INVALID_ARG;
  if (flags & ~TSV_ATTN_SIMT) return TSV_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return TSV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TSV_ERR_UNSUPPORTED;
  if (kv_stride_b < 0 || kv_stride_l < 0 || kv_stride_h < 0) return TSV_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || isinf(scale)) return TSV_ERR_INVALID_ARG;
  if (!anc_d && !parent_d) return TSV_ERR_INVALID_ARG;
  tsv_status st = check_batch(B, prefix_len_host, node_offsets_host);
  if (st != TSV_OK) return st;
  const int64_t N = node_offsets_host[B];
  if (N * (int64_t)Hq > INT32_MAX) return TSV_ERR_UNSUPPORTED;
  const bool use_tc = attention_uses_tc(dtype, flags);
  const bool use_keys = use_tc && use_keys_kernel(B, node_offsets_host, Hq, Hkv);
  if (use_tc) {
    if (!aligned16(q_d) || !aligned16(out_d) || !aligned16(k_cache_d) || !aligned16(v_cache_d) ||
        (anc_d && !aligned16(anc_d)))
      return TSV_ERR_INVALID_ARG;
    if (kv_stride_b % 8 || kv_stride_l % 8 || kv_stride_h % 8) return TSV_ERR_INVALID_ARG;
    if (!use_keys && kBM % (Hq / Hkv) != 0) return TSV_ERR_UNSUPPORTED;  // a tile holds whole GQA groups
  }
  if (scale == 0.f) scale = 1.f / sqrtf((float)D);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  AttnPlan plan;
  if (use_keys)
    build_plan_keys(plan, h->num_sms, B, prefix_len_host, node_offsets_host, Hq, Hkv, D, scale);
  else
    build_plan(plan, h->num_sms, B, prefix_len_host, node_offsets_host, Hq, Hkv, D, scale);
  const AttnLayout lay = attention_layout(plan, N, anc_d != nullptr, use_tc);
  if (lay.total > 0 && (!workspace_d || workspace_bytes < lay.total)) return TSV_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace_d);
  if (N == 0) return TSV_OK;

  if (!use_tc) {
    const uint32_t* anc = anc_d;
    if (!anc) {
      uint32_t* a = reinterpret_cast<uint32_t*>(ws + lay.anc_off);
      st = cuda_status(launch_tree_prepare(parent_d, node_offsets_d, B, a, nullptr, status_d, cs));
      if (st != TSV_OK) return st;
      anc = a;
    }
    return cuda_status(launch_attention_simt(dtype == TSV_BF16, q_d, k_cache_d, v_cache_d,
                                             kv_stride_b, kv_stride_l, kv_stride_h, out_d,
                                             prefix_len_d, node_offsets_d, anc, B, (int32_t)N, Hq,
                                             Hkv, D, scale, cs));
  }
  const int di = D == 64 ? 0 : 1;
  int64_t lmax = 1;
  for (int b = 0; b < B; ++b) lmax = std::max<int64_t>(lmax, (int64_t)plan.prefix[b] + plan.nodes[b]);
  CUtensorMap tmq, tmk, tmv;
  const int tile_rows = use_keys ? kKeysTileRows : kBM;
  const int box_rows = use_keys ? kKeysBlockKeys : kBN;
  st = encode_q_map(h, &tmq, q_d, N, Hq, Hq / Hkv, D, tile_rows);
  if (st != TSV_OK) return st;
  st = encode_kv_map(h, &tmk, k_cache_d, kv_stride_b, kv_stride_l, kv_stride_h, B, lmax, Hkv, D, box_rows);
  if (st != TSV_OK) return st;
  st = encode_kv_map(h, &tmv, v_cache_d, kv_stride_b, kv_stride_l, kv_stride_h, B, lmax, Hkv, D, box_rows);
  if (st != TSV_OK) return st;
  if (use_keys) {
    if (!h->keys_attr_set[di]) {
      if (attention_keys_set_attributes(D) != cudaSuccess) return TSV_ERR_CUDA;
      h->keys_attr_set[di] = true;
    }
    return cuda_status(launch_attention_keys(tmq, tmk, tmv, plan, parent_d, anc_d, out_d, status_d, cs));
  }
  int32_t* counters = reinterpret_cast<int32_t*>(ws + lay.ctr_off);
  float* part_o = reinterpret_cast<float*>(ws + lay.part_o_off);
  float* part_lse = reinterpret_cast<float*>(ws + lay.part_lse_off);
  if (!plan.tc_tile_pairs) {
    if (!h->tc1_attr_set[di]) {
      if (attention_tc1_set_attributes(D) != cudaSuccess) return TSV_ERR_CUDA;
      h->tc1_attr_set[di] = true;
    }
    return cuda_status(launch_attention_tc1(tmq, tmk, tmv, plan, parent_d, anc_d, out_d, part_o,
                                            part_lse, counters, status_d, cs));
  }
  if (!h->tc_attr_set[di]) {
    if (attention_tc_set_attributes(D) != cudaSuccess) return TSV_ERR_CUDA;
    h->tc_attr_set[di] = true;
  }
  return cuda_status(launch_attention_tc(tmq, tmk, tmv, plan, parent_d, anc_d, out_d, part_o,
                                         part_lse, counters, status_d, cs));
}

tsv_status tsv_tree_verify_greedy_workspace_size(tsv_handle h, int32_t B, int32_t N, int64_t V,
                                                 size_t* bytes) {
  if (!h || !bytes || B < 1 || B > TSV_MAX_BATCH || N < 0 || V < 1 || V > INT32_MAX)
    return TSV_ERR_INVALID_ARG;
  *bytes = greedy_workspace_bytes(B, N);
  return TSV_OK;
}

tsv_status tsv_tree_verify_greedy(tsv_handle h, const float* logits_d, int64_t V,
                                  const int32_t* tree_tokens_d, const int32_t* parent_d,
                                  const int32_t* node_offsets_d, int32_t B, int32_t N,
                                  int32_t* path_d, int32_t* accept_len_d, int32_t* bonus_d,
                                  void* workspace_d, size_t workspace_bytes, int32_t* status_d,
                                  void* stream) {
  if (!h || !tree_tokens_d || !parent_d || !node_offsets_d || !accept_len_d || !bonus_d ||
      !status_d)
    return TSV_ERR_INVALID_ARG;
  if (B < 1 || B > TSV_MAX_BATCH || N < 0 || V < 1 || V > INT32_MAX) return TSV_ERR_INVALID_ARG;
  if (N > 0 && (!logits_d || !path_d)) return TSV_ERR_INVALID_ARG;
  const int splits = greedy_splits(V, N, h->num_sms);
  if (!workspace_d || workspace_bytes < greedy_workspace_bytes(B, N)) return TSV_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace_d);
  int32_t* counters = reinterpret_cast<int32_t*>(ws);
  unsigned long long* rowbest = reinterpret_cast<unsigned long long*>(ws + greedy_counter_bytes(B));
  if (N == 0)
    return cuda_status(launch_greedy_walk(rowbest, tree_tokens_d, parent_d, node_offsets_d, B, path_d,
                                          accept_len_d, bonus_d, status_d, cs));
  return cuda_status(launch_greedy_verify(logits_d, V, N, splits, tree_tokens_d, parent_d,
                                          node_offsets_d, B, rowbest, counters, path_d, accept_len_d,
                                          bonus_d, status_d, (h->verify_overlap & TSV_OVERLAP_GREEDY) ? 1 : 0,
                                          cs));
}

tsv_status tsv_tree_verify_stochastic_workspace_size(tsv_handle h, int32_t B, int32_t N, int64_t V,
                                                     size_t* bytes) {
  if (!h || !bytes || B < 1 || B > TSV_MAX_BATCH || N < 0 || V < 1 || V > INT32_MAX)
    return TSV_ERR_INVALID_ARG;
  (void)N;
  *bytes = round256((size_t)B * 2 * (size_t)V * 4);  // two residual rows per request
  return TSV_OK;
}

static tsv_status verify_stochastic(tsv_handle h, const float* llm_logits_d, const float* ssm_probs_d,
                                    int64_t V, const int32_t* tree_tokens_d, const int32_t* parent_d,
                                    const int32_t* node_offsets_d, const float* u_accept_d,
                                    const float* u_sample_d, float temperature, int32_t top_k,
                                    float top_p, int32_t B, int32_t N, int32_t* path_d,
                                    int32_t* accept_len_d, int32_t* bonus_d, int32_t* n_tried_d,
                                    void* workspace_d, size_t workspace_bytes, int32_t* status_d,
                                    void* stream) {
  if (!h || !tree_tokens_d || !parent_d || !node_offsets_d || !accept_len_d || !bonus_d ||
      !status_d)
    return TSV_ERR_INVALID_ARG;
  if (B < 1 || B > TSV_MAX_BATCH || N < 0 || V < 1 || V > INT32_MAX) return TSV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || isinf(temperature)) return TSV_ERR_INVALID_ARG;
  if (top_k < 0 || !(top_p > 0.f) || top_p > 1.f) return TSV_ERR_INVALID_ARG;
  if (top_k > kMssMaxTopK || (top_p < 1.f && top_k == 0)) return TSV_ERR_UNSUPPORTED;
  if (N > 0 && (!llm_logits_d || !ssm_probs_d || !u_accept_d || !u_sample_d || !path_d))
    return TSV_ERR_INVALID_ARG;
  const size_t need = round256((size_t)B * 2 * (size_t)V * 4);
  if (!workspace_d || workspace_bytes < need) return TSV_ERR_INVALID_ARG;
  float* resid = static_cast<float*>(workspace_d);
  if (!h->mss_attr_set) {
    if (mss_set_attributes(h->device, &h->mss_staged_limit, h->mss_max_clusters) != cudaSuccess)
      return TSV_ERR_CUDA;
    h->mss_attr_set = true;
  }
  return cuda_status(launch_mss_verify(llm_logits_d, ssm_probs_d, V, tree_tokens_d, parent_d,
                                       node_offsets_d, u_accept_d, u_sample_d, 1.0f / temperature,
                                       top_k, top_p, B, resid, path_d, accept_len_d, bonus_d,
                                       n_tried_d, status_d, h->mss_staged_limit, h->mss_max_clusters,
                                       (h->verify_overlap & TSV_OVERLAP_STOCHASTIC_FULL) ? kMssBesideFull
                                       : (h->verify_overlap & TSV_OVERLAP_STOCHASTIC)    ? kMssBesideCompact
                                                                                         : 0,
                                       (h->verify_overlap & TSV_OVERLAP_GREEDY) ? 1 : 0,
                                       static_cast<cudaStream_t>(stream)));
}

tsv_status tsv_tree_verify_stochastic(tsv_handle h, const float* llm_logits_d,
                                      const float* ssm_probs_d, int64_t V,
                                      const int32_t* tree_tokens_d, const int32_t* parent_d,
                                      const int32_t* node_offsets_d, const float* u_accept_d,
                                      const float* u_sample_d, float temperature, int32_t B,
                                      int32_t N, int32_t* path_d, int32_t* accept_len_d,
                                      int32_t* bonus_d, int32_t* n_tried_d, void* workspace_d,
                                      size_t workspace_bytes, int32_t* status_d, void* stream) {
  return verify_stochastic(h, llm_logits_d, ssm_probs_d, V, tree_tokens_d, parent_d, node_offsets_d,
                           u_accept_d, u_sample_d, temperature, 0, 1.0f, B, N, path_d,
                           accept_len_d, bonus_d, n_tried_d, workspace_d, workspace_bytes,
                           status_d, stream);
}

tsv_status tsv_tree_verify_stochastic_warped(
    tsv_handle h, const float* llm_logits_d, const float* ssm_probs_d, int64_t V,
    const int32_t* tree_tokens_d, const int32_t* parent_d, const int32_t* node_offsets_d,
    const float* u_accept_d, const float* u_sample_d, float temperature, int32_t top_k, float top_p,
    int32_t B, int32_t N, int32_t* path_d, int32_t* accept_len_d, int32_t* bonus_d,
    int32_t* n_tried_d, void* workspace_d, size_t workspace_bytes, int32_t* status_d,
    void* stream) {
  return verify_stochastic(h, llm_logits_d, ssm_probs_d, V, tree_tokens_d, parent_d, node_offsets_d,
                           u_accept_d, u_sample_d, temperature, top_k, top_p, B, N, path_d,
                           accept_len_d, bonus_d, n_tried_d, workspace_d, workspace_bytes,
                           status_d, stream);
}

tsv_status tsv_kv_commit(tsv_handle h, tsv_dtype dtype, void* k_cache_d, void* v_cache_d,
                         int64_t kv_stride_b, int64_t kv_stride_l, int64_t kv_stride_h, int32_t B,
                         int32_t Hkv, int32_t D, const int32_t* prefix_len_d,
                         const int32_t* node_offsets_d, const int32_t* path_d,
                         const int32_t* accept_len_d, int32_t* new_len_d, int32_t* status_d,
                         void* stream) {
  if (!h || !k_cache_d || !v_cache_d || !prefix_len_d || !node_offsets_d || !path_d ||
      !accept_len_d || !status_d)
    return TSV_ERR_INVALID_ARG;
  if (dtype != TSV_F32 && dtype != TSV_BF16) return TSV_ERR_INVALID_ARG;
  if (B < 1 || B > TSV_MAX_BATCH || Hkv < 1 || D < 1) return TSV_ERR_INVALID_ARG;
  const int64_t esz = dtype == TSV_BF16 ? 2 : 4;
  // Whole 16-byte chunks: pointers, strides and the row of one head aligned.
  if ((reinterpret_cast<uintptr_t>(k_cache_d) | reinterpret_cast<uintptr_t>(v_cache_d)) & 15)
    return TSV_ERR_INVALID_ARG;
  if (((int64_t)D * esz) % 16 || (kv_stride_b * esz) % 16 || (kv_stride_l * esz) % 16 ||
      (kv_stride_h * esz) % 16 || kv_stride_b < 0 || kv_stride_l < 0 || kv_stride_h < 0)
    return TSV_ERR_INVALID_ARG;
  if ((int64_t)Hkv * D * esz / 16 > INT32_MAX) return TSV_ERR_UNSUPPORTED;
  return cuda_status(launch_kv_commit(static_cast<uint8_t*>(k_cache_d), static_cast<uint8_t*>(v_cache_d),
                                      kv_stride_b * esz, kv_stride_l * esz, kv_stride_h * esz, B, Hkv,
                                      (int32_t)(D * esz / 16), prefix_len_d, node_offsets_d, path_d,
                                      accept_len_d, new_len_d, status_d,
                                      static_cast<cudaStream_t>(stream)));
}

tsv_status tsv_tree_expand(tsv_handle h, const float* ssm_logits_d, int64_t V, int32_t F, int32_t k,
                           int32_t* tokens_d, void* stream) {
  if (!h || F < 0 || V < 1 || V > INT32_MAX || k < 1 || (int64_t)k > V) return TSV_ERR_INVALID_ARG;
  if (k > kMssMaxTopK) return TSV_ERR_UNSUPPORTED;
  if (F > 0 && (!ssm_logits_d || !tokens_d)) return TSV_ERR_INVALID_ARG;
  return cuda_status(
      launch_tree_expand(ssm_logits_d, V, F, k, tokens_d, h->num_sms, static_cast<cudaStream_t>(stream)));
}

tsv_status tsv_tree_merge(tsv_handle h, const int32_t* parent_d, const int32_t* tokens_d,
                          const int32_t* tree_offsets_d, const int32_t* request_trees_d, int32_t B,
                          int32_t* out_parent_d, int32_t* out_tokens_d, int32_t* out_source_d,
                          int32_t* out_count_d, int32_t* status_d, void* stream) {
  if (!h || !parent_d || !tokens_d || !tree_offsets_d || !request_trees_d || !out_parent_d ||
      !out_tokens_d || !out_count_d || !status_d)
    return TSV_ERR_INVALID_ARG;
  if (B < 1 || B > TSV_MAX_BATCH) return TSV_ERR_INVALID_ARG;
  return cuda_status(launch_tree_merge(parent_d, tokens_d, tree_offsets_d, request_trees_d, B, out_parent_d,
                                       out_tokens_d, out_source_d, out_count_d, status_d,
                                       static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
