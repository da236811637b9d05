// tsv_attention_tc.cu — tree attention on the 5th-generation tensor cores.
//
// What it computes (SpecInfer §4 Token Tree Verifier, "Tree Attention" and
// "Tree-Based Parallel Decoding"): every tree node attends to the shared
// prefix of the KV cache plus the tree keys of its own root-to-node path, all
// tree nodes of a request in one kernel through a topology-aware mask.  The
// cache / in-tree split and merge of Staged Speculative Decoding (§3,
// Implementation) becomes a split of each request's keys into chunks whose
// partial results are merged by log-sum-exp.
//
// One CTA = one unit (request b, KV head g, key chunk c, M-tile mt).  Its 128
// query rows are (node, head-in-group) pairs: all query heads that share KV
// head g sit in the same tile, so each streamed K/V row serves every tree node
// and every grouped head at once.  Warp roles (192 threads):
//   warp 4        TMA producer: K and V blocks of 64 rows x D, 128-byte
//                 swizzled, into a ring of kStages shared-memory stages.
//   warp 5        tcgen05 issuer: S = Q K^T into TMEM (double-buffered), then
//                 O += P V into a TMEM accumulator; also owns TMEM allocation.
//   warps 0-3     one thread per query row (= TMEM lane): reads S, applies the
//                 ancestor-bitset mask on the tree part of the keys, online
//                 softmax in base 2 with a lazily moved reference maximum,
//                 writes P (bf16) to shared memory, rescales O in TMEM when
//                 the reference moves, and finally normalises O and stores the
//                 output (one chunk) or a partial result + log2-sum-exp.
// attn_combine_kernel merges the partials of requests cut into several chunks.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_device.cuh"
#include "tsv_internal.h"

namespace tsv {

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;               // 128-byte column groups per row
  static constexpr int kStages = (D == 128) ? 4 : 8;   // K/V ring depth
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kTileBytes = kBN * D * 2;       // one K (or V) block
  static constexpr int kPBytes = kBM * kBN * 2;
  static constexpr int kAncWords = TSV_ANC_WORDS + 2;  // two zero words past the end
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffAnc = kOffP + kPBytes;
  static constexpr int kOffBar = kOffAnc + kBM * kAncWords * 4;
  static constexpr int kNumBars = 2 * kStages + 5;  // kv_full, kv_empty, s_full[2], p_full, pv_done, mma_done
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 256;               // S0 | S1 | O
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(2 * kBN + D <= (int)kTmemCols, "TMEM columns");
};

constexpr int kTcThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8 between rescales

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

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ AttnPlan plan, const __nv_bfloat16* __restrict__ q,
                        const uint32_t* __restrict__ anc, __nv_bfloat16* __restrict__ out,
                        float* __restrict__ part_o, float* __restrict__ part_lse,
                        int32_t* __restrict__ status) {
  using C = TcCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sP = smem + C::kOffP;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + C::kOffAnc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + S;
  uint64_t* s_full = bars + 2 * S;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* mma_done = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  volatile int* abort_v = abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- the unit
  const int unit = blockIdx.x;
  int lo = 0, hi = plan.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (plan.unit_start[mid] <= unit) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int local = unit - plan.unit_start[b];
  const int mtiles = plan.mtiles[b], nch = plan.n_chunks[b];
  const int mt = local % mtiles;
  const int cg = local / mtiles;
  const int c = cg % nch;
  const int g = cg / nch;
  const int G = plan.G;
  const int P = plan.prefix[b], n = plan.nodes[b], off = plan.node_off[b];
  const int R = n * G;
  const int row0 = mt * kBM;
  const int rows_valid = min(kBM, R - row0);
  const int k_begin = c * plan.chunk_keys;
  const int k_end = min(P + n, k_begin + plan.chunk_keys);
  const int nblk = (k_end - k_begin + kBN - 1) / kBN;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 128);  // every softmax thread arrives
    mbar_init(pv_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }

  // Q tile (rows past the request are zero) in the 128-byte-swizzled K-major
  // layout the MMA reads: row r, 16-byte chunk c8 of column group hf at
  // hf*kBM*128 + r*128 + (c8 ^ (r & 7))*16.
  for (int idx = tid; idx < kBM * (D / 8); idx += kTcThreads) {
    const int r = idx / (D / 8), ch = idx % (D / 8);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows_valid) {
      const int gr = row0 + r;
      const int node = gr / G, hr = gr - node * G;
      const uint4* src = reinterpret_cast<const uint4*>(
          q + ((size_t)(off + node) * plan.Hq + (size_t)g * G + hr) * D);
      val = __ldg(src + ch);
    }
    const int hf = ch >> 3, c8 = ch & 7;
    *reinterpret_cast<uint4*>(sQ + hf * (kBM * 128) + r * 128 + ((c8 ^ (r & 7)) << 4)) = val;
  }
  for (int idx = tid; idx < kBM * C::kAncWords; idx += kTcThreads) {
    const int r = idx / C::kAncWords, w = idx % C::kAncWords;
    uint32_t val = 0u;
    if (r < rows_valid && w < TSV_ANC_WORDS) {
      const int node = (row0 + r) / G;
      val = anc[(size_t)(off + node) * TSV_ANC_WORDS + w];
    }
    sAnc[idx] = val;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = mtiles > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % S;
        if (j >= S && !mbar_wait(&kv_empty[st], ((j / S) - 1) & 1, abort_v)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTileBytes);
        const int key0 = k_begin + j * kBN;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_4d(sK + st * C::kTileBytes + hf * (kBN * 128), &tmap_k, &kv_full[st], hf * 64, g,
                      key0, b, pol);
          tma_load_4d(sV + st * C::kTileBytes + hf * (kBN * 128), &tmap_v, &kv_full[st], hf * 64, g,
                      key0, b, pol);
        }
        ++issued;
      }
      if (*abort_v) {  // let copies still in flight land before the CTA exits
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait(&kv_full[j % S], (j / S) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, 1);
      const uint32_t tS0 = tmem, tO = tmem + 2 * kBN;
      const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV), pa = smem_u32(sP);
      auto issue_s = [&](int j) {
        const int st = j % S;
        const uint32_t dst = tS0 + (uint32_t)((j & 1) * kBN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          const uint32_t bo = st * C::kTileBytes + (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
          umma_bf16(dst, sdesc_sw128(qa + ao, 16, 1024), sdesc_sw128(ka + bo, 16, 1024), idS,
                    kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int j) {
        const int st = j % S;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t bo = st * C::kTileBytes + kk * 16 * 128;
          umma_bf16(tO, sdesc_sw128(pa + kk * 32, 16, 1024),
                    sdesc_sw128(va + bo, kBN * 128, 1024), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = nblk > 0 && mbar_wait(&kv_full[0], 0, abort_v);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit(&s_full[0]);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + 1 < nblk) {
          if (!mbar_wait(&kv_full[(j + 1) % S], ((j + 1) / S) & 1, abort_v)) break;
          tc_fence_after();
          issue_s(j + 1);
          umma_commit(&s_full[(j + 1) & 1]);
        }
        if (!mbar_wait(p_full, j & 1, abort_v)) break;
        tc_fence_after();
        issue_pv(j);
        umma_commit(pv_done);
        umma_commit(&kv_empty[j % S]);
      }
      umma_commit(mma_done);  // every MMA of this CTA has finished before TMEM is freed
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;
    const bool valid = r < rows_valid;
    const uint32_t* arow = sAnc + r * C::kAncWords;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = plan.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_v));
      if (!ok) break;
      tc_fence_after();
      float s[kBN];
      {
        float t0[32], t1[32];
        tmem_ld32(tmem + lane_base + (uint32_t)((j & 1) * kBN), t0);
        tmem_ld32(tmem + lane_base + (uint32_t)((j & 1) * kBN + 32), t1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          s[e] = t0[e];
          s[32 + e] = t1[e];
        }
      }
      const int key0 = k_begin + j * kBN;
      const uint64_t vis = !valid ? 0ull : (key0 + kBN <= P ? ~0ull : block_visibility(arow, key0 - P));
      float bmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < kBN; ++e) {
        s[e] = ((vis >> e) & 1ull) ? s[e] * sl2 : -INFINITY;
        bmax = fmaxf(bmax, s[e]);
      }
      // Move the reference maximum only when the block's max exceeds it by
      // more than the threshold (always on the first visible block).
      float alpha = 1.f;
      bool resc = false;
      if (bmax > m_ref + kRescaleThreshold) {
        alpha = fast_exp2(m_ref - bmax);  // 0 when m_ref = -inf
        m_ref = bmax;
        resc = true;
      }
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;
      uint32_t pk[kBN / 2];
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < kBN; e += 2) {
        const float p0 = fast_exp2(s[e] - mref), p1 = fast_exp2(s[e + 1] - mref);
        psum += p0 + p1;
        pk[e >> 1] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + psum;
      if (j > 0) {  // PV of the previous block done: P buffer free, O stable
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort_v));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
          }
        }
      }
      uint8_t* prow = sP + r * 128;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8)
        *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
      // Rows of the last block past the request's keys may hold anything
      // (even NaN): zero them in V so that 0 * garbage never reaches O.
      const int vrows = k_end - key0;
      if (vrows < kBN) {
        uint8_t* vt = sV + (j % S) * C::kTileBytes;
        const int pieces = (kBN - vrows) * C::kHalves * 8;
        for (int p = r; p < pieces; p += 128) {
          const int row = vrows + p / (C::kHalves * 8);
          const int rem = p % (C::kHalves * 8);
          *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kBN * 128) + row * 128 + ((rem & 7) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && nblk > 0) ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (nblk - 1) & 1, abort_v));
    if (ok && nblk > 0) {
      tc_fence_after();
      const int gr = row0 + r;
      const int node = gr / G;
      const int h = g * G + (gr - node * G);
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      if (nch == 1) {
        __nv_bfloat16* dst = out + ((size_t)(off + node) * plan.Hq + h) * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              d4[e] = make_uint4(pack_bf16x2(o[8 * e] * inv_l, o[8 * e + 1] * inv_l),
                                 pack_bf16x2(o[8 * e + 2] * inv_l, o[8 * e + 3] * inv_l),
                                 pack_bf16x2(o[8 * e + 4] * inv_l, o[8 * e + 5] * inv_l),
                                 pack_bf16x2(o[8 * e + 6] * inv_l, o[8 * e + 7] * inv_l));
          }
        }
      } else {
        const int64_t prow_i = plan.part_row[b] + (int64_t)(g * nch + c) * R + gr;
        float* dst = part_o + prow_i * D;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
          if (valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(o[4 * e] * inv_l, o[4 * e + 1] * inv_l, o[4 * e + 2] * inv_l,
                                  o[4 * e + 3] * inv_l);
          }
        }
        if (valid) part_lse[prow_i] = l > 0.f ? m_ref + log2f(l) : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_v) status[b] = TSV_ERR_TIMEOUT;
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merges the per-chunk partials of one (request, KV head): out = sum_c w_c o_c
// / sum_c w_c with w_c = 2^(lse_c - max lse).
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const __grid_constant__ AttnPlan plan, const float* __restrict__ part_o,
                        const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out) {
  const int b = blockIdx.z, g = blockIdx.y;
  const int nch = plan.n_chunks[b];
  if (nch <= 1) return;
  const int D = plan.D, G = plan.G, R = plan.nodes[b] * G, off = plan.node_off[b];
  const int D4 = D / 4;
  const int64_t base0 = plan.part_row[b] + (int64_t)g * nch * R;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < R * D4; e += gridDim.x * blockDim.x) {
    const int r = e / D4, d4 = e - (e / D4) * D4;
    float M = -INFINITY;
    for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, part_lse[base0 + (int64_t)cc * R + r]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = 0; cc < nch; ++cc) {
      const int64_t pr = base0 + (int64_t)cc * R + r;
      const float lse = part_lse[pr];
      if (lse == -INFINITY) continue;
      const float w = exp2f(lse - M);
      const float4 o = reinterpret_cast<const float4*>(part_o + pr * D)[d4];
      wsum += w;
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int node = r / G, h = g * G + (r - node * G);
    uint2 v = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2*>(out + ((size_t)(off + node) * plan.Hq + h) * D + d4 * 4) = v;
  }
}

size_t attention_tc_smem_bytes(int D) {
  return D == 64 ? (size_t)TcCfg<64>::kSmemBytes : (size_t)TcCfg<128>::kSmemBytes;
}

cudaError_t attention_tc_set_attributes(int D) {
  if (D == 64)
    return cudaFuncSetAttribute(tree_attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcCfg<64>::kSmemBytes);
  return cudaFuncSetAttribute(tree_attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcCfg<128>::kSmemBytes);
}

cudaError_t launch_attention_tc(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                const AttnPlan& plan, const void* q, const uint32_t* anc,
                                void* out, float* part_o, float* part_lse, int32_t* status,
                                int num_sms, cudaStream_t st) {
  (void)num_sms;
  if (plan.n_units == 0) return cudaSuccess;
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  if (plan.D == 64)
    tree_attn_tc_kernel<64><<<plan.n_units, kTcThreads, TcCfg<64>::kSmemBytes, st>>>(
        tmap_k, tmap_v, plan, qb, anc, ob, part_o, part_lse, status);
  else
    tree_attn_tc_kernel<128><<<plan.n_units, kTcThreads, TcCfg<128>::kSmemBytes, st>>>(
        tmap_k, tmap_v, plan, qb, anc, ob, part_o, part_lse, status);
  return cudaGetLastError();
}

cudaError_t launch_attention_combine(const AttnPlan& plan, const float* part_o,
                                     const float* part_lse, void* out, cudaStream_t st) {
  if (plan.part_rows_total == 0) return cudaSuccess;
  int max_r = 0;
  for (int b = 0; b < plan.B; ++b)
    if (plan.n_chunks[b] > 1 && plan.nodes[b] * plan.G > max_r) max_r = plan.nodes[b] * plan.G;
  const int elems = max_r * (plan.D / 4);
  int gx = (elems + 255) / 256;
  if (gx > 64) gx = 64;
  dim3 grid(gx, plan.Hkv, plan.B);
  attn_combine_kernel<<<grid, 256, 0, st>>>(plan, part_o, part_lse,
                                            static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace tsv
