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
//   warp 4        TMA producer: the Q tile first, then K and V blocks of 64
//                 rows x D, 128-byte swizzled, into a ring of kStages stages.
//                 It starts right after the barriers exist, so the first
//                 loads overlap everything else the CTA sets up.
//   warp 5        tcgen05 issuer: S = Q K^T into TMEM (two buffers), then
//                 O += P V into a TMEM accumulator; owns TMEM allocation.
//   warps 0-3     one thread per query row (= TMEM lane).  Set-up: the
//                 ancestor bitsets of the tile's nodes, read from the
//                 prepared array or computed here from parent[] by pointer
//                 jumping.  Loop: read S, mask the tree part of the keys with
//                 the bitset, online softmax in base 2 with a lazily moved
//                 reference maximum, write P (bf16, two buffers) to shared
//                 memory, rescale O in TMEM when the reference moves.  End:
//                 normalise and store the output; when the request's keys are
//                 split over several CTAs, store a partial + log2-sum-exp and
//                 let the last CTA of the group (atomic counter, no waiting)
//                 merge the partials into the output.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kTcThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8 between rescales

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;               // 128-byte column groups per row
  static constexpr int kStages = (D == 128) ? 4 : 8;   // K/V ring depth
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kTileBytes = kBN * D * 2;       // one K (or V) block
  static constexpr int kPBytes = kBM * kBN * 2;        // one P buffer
  static constexpr int kAncWords = TSV_ANC_WORDS + 2;  // two zero words past the end
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffAnc = kOffP + 2 * kPBytes;
  static constexpr int kOffBar = kOffAnc + kBM * kAncWords * 4;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done[2], mma_done
  static constexpr int kNumBars = 1 + 2 * kStages + 7;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kTmemCols = 256;               // S0 | S1 | O
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(2 * kBN + D <= (int)kTmemCols, "TMEM columns");
  // Pointer-jumping scratch (two bitset buffers + two jump buffers) reuses the P buffers.
  static_assert(2 * TSV_MAX_NODES * TSV_ANC_WORDS * 4 + 2 * TSV_MAX_NODES * 4 <= 2 * kPBytes,
                "ancestor scratch");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ AttnPlan plan, const int32_t* __restrict__ parent,
                        const uint32_t* __restrict__ anc, __nv_bfloat16* __restrict__ out,
                        float* __restrict__ part_o, float* __restrict__ part_lse,
                        int32_t* __restrict__ counters, int32_t* __restrict__ status) {
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
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + S;
  uint64_t* s_full = kv_empty + S;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* mma_done = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  int* bad_tree = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  int* last_cta = reinterpret_cast<int*>(smem + C::kOffMisc + 12);
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
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);  // every softmax thread arrives
      mbar_init(&pv_done[x], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *bad_tree = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      // Q tile: box (64 d, G heads, 128/G nodes) lands as 128 rows r = node*G + head.
      mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(sQ + hf * (kBM * 128), &tmap_q, q_full, hf * 64, g * G, off + row0 / G,
                    l2_policy_evict_first());
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
        mbar_wait(q_full, 0, nullptr);
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait(&kv_full[j % S], (j / S) & 1, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
    named_bar(kBarSetup, 160);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
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
        const uint32_t pbuf = pa + (uint32_t)((j & 1) * C::kPBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t bo = st * C::kTileBytes + kk * 16 * 128;
          umma_bf16(tO, sdesc_sw128(pbuf + kk * 32, 16, 1024),
                    sdesc_sw128(va + bo, kBN * 128, 1024), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = nblk > 0 && mbar_wait(q_full, 0, abort_v) && mbar_wait(&kv_full[0], 0, abort_v);
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
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_v)) break;
        tc_fence_after();
        issue_pv(j);
        umma_commit(&pv_done[j & 1]);
        umma_commit(&kv_empty[j % S]);
      }
      umma_commit(mma_done);  // every MMA of this CTA has finished before TMEM is freed
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;
    const bool valid = r < rows_valid;
    // Ancestor bitsets of the tile's rows.
    if (anc != nullptr) {
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(anc + (size_t)(off + (row0 + r) / G) * TSV_ANC_WORDS);
        const uint4 a0 = __ldg(src), a1 = __ldg(src + 1);
        uint32_t* dst = sAnc + r * C::kAncWords;
        dst[0] = a0.x; dst[1] = a0.y; dst[2] = a0.z; dst[3] = a0.w;
        dst[4] = a1.x; dst[5] = a1.y; dst[6] = a1.z; dst[7] = a1.w;
        dst[8] = 0u; dst[9] = 0u;
      }
    } else {
      const uint32_t* A = ancestors_by_pointer_jumping(parent + off, n,
                                                       reinterpret_cast<uint32_t*>(sP), bad_tree);
      const bool bad = *bad_tree != 0;
      if (valid) {
        const int node = (row0 + r) / G;
        uint32_t* dst = sAnc + r * C::kAncWords;
#pragma unroll
        for (int w = 0; w < TSV_ANC_WORDS; ++w) dst[w] = bad ? 0u : A[node * TSV_ANC_WORDS + w];
        dst[8] = 0u;
        dst[9] = 0u;
      }
      if (local == 0 && tid == 0) status[b] = bad ? TSV_ERR_BAD_TREE : TSV_OK;
      named_bar(kBarSoftmax, 128);  // scratch (the P buffers) free again
    }
    tc_fence_before();
    named_bar(kBarSetup, 160);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
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
      // P buffer j&1 was last read by PV(j-2); O must hold PV(j-1) before a rescale.
      if (j >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[j & 1], ((j - 2) >> 1) & 1, abort_v));
        if (!ok) break;
      }
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_v));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tmem + lane_base + (uint32_t)(2 * kBN + cc), o);
        }
      }
      uint8_t* prow = sP + (j & 1) * C::kPBytes + r * 128;
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
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok && nblk > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&pv_done[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1, abort_v));
    // Agree on success CTA-wide: the merge below has named barriers that all
    // 128 softmax threads must reach.
    ok = !named_bar_or(kBarSoftmax, 128, !ok);
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
        // Partial of this chunk, then the group's last CTA merges all chunks.
        const int64_t base0 = plan.part_row[b] + (int64_t)g * nch * R;
        const int64_t prow_i = base0 + (int64_t)c * R + gr;
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
        __threadfence();
        named_bar(kBarSoftmax, 128);
        int32_t* ctr = counters + plan.ctr_base[b] + g * mtiles + mt;
        if (tid == 0) *last_cta = atomicAdd(ctr, 1) == nch - 1;
        named_bar(kBarSoftmax, 128);
        if (*last_cta) {
          __threadfence();
          // Warp w merges rows w, w+4, ...; each lane owns D/32 columns.
          constexpr int E = D / 32;
          for (int rr = warp; rr < rows_valid; rr += 4) {
            const int grr = row0 + rr;
            float M = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(part_lse + base0 + (int64_t)cc * R + grr));
            float acc[E], wsum = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
              const int64_t pr = base0 + (int64_t)cc * R + grr;
              const float lse = __ldcg(part_lse + pr);
              if (lse == -INFINITY) continue;
              const float w = fast_exp2(lse - M);
              wsum += w;
              const float* src = part_o + pr * D + lane * E;
              if constexpr (E == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
              } else {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
                acc[0] += w * v.x; acc[1] += w * v.y;
              }
            }
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            const int nd = grr / G, hh = g * G + (grr - nd * G);
            __nv_bfloat16* o = out + ((size_t)(off + nd) * plan.Hq + hh) * D + lane * E;
            if constexpr (E == 4) {
              *reinterpret_cast<uint2*>(o) =
                  make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
            } else {
              *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            }
          }
          if (tid == 0) *ctr = 0;  // leave the counter zeroed for the next call
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_v) status[b] = TSV_ERR_TIMEOUT;
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, C::kTmemCols);
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

cudaError_t launch_attention_tc(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const AttnPlan& plan,
                                const int32_t* parent, const uint32_t* anc, void* out,
                                float* part_o, float* part_lse, int32_t* counters,
                                int32_t* status, cudaStream_t st) {
  if (plan.n_units == 0) return cudaSuccess;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  if (plan.D == 64)
    tree_attn_tc_kernel<64><<<plan.n_units, kTcThreads, TcCfg<64>::kSmemBytes, st>>>(
        tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
  else
    tree_attn_tc_kernel<128><<<plan.n_units, kTcThreads, TcCfg<128>::kSmemBytes, st>>>(
        tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
  return cudaGetLastError();
}

}  // namespace tsv
