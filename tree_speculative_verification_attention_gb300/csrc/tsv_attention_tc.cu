// tsv_attention_tc.cu — tree attention on the 5th-generation tensor cores,
// query rows on the TMEM lanes.
//
// What it computes (SpecInfer §4 Token Tree Verifier, "Tree Attention" and
// "Tree-Based Parallel Decoding"): every tree node attends to the shared
// prefix of the KV cache plus the tree keys of its own root-to-node path, all
// tree nodes of a request in one kernel through a topology-aware mask.  The
// cache / in-tree split and merge of Staged Speculative Decoding (§3,
// Implementation) becomes a split of each request's keys into chunks whose
// partial results are merged by log-sum-exp.
//
// One CTA = one unit (request b, KV head g, key chunk c, pair of M-tiles).
// The 128 query rows of an M-tile are (node, head-in-group) pairs: all query
// heads that share KV head g sit in the same tiles, and the two tiles of a
// CTA read every streamed K/V block once from shared memory, so each K/V row
// serves up to 256 query rows.  Warp roles (320 threads):
//   warp 8        TMA producer: the Q tiles first, then K and V blocks of 64
//                 rows x D, 128-byte swizzled, into a ring of kStages stages.
//   warp 9        tcgen05 issuer and TMEM owner (512 columns: per tile two S
//                 buffers and the O accumulator).  Per block: S_t = Q_t K^T
//                 for both tiles, then O_t += P_t V with P_t read from TMEM.
//   warps 0-3,    softmax warpgroup of tile 0 and tile 1: one thread per query
//   warps 4-7     row (= TMEM lane).  Set-up: the ancestor bitset of the row's
//                 node (prepared, or by walking parent[] up to the root).
//                 Loop: read S, mask the tree part of the keys with the bitset,
//                 online softmax in base 2 with a lazily moved reference
//                 maximum, P in bf16 written back over S in TMEM, O rescaled in
//                 TMEM when the reference moves.  End: normalise and store the
//                 output; when a request's keys are split over several CTAs,
//                 store a partial + log2-sum-exp and let the last CTA of the
//                 group (atomic counter, no waiting) merge the partials.
// Two softmax warpgroups put two warps on each SM sub-partition, so one
// warp's exponentials overlap the other's TMEM traffic and waits.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kTcSoftmaxThreads = 256;  // two warpgroups, one per M-tile
constexpr int kTcThreads = kTcSoftmaxThreads + 64;
constexpr int kTcProducerWarp = 8, kTcMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8 between rescales
constexpr int kBarTcSetup = 1;             // softmax warps + MMA warp
constexpr int kBarTcSoftmax = 2;           // both softmax warpgroups

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;               // 128-byte column groups per row
  static constexpr int kStages = (D == 128) ? 4 : 8;   // K/V ring depth
  static constexpr int kQTile = kBM * D * 2;           // one M-tile of Q
  static constexpr int kTileBytes = kBN * D * 2;       // one K (or V) block
  static constexpr int kAncWords = TSV_ANC_WORDS + 2;  // two zero words past the end
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffAnc = kOffV + kStages * kTileBytes;
  static constexpr int kOffPar = kOffAnc + 2 * kBM * kAncWords * 4;
  static constexpr int kOffBar = kOffPar + TSV_MAX_NODES * 4;
  // q_full, kv_full[S], kv_empty[S], per tile s_full[2] p_full[2] pv_done[2], mma_done
  static constexpr int kNumBars = 1 + 2 * kStages + 12 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kTileCols = 256;               // S0 | S1 | O per tile
  static constexpr uint32_t kTmemCols = 2 * kTileCols;
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kTileBytes % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(2 * kBN + D <= (int)kTileCols, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
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
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + C::kOffAnc);
  int32_t* sPar = reinterpret_cast<int32_t*>(smem + C::kOffPar);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + S;
  uint64_t* tile_bars = kv_empty + S;  // tile t: s_full[2], p_full[2], pv_done[2] at 6t
  uint64_t* mma_done = tile_bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  int* last_cta = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
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
  const int npairs = (mtiles + 1) >> 1;
  const int pr = local % npairs;
  const int cg = local / npairs;
  const int c = cg % nch;
  const int g = cg / nch;
  const int G = plan.G;
  const int P = plan.prefix[b], n = plan.nodes[b], off = plan.node_off[b];
  const int R = n * G;
  const int ntiles = min(2, mtiles - 2 * pr);  // 1 or 2
  const int k_begin = c * plan.chunk_keys;
  const int k_end = min(P + n, k_begin + plan.chunk_keys);
  const int nblk = (k_end - k_begin + kBN - 1) / kBN;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t)
      for (int x = 0; x < 2; ++x) {
        mbar_init(&tile_bars[6 * t + x], 1);        // s_full
        mbar_init(&tile_bars[6 * t + 2 + x], 128);  // p_full: every softmax thread of the tile
        mbar_init(&tile_bars[6 * t + 4 + x], 1);    // pv_done
      }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kTcProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      // Q tile t: box (64 d, G heads, 128/G nodes) lands as 128 rows r = node*G + head.
      mbar_arrive_expect_tx(q_full, ntiles * C::kQTile);
      for (int t = 0; t < ntiles; ++t)
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(sQ + t * C::kQTile + hf * (kBM * 128), &tmap_q, q_full, hf * 64, g * G,
                      off + (2 * pr + t) * kBM / G, l2_policy_evict_first());
      const uint64_t pol = npairs > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
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
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
    named_bar(kBarTcSetup, kTcSoftmaxThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, 1);
      // Base descriptors, built once; an operand at byte offset x from its base
      // is the base plus x / 16 (the start-address field, no carry out of it).
      const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      auto issue_s = [&](int t, int j) {
        const uint32_t dst = tmem + t * C::kTileCols + (uint32_t)((j & 1) * kBN);
        const uint64_t da = dq + (uint64_t)((t * C::kQTile) >> 4);
        const uint64_t db = dk + (uint64_t)(((j % S) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4;
          umma_bf16(dst, da + ao, db + bo, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&tile_bars[6 * t + (j & 1)]);
      };
      auto issue_pv = [&](int t, int j) {
        const uint32_t pa = tmem + t * C::kTileCols + (uint32_t)((j & 1) * kBN);  // P over S(j)
        const uint32_t tO = tmem + t * C::kTileCols + 2 * kBN;
        const uint64_t db = dv + (uint64_t)(((j % S) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_bf16_ts(tO, pa + kk * 8, db + (uint32_t)((kk * 16 * 128) >> 4), idPV,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&tile_bars[6 * t + 4 + (j & 1)]);
      };
      bool ok = nblk > 0 && mbar_wait(q_full, 0, abort_v) && mbar_wait(&kv_full[0], 0, abort_v);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) issue_s(t, 0);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + 1 < nblk) {
          if (!mbar_wait(&kv_full[(j + 1) % S], ((j + 1) / S) & 1, abort_v)) break;
          tc_fence_after();
          for (int t = 0; t < ntiles; ++t) issue_s(t, j + 1);
        }
        for (int t = 0; ok && t < ntiles; ++t) {
          if (!mbar_wait(&tile_bars[6 * t + 2 + (j & 1)], (j >> 1) & 1, abort_v)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, j);
        }
        if (ok) umma_commit(&kv_empty[j % S]);
      }
      umma_commit(mma_done);  // every MMA of this CTA has finished before TMEM is freed
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // M-tile of this warpgroup
    const int r = tid & 127;  // row within the tile = TMEM lane
    const int row0 = (2 * pr + t) * kBM;
    const bool tile_on = t < ntiles;
    const int rows_valid = tile_on ? min(kBM, R - row0) : 0;
    const bool valid = r < rows_valid;
    uint64_t* s_full = tile_bars + 6 * t;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = s_full + 4;
    // Ancestor bitset of this row's node.
    uint32_t* arow = sAnc + (t * kBM + r) * C::kAncWords;
#pragma unroll
    for (int w = 0; w < C::kAncWords; ++w) arow[w] = 0u;
    if (anc != nullptr) {
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(anc + (size_t)(off + (row0 + r) / G) * TSV_ANC_WORDS);
        const uint4 a0 = __ldg(src), a1 = __ldg(src + 1);
        arow[0] = a0.x; arow[1] = a0.y; arow[2] = a0.z; arow[3] = a0.w;
        arow[4] = a1.x; arow[5] = a1.y; arow[6] = a1.z; arow[7] = a1.w;
      }
    } else {
      // parent[] of the request (n <= 256 = one entry per softmax thread),
      // validated, then each row walks from its node up to the root.
      int p = -1;
      if (tid < n) {
        p = __ldg(parent + off + tid);
        sPar[tid] = p;
      }
      const bool bad = named_bar_or(kBarTcSoftmax, kTcSoftmaxThreads, tid < n && (p < -1 || p >= tid));
      if (local == 0 && tid == 0) status[b] = bad ? TSV_ERR_BAD_TREE : TSV_OK;
      if (valid && !bad)
        for (int a = (row0 + r) / G; a >= 0; a = sPar[a]) arow[a >> 5] |= 1u << (a & 31);
    }
    tc_fence_before();
    named_bar(kBarTcSetup, kTcSoftmaxThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tcol = tmem + lane_base + t * C::kTileCols;
    const float sl2 = plan.scale_log2;
    const int my_nblk = tile_on ? nblk : 0;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < my_nblk; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_v));
      if (!ok) break;
      tc_fence_after();
      const uint32_t sbuf = tcol + (uint32_t)((j & 1) * kBN);
      float s[kBN];
      {
        float t0[32], t1[32];
        tmem_ld32(sbuf, t0);
        tmem_ld32(sbuf + 32, t1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          s[e] = t0[e];
          s[32 + e] = t1[e];
        }
      }
      const int key0 = k_begin + j * kBN;
      if (key0 + kBN > P) {  // uniform: the block reaches the tree keys (or past the request)
        const uint64_t vis = valid ? block_visibility(arow, key0 - P) : 0ull;
#pragma unroll
        for (int e = 0; e < kBN; ++e) s[e] = ((vis >> e) & 1ull) ? s[e] : -INFINITY;
      } else if (!valid) {
#pragma unroll
        for (int e = 0; e < kBN; ++e) s[e] = -INFINITY;
      }
      // Raw maximum (the scale is positive, so it commutes with the max).
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int e = 4; e < kBN; ++e) mx[e & 3] = fmaxf(mx[e & 3], s[e]);
      const float bmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      // Move the reference maximum only when the block's max exceeds it by
      // more than the threshold (always on the first visible block).
      float alpha = 1.f;
      bool resc = false;
      if (bmax > m_ref + kRescaleThreshold) {
        alpha = fast_exp2(m_ref - bmax);  // 0 when m_ref = -inf
        m_ref = bmax;
        resc = true;
      }
      const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;
      uint32_t pk[kBN / 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < kBN; e += 2) {
        const float p0 = fast_exp2(fmaf(s[e], sl2, neg_ref));
        const float p1 = fast_exp2(fmaf(s[e + 1], sl2, neg_ref));
        ps[(e >> 1) & 3] += p0 + p1;
        pk[e >> 1] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      // O must hold PV(j-1) before it is rescaled.
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_v));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tcol + (uint32_t)(2 * kBN + cc), o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tcol + (uint32_t)(2 * kBN + cc), o);
        }
      }
      // P (bf16, two per column) over the first 32 columns of S(j), whose
      // values are all in registers now.
      {
        uint32_t h0[16], h1[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          h0[e] = pk[e];
          h1[e] = pk[16 + e];
        }
        tmem_st16u(sbuf, h0);
        tmem_st16u(sbuf + 16, h1);
      }
      // Rows of the last block past the request's keys may hold anything
      // (even NaN): zero them in V so that 0 * garbage never reaches O.  Tile
      // 0's warpgroup does it; PV of tile 1 is issued after PV of tile 0.
      const int vrows = k_end - key0;
      if (t == 0 && vrows < kBN) {
        uint8_t* vt = sV + (j % S) * C::kTileBytes;
        const int pieces = (kBN - vrows) * C::kHalves * 8;
        for (int q = r; q < pieces; q += kBM) {
          const int row = vrows + q / (C::kHalves * 8);
          const int rem = q % (C::kHalves * 8);
          *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kBN * 128) + row * 128 + ((rem & 7) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok && my_nblk > 0)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&pv_done[(my_nblk - 1) & 1], ((my_nblk - 1) >> 1) & 1, abort_v));
    // Agree on success CTA-wide: the merge below has named barriers that all
    // 256 softmax threads must reach.
    ok = !named_bar_or(kBarTcSoftmax, kTcSoftmaxThreads, !ok);
    if (ok && nblk > 0) {
      if (tile_on) tc_fence_after();
      const int gr = row0 + r;
      const int node = gr / G;
      const int h = g * G + (gr - node * G);
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      if (nch == 1) {
        if (tile_on) {
          __nv_bfloat16* dst = out + ((size_t)(off + node) * plan.Hq + h) * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(tcol + (uint32_t)(2 * kBN + cc), o);
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
        }
      } else {
        // Partial of this chunk, then the group's last CTA merges all chunks.
        const int64_t base0 = plan.part_row[b] + (int64_t)g * nch * R;
        if (tile_on) {
          const int64_t prow_i = base0 + (int64_t)c * R + gr;
          float* dst = part_o + prow_i * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(tcol + (uint32_t)(2 * kBN + cc), o);
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
        __threadfence();
        named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
        int32_t* ctr = counters + plan.ctr_base[b] + g * npairs + pr;
        if (tid == 0) *last_cta = atomicAdd(ctr, 1) == nch - 1;
        named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
        if (*last_cta) {
          __threadfence();
          // Warp w merges rows w, w+8, ... of the pair.  Lane c holds the
          // log2-sum-exp of chunks c and c + 32 (at most 64 chunks); the
          // weights meet by shuffles, then each lane owns D/32 columns and
          // keeps eight chunks' loads in flight.
          constexpr int E = D / 32;
          const int prow0 = 2 * pr * kBM;
          const int rows_pair = min(2 * kBM, R - prow0);
          for (int rr = warp; rr < rows_pair; rr += kTcSoftmaxThreads / 32) {
            const int grr = prow0 + rr;
            const float l0 = lane < nch ? __ldcg(part_lse + base0 + (int64_t)lane * R + grr) : -INFINITY;
            const float l1 = lane + 32 < nch ? __ldcg(part_lse + base0 + (int64_t)(lane + 32) * R + grr) : -INFINITY;
            float M = fmaxf(l0, l1);
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
            const float w0 = (l0 == -INFINITY) ? 0.f : fast_exp2(l0 - M);
            const float w1 = (l1 == -INFINITY) ? 0.f : fast_exp2(l1 - M);
            float wsum = w0 + w1;
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o2);
            const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
            float acc[E];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = 0.f;
            const float* src0 = part_o + (base0 + grr) * D + lane * E;
            for (int c0 = 0; c0 < nch; c0 += 8) {
              float v[8][E];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                if (c0 + u < nch) {
                  const float* src = src0 + (int64_t)(c0 + u) * R * D;
                  if constexpr (E == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
                    v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                  } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
                    v[u][0] = x.x; v[u][1] = x.y;
                  }
                }
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int cc = c0 + u;
                const float w = __shfl_sync(0xffffffffu, cc < 32 ? w0 : w1, cc & 31);
                if (cc < nch && w > 0.f) {
#pragma unroll
                  for (int e = 0; e < E; ++e) acc[e] += w * v[u][e];
                }
              }
            }
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
  if (warp == kTcMmaWarp) {
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
