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
// One CTA = one unit (request b, KV head g, key chunk c, tile pair tp): two
// query tiles of 128 rows, rows = (node, head-in-group) pairs, so all query
// heads that share KV head g sit in the same tiles and each streamed K/V row
// serves every tree node and every grouped head of both tiles at once.  Keys
// go in blocks of 128, so both MMAs of a block have N >= 128 (smaller N runs
// the tensor pipe below its rate).  Warp roles (320 threads):
//   warp 8        TMA producer.  Lane 0: both Q tiles, then K blocks into a
//                 2-stage ring, each released once both tiles' S have read
//                 it; lane 1: V blocks into a 2-stage ring, released after
//                 both tiles' PV.
//   warp 9        tcgen05 issuer and TMEM owner (S_0 | S_1 | O_0 | O_1).
//                 Per block j it issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1):
//                 while one tile's softmax runs, the tensor pipe works for the
//                 other.  O_t += P_t V reads P_t from TMEM.
//   warps 0-7     softmax.  Warps 0-3 serve tile 0 and warps 4-7 tile 1; each
//                 thread owns the row on its TMEM lane and all 128 keys of a
//                 block.  Set-up: the ancestor bitset of the row's node
//                 (prepared, or by walking parent[] up to the root).  Loop:
//                 read S, mask the tree part of the keys with the bitset (and
//                 keys past the chunk by count), base-2 online softmax with a
//                 lazily moved reference maximum, O_t rescaled in TMEM when
//                 the reference moves, P in bf16 written back over the tile's
//                 S columns.  End: normalise and store; when a request's keys
//                 are split over several CTAs, store a partial + log2-sum-exp
//                 and let the last CTA of the group (atomic counter, no
//                 waiting) merge the partials.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kTcSoftmaxThreads = 256;
constexpr int kTcThreads = kTcSoftmaxThreads + 64;
constexpr int kTcProducerWarp = 8, kTcMmaWarp = 9;
constexpr int kTcTiles = 2;                // query tiles of 128 rows per CTA
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8 between rescales
constexpr int kBarTcSetup = 1;             // softmax warps + MMA warp
constexpr int kBarTcSoftmax = 2;           // softmax warps

template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;      // 128-byte column groups per row
  static constexpr int kKStages = 2, kVStages = 2;
  static constexpr int kQTileBytes = kBM * D * 2;
  static constexpr int kQBytes = kTcTiles * kQTileBytes;
  static constexpr int kTileBytes = kBN * D * 2;  // one K (or V) block
  static constexpr int kAncWords = TSV_ANC_WORDS + 2;  // two zero words past the end
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffAnc = kOffV + kVStages * kTileBytes;
  static constexpr int kOffPar = kOffAnc + kTcTiles * kBM * kAncWords * 4;
  static constexpr int kOffLse = kOffPar + TSV_MAX_NODES * 4;  // float [256]: the pair's rows
  static constexpr int kOffBar = kOffLse + kTcTiles * kBM * 4;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[tile],
  // p_full[tile], pv_done[tile], mma_done
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 * kTcTiles + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kColO = kTcTiles * kBN;        // S0 | S1 | O0 | O1
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kTileBytes % 1024 == 0, "swizzle atoms");
  static_assert(kQTileBytes % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kColO + kTcTiles * D <= kTmemCols, "TMEM columns");
  static_assert(kOffV == kOffK + kKStages * kTileBytes, "the K and V rings are contiguous");
  static_assert((kKStages + kVStages) * kTileBytes >= (64 + 1) * kBM * 4, "merge weights fit in the K/V rings");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert((kKStages + kVStages) * kTileBytes >= kTcTiles * kBM * D * 4, "cluster partials fit in the K/V rings");
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
  constexpr int SK = C::kKStages, SV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + C::kOffAnc);
  int32_t* sPar = reinterpret_cast<int32_t*>(smem + C::kOffPar);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;       // [tile]
  uint64_t* p_full = s_full + kTcTiles;  // [tile]
  uint64_t* pv_done = p_full + kTcTiles;  // [tile]
  uint64_t* mma_done = pv_done + kTcTiles;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  int* last_cta = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  volatile int* abort_v = abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- the unit
  // (request b, KV head g, key chunk c, tile pair tp): query rows
  // [256 tp, 256 tp + 256) of the request, tile t = rows 256 tp + 128 t ...
  const int unit = blockIdx.x;
  int lo = 0, hi = plan.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (plan.unit_start[mid] <= unit) lo = mid; else hi = mid;
  }
  const int b = plan.slot_req[lo];
  const int local = unit - plan.unit_start[lo];
  const int mtiles = plan.mtiles[b], nch = plan.n_chunks[b];
  const int pairs = (mtiles + kTcTiles - 1) / kTcTiles;
  // Clustered plans (plan.cluster == nch): the chunks of one (KV head, tile
  // pair) are consecutive units and form one cluster, rank = chunk.
  const bool clustered = plan.cluster > 1;
  const int tp = clustered ? (local / nch) % pairs : local % pairs;
  const int c = clustered ? local % nch : (local / pairs) % nch;
  const int g = clustered ? local / nch / pairs : local / pairs / nch;
  const int G = plan.G;
  const int P = plan.prefix[b], n = plan.nodes[b], off = plan.node_off[b];
  const int R = n * G;
  const int row0 = tp * kTcTiles * kBM;
  const int ntiles = min(kTcTiles, mtiles - tp * kTcTiles);  // 1 or 2
  const int k_begin = c * plan.chunk_keys;
  const int k_end = min(P + n, k_begin + plan.chunk_keys);
  const int nblk = (k_end - k_begin + kBN - 1) / kBN;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kBM);  // every thread of the tile
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // the previous kernel's results are visible from here on
  // The next kernel may be scheduled now: it waits for this one's completion
  // itself, and it is launched only once every CTA of this grid has started,
  // so it only takes SM room this grid leaves free (verification launched to
  // run beside this attention fills that room).
  pdl_trigger();

  if (warp == kTcProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = mtiles > kTcTiles ? l2_policy_evict_last() : l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      // Q tile t: box (64 d, G heads, 128/G nodes) lands as 128 rows r = node*G + head.
      mbar_arrive_expect_tx(q_full, ntiles * C::kQTileBytes);
      for (int t = 0; t < ntiles; ++t)
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(sQ + t * C::kQTileBytes + hf * (kBM * 128), &tmap_q, q_full, hf * 64, g * G,
                      off + (row0 + t * kBM) / G, l2_policy_evict_first());
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % SK;
        if (j >= SK && !mbar_wait(&k_empty[st], ((j / SK) - 1) & 1, abort_v)) break;
        mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_4d(sK + st * C::kTileBytes + hf * (kBN * 128), &tmap_k, &k_full[st], hf * 64, g,
                      k_begin + j * kBN, b, pol);
        ++issued;
      }
      if (*abort_v) {  // let copies still in flight land before the CTA exits
        mbar_wait(q_full, 0, nullptr);
        for (int j = (issued > SK ? issued - SK : 0); j < issued; ++j)
          mbar_wait(&k_full[j % SK], (j / SK) & 1, nullptr);
      }
    } else if (lane == 1) {
      tma_prefetch_desc(&tmap_v);
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % SV;
        if (j >= SV && !mbar_wait(&v_empty[st], ((j / SV) - 1) & 1, abort_v)) break;
        mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_4d(sV + st * C::kTileBytes + hf * (kBN * 128), &tmap_v, &v_full[st], hf * 64, g,
                      k_begin + j * kBN, b, pol);
        ++issued;
      }
      if (*abort_v)
        for (int j = (issued > SV ? issued - SV : 0); j < issued; ++j)
          mbar_wait(&v_full[j % SV], (j / SV) & 1, nullptr);
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
      // S_t = Q_t K(j)^T into the tile's S columns.
      auto issue_s = [&](int t, int j) {
        const uint32_t dst = tmem + (uint32_t)(t * kBN);
        const uint64_t da = dq + (uint64_t)((t * C::kQTileBytes) >> 4);
        const uint64_t db = dk + (uint64_t)(((j % SK) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4;
          umma_bf16(dst, da + ao, db + bo, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[t]);
      };
      // O_t += P_t V(j): P_t (128 keys, bf16, two per column) over the tile's
      // first 64 S columns, read from TMEM.
      auto issue_pv = [&](int t, int j) {
        const uint32_t pa = tmem + (uint32_t)(t * kBN);
        const uint64_t db = dv + (uint64_t)(((j % SV) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_bf16_ts(tmem + C::kColO + t * D, pa + kk * 8, db + (uint32_t)((kk * 16 * 128) >> 4), idPV,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[t]);
      };
      // Order: S_0(0) S_1(0), then per block PV_0(j) S_0(j+1) PV_1(j) S_1(j+1):
      // while one tile's softmax runs, the tensor pipe works for the other.
      bool ok = nblk > 0 && mbar_wait(q_full, 0, abort_v) && mbar_wait(&k_full[0], 0, abort_v);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t) issue_s(t, 0);
        umma_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        const bool more = j + 1 < nblk;
        if (!mbar_wait(&v_full[j % SV], (j / SV) & 1, abort_v)) break;
        if (!mbar_wait(&p_full[0], j & 1, abort_v)) break;
        tc_fence_after();
        issue_pv(0, j);
        if (more) {
          if (!mbar_wait(&k_full[(j + 1) % SK], ((j + 1) / SK) & 1, abort_v)) break;
          tc_fence_after();
          issue_s(0, j + 1);
        }
        if (ntiles > 1) {
          if (!mbar_wait(&p_full[1], j & 1, abort_v)) break;
          tc_fence_after();
          issue_pv(1, j);
        }
        umma_commit(&v_empty[j % SV]);
        if (more) {
          if (ntiles > 1) issue_s(1, j + 1);
          umma_commit(&k_empty[(j + 1) % SK]);
        }
      }
      umma_commit(mma_done);  // every MMA of this CTA has finished before TMEM is freed
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;        // query tile
    const int r = tid & (kBM - 1);  // row of the tile = TMEM lane
    const int rows_valid = min(kBM, R - (row0 + t * kBM));  // <= 0 for a missing tile
    const bool valid = r < rows_valid;
    const int grow = row0 + t * kBM + r;  // row of the request
    // Ancestor bitset of this row's node.
    uint32_t* arow = sAnc + (t * kBM + r) * C::kAncWords;
#pragma unroll
    for (int w = 0; w < C::kAncWords; ++w) arow[w] = 0u;
    if (anc != nullptr) {
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(anc + (size_t)(off + grow / G) * TSV_ANC_WORDS);
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
        for (int a = grow / G; a >= 0; a = sPar[a]) arow[a >> 5] |= 1u << (a & 31);
    }
    tc_fence_before();
    named_bar(kBarTcSetup, kTcSoftmaxThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t sbuf = trow + (uint32_t)(t * kBN);               // S_t / P_t of this row
    const uint32_t o_mine = trow + C::kColO + (uint32_t)(t * D);    // O_t of this row
    const float sl2 = plan.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    // No barrier inside the loop: a timed-out wait ends this warp's loop
    // (every wait is bounded and sets the CTA's abort flag, so the other
    // warps' waits end quickly too); the CTA agrees after the loop.
    bool ok = true;
    const bool active = t < ntiles;
    // One block: false when a wait timed out (the CTA's abort flag is set).
    // `masked` (BoolTag<true>) for a block that reaches the tree keys or the
    // chunk's end: the ancestor mask and the key count apply.
    auto block_step = [&](int j, auto masked) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, abort_v))) return false;
      tc_fence_after();
      // The row's 128 scores: four loads in flight, one wait.
      float s[kBN];
      {
        uint32_t sr[kBN / 32][32];
#pragma unroll
        for (int q4 = 0; q4 < kBN / 32; ++q4) tmem_ld32_nowait(sbuf + 32 * q4, sr[q4]);
        tmem_wait_ld_tie32(sr[0]);
        reg_tie32(sr[1]);
        reg_tie32(sr[2]);
        reg_tie32(sr[3]);
#pragma unroll
        for (int e = 0; e < kBN; ++e) s[e] = __uint_as_float(sr[e >> 5][e & 31]);
      }
      const int key0 = k_begin + j * kBN;  // this block's first key
      if constexpr (decltype(masked)::value) {  // the block reaches the tree keys (or the end)
        // Keys key0 + e are visible iff e < k_end - key0 and they are prefix
        // keys or the row's node and its ancestors.
        const int lim = k_end - key0;  // 1 .. 128
        const uint64_t m0 = lim >= 64 ? ~0ull : ((1ull << lim) - 1ull);
        const uint64_t m1 = lim >= 128 ? ~0ull : (lim > 64 ? ((1ull << (lim - 64)) - 1ull) : 0ull);
        const uint64_t v0 = valid ? block_visibility(arow, key0 - P) & m0 : 0ull;
        const uint64_t v1 = (valid && lim > 64) ? block_visibility(arow, key0 + 64 - P) & m1 : 0ull;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          s[e] = ((v0 >> e) & 1ull) ? s[e] : -INFINITY;
          s[64 + e] = ((v1 >> e) & 1ull) ? s[64 + e] : -INFINITY;
        }
      }
      // Four independent chains of three-input maxima (two keys per step).
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int e = 4; e < kBN; e += 2) mx[(e >> 1) & 3] = fmax3(mx[(e >> 1) & 3], s[e], s[e + 1]);
      // Raw maximum times the (positive) scale = maximum of the scaled scores.
      const float hmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      // Move the reference only when a score exceeds it by more than the
      // threshold (always on the first visible block).
      float alpha = 1.f;
      if (hmax > m_ref + kRescaleThreshold) {
        alpha = fast_exp2(m_ref - hmax);  // 0 when m_ref = -inf
        m_ref = hmax;
      }
      l *= alpha;
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O_t must hold PV_t(j-1) before it is rescaled (lanes with alpha = 1
        // rewrite their row unchanged: TMEM loads and stores are warp-wide).
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[t], (j - 1) & 1, abort_v))) {
          return false;
        }
        tc_fence_after();
        // 16 columns at a time, so the scores can stay in registers meanwhile;
        // the wait for the P stores below also covers these stores.
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 16) {
          float o[16];
          tmem_ld16(o_mine + cc, o);
          uint32_t u[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(o[e] * alpha);
          tmem_st16u_nowait(o_mine + cc, u);
        }
      }
      const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;
      // Two keys per step: the exponent arguments by one paired FMA, the row
      // sums in four paired accumulators.
      const uint64_t sl2x2 = f2_pack(sl2, sl2), refx2 = f2_pack(neg_ref, neg_ref);
      uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {  // 32 keys -> 16 P columns at a time
        uint32_t h[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t x2 = ffma2(f2_pack(s[32 * hh + e], s[32 * hh + e + 1]), sl2x2, refx2);
          const float p0 = fast_exp2(f2_lo(x2));
          const float p1 = fast_exp2(f2_hi(x2));
          ps2[(e >> 1) & 3] = fadd2(ps2[(e >> 1) & 3], f2_pack(p0, p1));
          h[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16u_nowait(sbuf + 16 * hh, h);
      }
      tmem_wait_st();  // P is in TMEM before the arrival below
      const uint64_t pq = fadd2(fadd2(ps2[0], ps2[1]), fadd2(ps2[2], ps2[3]));
      l += f2_lo(pq) + f2_hi(pq);
      // V rows of the last block past the request's keys may hold anything
      // (even NaN): once the block has landed, tile 0 zeroes them before
      // either tile's PV reads the block (PV_1 follows PV_0), so that
      // 0 * garbage never reaches O.
      const int vrows = k_end - key0;
      if (t == 0 && vrows < kBN) {
        if (!__all_sync(0xffffffffu, mbar_wait(&v_full[j % SV], (j / SV) & 1, abort_v))) {
          return false;
        }
        uint8_t* vt = sV + (j % SV) * C::kTileBytes;
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
      mbar_arrive(&p_full[t]);
      return true;
    };
    // Blocks wholly inside the prefix take no mask: every row sees all their
    // keys (rows past the request compute on finite inputs in their own TMEM
    // lanes and are never stored).  The blocks from the first that reaches
    // the tree keys (or the end of the chunk) on apply it.
    const int jm = active ? min(nblk, max(0, (P - k_begin) / kBN)) : 0;
    for (int j = 0; ok && active && j < jm; ++j) ok = block_step(j, BoolTag<false>{});
    for (int j = jm; ok && active && j < nblk; ++j) ok = block_step(j, BoolTag<true>{});
    // The tile's last PV must be complete before the epilogue reads O_t.
    if (active && ok && nblk > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (nblk - 1) & 1, abort_v));
    // Agree on success CTA-wide: the merge below has barriers that all 256
    // softmax threads must reach.
    ok = !named_bar_or(kBarTcSoftmax, kTcSoftmaxThreads, active && !ok);
    if (clustered)  // a chunk of weight 0 (no keys, no success) is skipped by the merge
      sLse[t * kBM + r] = (ok && nblk > 0 && active && l > 0.f) ? m_ref + log2f(l) : -INFINITY;
    if (ok && nblk > 0) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const int node = grow / G;
      const int h = g * G + (grow - node * G);
      if (nch == 1) {
        if (active) {
          __nv_bfloat16* dst = out + ((size_t)(off + node) * plan.Hq + h) * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(o_mine + cc, o);
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
      } else if (clustered) {
        // Partial of this chunk, normalised, into this CTA's idle K/V rings:
        // row t * 128 + r of the pair; the cluster merges after the loop.
        if (active) {
          float* dst = reinterpret_cast<float*>(sK) + (size_t)(t * kBM + r) * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(o_mine + cc, o);
            float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(o[4 * e] * inv_l, o[4 * e + 1] * inv_l, o[4 * e + 2] * inv_l,
                                  o[4 * e + 3] * inv_l);
          }
        }
      } else {
        // Partial of this chunk, then the group's last CTA merges all chunks.
        const int64_t base0 = plan.part_row[b] + (int64_t)g * nch * R;
        if (active) {
          const int64_t prow_i = base0 + (int64_t)c * R + grow;
          float* dst = part_o + prow_i * D;
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            float o[32];
            tmem_ld32(o_mine + cc, o);
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
        int32_t* ctr = counters + plan.ctr_base[b] + g * mtiles + tp;
        if (tid == 0) *last_cta = atomicAdd(ctr, 1) == nch - 1;
        named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
        if (*last_cta) {
          __threadfence();
          // Merge, one tile at a time: first the chunk weights of every row
          // (the idle K/V rings hold them: [chunk][row] weights, then [row]
          // inverse sums), then rows x 4-column groups, four groups x four
          // chunks of loads in flight.
          float* sW = reinterpret_cast<float*>(sK);
          for (int tt = 0; tt < ntiles; ++tt) {
            const int trow0 = row0 + tt * kBM;
            const int trows = min(kBM, R - trow0);
            if (tid < trows) {
              const float* lse = part_lse + base0 + trow0 + tid;
              float M2 = -INFINITY;
#pragma unroll 8
              for (int cc = 0; cc < nch; ++cc) M2 = fmaxf(M2, __ldcg(lse + (int64_t)cc * R));
              float wsum = 0.f;
#pragma unroll 8
              for (int cc = 0; cc < nch; ++cc) {
                const float x = __ldcg(lse + (int64_t)cc * R);
                const float w = x == -INFINITY ? 0.f : fast_exp2(x - M2);
                sW[cc * kBM + tid] = w;
                wsum += w;
              }
              sW[64 * kBM + tid] = wsum > 0.f ? 1.f / wsum : 0.f;
            }
            named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
            constexpr int D4 = D / 4;
            const int items = trows * D4;
            const int64_t cstride = (int64_t)R * D;  // floats between chunks of a row
            for (int i0 = tid; i0 < items; i0 += 4 * kTcSoftmaxThreads) {
              float4 acc[4];
              int rr[4];
              const float* src[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = min(i0 + u * kTcSoftmaxThreads, items - 1);  // clamped: duplicates are harmless
                rr[u] = i / D4;
                src[u] = part_o + (base0 + trow0 + rr[u]) * D + (i - rr[u] * D4) * 4;
                acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
              for (int c0 = 0; c0 < nch; c0 += 4) {
                float4 v[4][4];
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2)
#pragma unroll
                  for (int u = 0; u < 4; ++u)
                    if (c0 + k2 < nch)
                      v[k2][u] = __ldcg(reinterpret_cast<const float4*>(src[u] + (c0 + k2) * cstride));
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2)
#pragma unroll
                  for (int u = 0; u < 4; ++u)
                    if (c0 + k2 < nch) {
                      const float w = sW[(c0 + k2) * kBM + rr[u]];
                      acc[u].x += w * v[k2][u].x;
                      acc[u].y += w * v[k2][u].y;
                      acc[u].z += w * v[k2][u].z;
                      acc[u].w += w * v[k2][u].w;
                    }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * kTcSoftmaxThreads;
                if (i >= items) break;
                const float inv = sW[64 * kBM + rr[u]];
                const int grr = trow0 + rr[u], nd = grr / G, hh = g * G + (grr - nd * G);
                __nv_bfloat16* o = out + ((size_t)(off + nd) * plan.Hq + hh) * D + (i - rr[u] * D4) * 4;
                *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc[u].x * inv, acc[u].y * inv),
                                                          pack_bf16x2(acc[u].z * inv, acc[u].w * inv));
              }
            }
            named_bar(kBarTcSoftmax, kTcSoftmaxThreads);  // sW is rewritten for the next tile
          }
          if (tid == 0) *ctr = 0;  // leave the counter zeroed for the next call
        }
      }
    }
  }

  // ---------------------------------------------------------------- cluster merge
  // Rank c merges rows [c * 256 / nch, (c + 1) * 256 / nch) of the pair: each
  // output item loads its row's log-sum-exps and its 16 bytes of every
  // chunk's partial from the cluster's shared memory in one round, then
  // weighs them (w = 2^(lse - max lse); a chunk of weight 0 is skipped).
  __syncwarp();
  if (clustered) {
    cluster_sync_all();  // every chunk's partial and log-sum-exps are in place
    if (warp < kTcSoftmaxThreads / 32) {
      const int npr = min(kTcTiles * kBM, R - row0);  // valid rows of the pair
      const int r_lo = (c * npr) / nch, r_hi = ((c + 1) * npr) / nch;
      constexpr int D4 = D / 4;
      const uint32_t part_s = smem_u32(sK);
      for (int i = tid; i < (r_hi - r_lo) * D4; i += kTcSoftmaxThreads) {
        const int pr = r_lo + i / D4, d4 = i % D4;
        float lse[8];
        float4 v[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          if (cc < nch) {
            lse[cc] = ld_dsmem_f32(mapa_shared(smem_u32(sLse + pr), (uint32_t)cc));
            v[cc] = ld_dsmem_f32x4(mapa_shared(part_s + (uint32_t)(pr * D + 4 * d4) * 4, (uint32_t)cc));
          }
        float M = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          if (cc < nch) M = fmaxf(M, lse[cc]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          if (cc < nch) {
            const float w = (M == -INFINITY || lse[cc] == -INFINITY) ? 0.f : fast_exp2(lse[cc] - M);
            if (w > 0.f) {
              acc.x += w * v[cc].x;
              acc.y += w * v[cc].y;
              acc.z += w * v[cc].z;
              acc.w += w * v[cc].w;
              wsum += w;
            }
          }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        const int grr = row0 + pr, nd = grr / G, hh = g * G + (grr - nd * G);
        __nv_bfloat16* o = out + ((size_t)(off + nd) * plan.Hq + hh) * D + 4 * d4;
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
      }
    }
    cluster_sync_all();  // every CTA keeps its shared memory until its peers have read it
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
    return launch_pdl(tree_attn_tc_kernel<64>, dim3(plan.n_units), dim3(kTcThreads), TcCfg<64>::kSmemBytes, st,
                      plan.cluster > 1 ? (unsigned)plan.cluster : 0u,
                      tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
  return launch_pdl(tree_attn_tc_kernel<128>, dim3(plan.n_units), dim3(kTcThreads), TcCfg<128>::kSmemBytes, st,
                    plan.cluster > 1 ? (unsigned)plan.cluster : 0u,
                    tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
}

}  // namespace tsv
