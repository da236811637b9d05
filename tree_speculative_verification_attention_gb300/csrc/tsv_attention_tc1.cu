// tsv_attention_tc1.cu — tree attention on the 5th-generation tensor cores,
// query rows on the TMEM lanes, one 128-row query tile per CTA.  Used when no
// request has more than 128 query rows per KV head: one tile per (request, KV
// head), so the tile-pair kernel would leave half its softmax warps idle;
// here both warp groups serve the one tile, each taking half of every key
// block.
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
// head g sit in the same tiles, so each streamed K/V row serves every tree
// node and every grouped head at once.  Keys go in blocks of 128, so both
// MMAs of a block have N >= 128 (smaller N runs the tensor pipe below its
// rate).  Warp roles (320 threads):
//   warp 8        TMA producer.  Lane 0: the Q tile, then K blocks into a
//                 3-stage ring, each released as soon as S has read it; lane
//                 1: V blocks into a 2-stage ring, released after PV.
//   warp 9        tcgen05 issuer and TMEM owner (S0 | S1 | O0 | O1): S(j+1) =
//                 Q K^T is issued before PV(j), so the next scores are ready
//                 when the softmax of a block ends; O_h += P_h V_h reads P_h
//                 from TMEM, one accumulator per key half.
//   warps 0-7     softmax.  Warp w serves the rows on TMEM lanes 32(w%4).. and
//                 key half h = w/4 (64 keys) of every block.  The two halves
//                 of a row are independent online softmaxes (own reference
//                 maximum, row sum and O accumulator), so no barrier is needed
//                 inside the loop; they are combined once at the end.  Set-up:
//                 the ancestor bitset of the row's node (prepared, or by
//                 walking parent[] up to the root).  Loop: read S, mask the
//                 tree part of the keys with the bitset, base-2 softmax with a
//                 lazily moved reference maximum, P in bf16 written back over
//                 the thread's own S columns, O_h rescaled in TMEM when the
//                 reference moves.  End: combine the halves, normalise and
//                 store; when a request's keys are split over several CTAs,
//                 store a partial + log2-sum-exp and let the last CTA of the
//                 group (atomic counter, no waiting) merge the partials.
#include <cuda_bf16.h>
#include <math.h>

#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kTcSoftmaxThreads = 256;
constexpr int kTcThreads = kTcSoftmaxThreads + 64;
constexpr int kTcProducerWarp = 8, kTcMmaWarp = 9;
constexpr int kHalfKeys = kBN / 2;         // keys of a block per softmax thread
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8 between rescales
constexpr int kBarTcSetup = 1;             // softmax warps + MMA warp
constexpr int kBarTcSoftmax = 2;           // softmax warps

template <int D>
struct Tc1Cfg {
  static constexpr int kHalves = D / 64;      // 128-byte column groups per row
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kTileBytes = kBN * D * 2;  // one K (or V) block
  static constexpr int kAncWords = TSV_ANC_WORDS + 2;  // two zero words past the end
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffAnc = kOffV + kVStages * kTileBytes;
  static constexpr int kOffPar = kOffAnc + kBM * kAncWords * 4;
  static constexpr int kOffX = kOffPar + TSV_MAX_NODES * 4;  // float [4][128]: per-half row values
  static constexpr int kOffBar = kOffX + 4 * kBM * 4;
  // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2],
  // p_full[half][2], pv_done[half][2], mma_done
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 4 + 4 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kColO = 2 * kBN;               // S0 | S1 | O0 | O1 (D columns each)
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kTileBytes % 1024 == 0, "swizzle atoms");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kColO + 2 * D <= kTmemCols, "TMEM columns");
  static_assert(kKStages * kTileBytes >= (64 + 1) * kBM * 4, "merge weights fit in the K ring");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    tree_attn_tc1_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ AttnPlan plan, const int32_t* __restrict__ parent,
                        const uint32_t* __restrict__ anc, __nv_bfloat16* __restrict__ out,
                        float* __restrict__ part_o, float* __restrict__ part_lse,
                        int32_t* __restrict__ counters, int32_t* __restrict__ status) {
  using C = Tc1Cfg<D>;
  constexpr int SK = C::kKStages, SV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + C::kOffAnc);
  int32_t* sPar = reinterpret_cast<int32_t*>(smem + C::kOffPar);
  float* sX = reinterpret_cast<float*>(smem + C::kOffX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;
  uint64_t* p_full = s_full + 2;   // [half][2]
  uint64_t* pv_done = p_full + 4;  // [half][2]
  uint64_t* mma_done = pv_done + 4;
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
  const int b = plan.slot_req[lo];
  const int local = unit - plan.unit_start[lo];
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
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) mbar_init(&s_full[x], 1);
    for (int x = 0; x < 4; ++x) {
      mbar_init(&p_full[x], kTcSoftmaxThreads / 2);  // every thread of the key half
      mbar_init(&pv_done[x], 1);
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
    const uint64_t pol = mtiles > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      // Q tile: box (64 d, G heads, 128/G nodes) lands as 128 rows r = node*G + head.
      mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(sQ + hf * (kBM * 128), &tmap_q, q_full, hf * 64, g * G, off + row0 / G,
                    l2_policy_evict_first());
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
      auto issue_s = [&](int j) {
        const uint32_t dst = tmem + (uint32_t)((j & 1) * kBN);
        const uint64_t db = dk + (uint64_t)(((j % SK) * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = ((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4;
          const uint32_t bo = ((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4;
          umma_bf16(dst, dq + ao, db + bo, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        umma_commit(&k_empty[j % SK]);  // K(j) is free once S(j) has read it
      };
      auto issue_pv = [&](int h, int j) {
        // P_h sits over the first 32 of key half h's 64 S columns; V_h is rows
        // 64h .. 64h+63 of the V block.
        const uint32_t pa = tmem + (uint32_t)((j & 1) * kBN + h * kHalfKeys);
        const uint64_t db = dv + (uint64_t)(((j % SV) * C::kTileBytes + h * kHalfKeys * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHalfKeys / 16; ++kk)
          umma_bf16_ts(tmem + C::kColO + h * D, pa + kk * 8, db + (uint32_t)((kk * 16 * 128) >> 4), idPV,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[2 * h + (j & 1)]);
      };
      bool ok = nblk > 0 && mbar_wait(q_full, 0, abort_v) && mbar_wait(&k_full[0], 0, abort_v);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + 1 < nblk) {
          if (!mbar_wait(&k_full[(j + 1) % SK], ((j + 1) / SK) & 1, abort_v)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!mbar_wait(&v_full[j % SV], (j / SV) & 1, abort_v)) break;
        for (int h = 0; ok && h < 2; ++h) {
          if (!mbar_wait(&p_full[2 * h + (j & 1)], (j >> 1) & 1, abort_v)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(h, j);
        }
        if (ok) umma_commit(&v_empty[j % SV]);
      }
      umma_commit(mma_done);  // every MMA of this CTA has finished before TMEM is freed
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int hk = warp >> 2;       // key half of every block
    const int r = tid & (kBM - 1);  // row = TMEM lane
    const bool valid = r < rows_valid;
    // Ancestor bitset of this row's node (built by the half-0 thread of the row).
    uint32_t* arow = sAnc + r * C::kAncWords;
    if (hk == 0) {
#pragma unroll
      for (int w = 0; w < C::kAncWords; ++w) arow[w] = 0u;
    }
    if (anc != nullptr) {
      if (valid && hk == 0) {
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
      if (valid && hk == 0 && !bad)
        for (int a = (row0 + r) / G; a >= 0; a = sPar[a]) arow[a >> 5] |= 1u << (a & 31);
    }
    tc_fence_before();
    named_bar(kBarTcSetup, kTcSoftmaxThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t o_mine = trow + C::kColO + (uint32_t)(hk * D);  // O_h of this row
    uint64_t* p_mine = p_full + 2 * hk;
    uint64_t* pv_mine = pv_done + 2 * hk;
    const float sl2 = plan.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    // No barrier inside the loop: a timed-out wait ends this warp's loop
    // (every wait is bounded and sets the CTA's abort flag, so the other
    // warps' waits end quickly too); the CTA agrees after the loop.
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_v))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbuf = trow + (uint32_t)((j & 1) * kBN + hk * kHalfKeys);
      float s[kHalfKeys];
      tmem_ld32(sbuf, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld32(sbuf + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      const int key0 = k_begin + j * kBN + hk * kHalfKeys;  // this half's first key
      if (key0 + kHalfKeys > P) {  // uniform per warp: the half reaches the tree keys (or the end)
        // Visible: keys before the chunk end that are prefix keys or the
        // row's node and its ancestors.
        const int lim = k_end - key0;
        const uint64_t vis = (valid && lim > 0)
                                 ? block_visibility(arow, key0 - P) & (lim >= 64 ? ~0ull : ((1ull << lim) - 1ull))
                                 : 0ull;
#pragma unroll
        for (int e = 0; e < kHalfKeys; ++e) s[e] = ((vis >> e) & 1ull) ? s[e] : -INFINITY;
      } else if (!valid) {
#pragma unroll
        for (int e = 0; e < kHalfKeys; ++e) s[e] = -INFINITY;
      }
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int e = 4; e < kHalfKeys; ++e) mx[e & 3] = fmaxf(mx[e & 3], s[e]);
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
        // O_h must hold PV_h(j-1) before it is rescaled (lanes with alpha = 1
        // rewrite their row unchanged: TMEM loads and stores are warp-wide).
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_mine[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_v))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(o_mine + cc, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(o_mine + cc, o);
        }
      }
      const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;
      uint32_t h0[16], h1[16];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < kHalfKeys; e += 2) {
        const float p0 = fast_exp2(fmaf(s[e], sl2, neg_ref));
        const float p1 = fast_exp2(fmaf(s[e + 1], sl2, neg_ref));
        ps[(e >> 1) & 3] += p0 + p1;
        if (e < 32) h0[e >> 1] = pack_bf16x2(p0, p1);
        else h1[(e - 32) >> 1] = pack_bf16x2(p0, p1);
      }
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      // P (bf16, two per column) over the first 32 of this thread's 64 S columns.
      tmem_st16u(sbuf, h0);
      tmem_st16u(sbuf + 16, h1);
      // V rows of the last block past the request's keys may hold anything
      // (even NaN): once the block has landed, each half zeroes the rows its
      // own PV reads, so that 0 * garbage never reaches O.
      const int vrows = k_end - (k_begin + j * kBN);
      if (vrows < kBN) {
        const int first = max(vrows, hk * kHalfKeys), last = (hk + 1) * kHalfKeys;
        if (first < last) {
          if (!__all_sync(0xffffffffu, mbar_wait(&v_full[j % SV], (j / SV) & 1, abort_v))) {
            ok = false;
            break;
          }
          uint8_t* vt = sV + (j % SV) * C::kTileBytes;
          const int pieces = (last - first) * C::kHalves * 8;
          for (int q = r; q < pieces; q += kBM) {
            const int row = first + q / (C::kHalves * 8);
            const int rem = q % (C::kHalves * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * (kBN * 128) + row * 128 + ((rem & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
      }
      tc_fence_before();
      mbar_arrive(&p_mine[j & 1]);
    }
    // Both halves' last PV must be complete before the epilogue reads O0 and O1.
    if (ok && nblk > 0) {
      const int jl = nblk - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[jl & 1], (jl >> 1) & 1, abort_v) &&
                                       mbar_wait(&pv_done[2 + (jl & 1)], (jl >> 1) & 1, abort_v));
    }
    // Agree on success CTA-wide: the epilogue has barriers that all 256
    // softmax threads must reach.
    ok = !named_bar_or(kBarTcSoftmax, kTcSoftmaxThreads, !ok);
    if (ok && nblk > 0) {
      tc_fence_after();
      // Combine the halves of each row: weights 2^(m_h - M), sum L (the same
      // order in both threads of a row).
      sX[hk * kBM + r] = m_ref;
      sX[(2 + hk) * kBM + r] = l;
      named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
      const float m0 = sX[r], m1 = sX[kBM + r];
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M);
      const float w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
      const float L = w0 * sX[2 * kBM + r] + w1 * sX[3 * kBM + r];
      const float inv_l = L > 0.f ? 1.f / L : 0.f;
      const float c0 = w0 * inv_l, c1 = w1 * inv_l;
      const int gr = row0 + r;
      const int node = gr / G;
      const int h = g * G + (gr - node * G);
      constexpr int kOHalf = D / 2;  // output columns this thread writes
      const uint32_t oc0 = trow + C::kColO + (uint32_t)(hk * kOHalf);
      if (nch == 1) {
        __nv_bfloat16* dst = out + ((size_t)(off + node) * plan.Hq + h) * D + hk * kOHalf;
#pragma unroll 1
        for (int cc = 0; cc < kOHalf; cc += 32) {
          float o[32], o1[32];
          tmem_ld32(oc0 + cc, o);
          tmem_ld32(oc0 + D + cc, o1);
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float v[8];
#pragma unroll
              for (int x = 0; x < 8; ++x) v[x] = c0 * o[8 * e + x] + c1 * o1[8 * e + x];
              d4[e] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                 pack_bf16x2(v[6], v[7]));
            }
          }
        }
      } else {
        // Partial of this chunk, then the group's last CTA merges all chunks.
        const int64_t base0 = plan.part_row[b] + (int64_t)g * nch * R;
        const int64_t prow_i = base0 + (int64_t)c * R + gr;
        float* dst = part_o + prow_i * D + hk * kOHalf;
#pragma unroll 1
        for (int cc = 0; cc < kOHalf; cc += 32) {
          float o[32], o1[32];
          tmem_ld32(oc0 + cc, o);
          tmem_ld32(oc0 + D + cc, o1);
          if (valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(c0 * o[4 * e] + c1 * o1[4 * e], c0 * o[4 * e + 1] + c1 * o1[4 * e + 1],
                                  c0 * o[4 * e + 2] + c1 * o1[4 * e + 2], c0 * o[4 * e + 3] + c1 * o1[4 * e + 3]);
          }
        }
        if (valid && hk == 0) part_lse[prow_i] = L > 0.f ? M + log2f(L) : -INFINITY;
        __threadfence();
        named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
        int32_t* ctr = counters + plan.ctr_base[b] + g * mtiles + mt;
        if (tid == 0) *last_cta = atomicAdd(ctr, 1) == nch - 1;
        named_bar(kBarTcSoftmax, kTcSoftmaxThreads);
        if (*last_cta) {
          __threadfence();
          // Merge: first the chunk weights of every row (the idle K ring holds
          // them: [chunk][row] weights, then [row] inverse sums), then rows x
          // 4-column groups, four groups x four chunks of loads in flight.
          float* sW = reinterpret_cast<float*>(sK);
          if (tid < rows_valid) {
            const float* lse = part_lse + base0 + row0 + tid;
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
          const int items = rows_valid * D4;
          const int64_t cstride = (int64_t)R * D;  // floats between chunks of a row
          for (int i0 = tid; i0 < items; i0 += 4 * kTcSoftmaxThreads) {
            float4 acc[4];
            int rr[4];
            const float* src[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = min(i0 + u * kTcSoftmaxThreads, items - 1);  // clamped: duplicates are harmless
              rr[u] = i / D4;
              src[u] = part_o + (base0 + row0 + rr[u]) * D + (i - rr[u] * D4) * 4;
              acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int c0 = 0; c0 < nch; c0 += 4) {
              float4 v[4][4];
#pragma unroll
              for (int k2 = 0; k2 < 4; ++k2)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (c0 + k2 < nch) v[k2][u] = __ldcg(reinterpret_cast<const float4*>(src[u] + (c0 + k2) * cstride));
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
              const int grr = row0 + rr[u], nd = grr / G, hh = g * G + (grr - nd * G);
              __nv_bfloat16* o = out + ((size_t)(off + nd) * plan.Hq + hh) * D + (i - rr[u] * D4) * 4;
              *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc[u].x * inv, acc[u].y * inv),
                                                        pack_bf16x2(acc[u].z * inv, acc[u].w * inv));
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

size_t attention_tc1_smem_bytes(int D) {
  return D == 64 ? (size_t)Tc1Cfg<64>::kSmemBytes : (size_t)Tc1Cfg<128>::kSmemBytes;
}

cudaError_t attention_tc1_set_attributes(int D) {
  if (D == 64)
    return cudaFuncSetAttribute(tree_attn_tc1_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Tc1Cfg<64>::kSmemBytes);
  return cudaFuncSetAttribute(tree_attn_tc1_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Tc1Cfg<128>::kSmemBytes);
}

cudaError_t launch_attention_tc1(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                const CUtensorMap& tmap_v, const AttnPlan& plan,
                                const int32_t* parent, const uint32_t* anc, void* out,
                                float* part_o, float* part_lse, int32_t* counters,
                                int32_t* status, cudaStream_t st) {
  if (plan.n_units == 0) return cudaSuccess;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  if (plan.D == 64)
    return launch_pdl(tree_attn_tc1_kernel<64>, dim3(plan.n_units), dim3(kTcThreads), Tc1Cfg<64>::kSmemBytes, st, 0u,
                      tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
  return launch_pdl(tree_attn_tc1_kernel<128>, dim3(plan.n_units), dim3(kTcThreads), Tc1Cfg<128>::kSmemBytes, st, 0u,
                    tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, part_o, part_lse, counters, status);
}

}  // namespace tsv
