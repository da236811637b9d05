// tsv_attention_keys.cu — tree attention for small trees, keys on the TMEM lanes.
//
// Same result as the rows-on-lanes kernel (SpecInfer §4 "Tree Attention" and
// "Tree-Based Parallel Decoding"; the key range split into chunks merged by
// log-sum-exp as in Staged Speculative Decoding §3), laid out for the common
// verification case where a request's tree, times the query heads sharing one
// KV head, is at most 64 query rows.  The 128 keys of a block sit on the TMEM
// lanes and the query rows on the columns, so every thread owns one key and
// computes exponentials only for the rows that exist:
//
//   S^T = K Q^T      M = 128 keys, N = 64 rows, K = D          (A = K tile, B = Q tile)
//   O^T += V^T P^T   M = 128 (d), N = 64 rows, K = 128 keys    (A = V tile, M-major)
//   L^T += 1 P^T     M = 128,     N = 64 rows, K = 128 keys    (row sums on the tensor core)
//
// Eight key-lane warps: warps w and w+4 share TMEM lanes 32(w%4).. and split
// every 16-row column group into two halves of 8 rows.  Rows beyond the tree
// carry a reference maximum of +inf, so their probabilities are zero without
// any per-element test; only blocks that reach the tree part of the keys
// apply the ancestor mask, built once per CTA from parent[] (loaded at entry)
// as "rows that see tree key j" bit masks.  A row's reference maximum moves
// only when a visible score exceeds it by more than 2^32 (always on its first
// visible block): one OR-reducing named barrier per block decides, and the
// rare move is a warp-shuffle maximum plus a rescale of O^T and L^T in TMEM.
//
// When a request's keys are split into K chunks (K <= 8), the K CTAs of a
// chunk group form one cluster: each leaves its normalised partial and
// log2-sum-exp in its own shared memory, and CTA rank c merges the c-th
// share of the rows through distributed shared memory (weights first, then
// 16-byte loads kept in flight together) — no global partials, no atomics,
// no second kernel.
//
// Warp roles (320 threads): warps 0-7 key lanes (softmax, P^T, epilogue),
// warp 8 TMA producer (Q tile, then K/V blocks of 128 keys into a 3-stage
// ring), warp 9 tcgen05 issuer and TMEM owner.  P^T of a block is written
// over that block's K tile, which S^T has finished reading, so the ring
// needs no separate P buffers and three 64 KB stages fit next to Q.
#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kKeysLaneThreads = 256;
constexpr int kKeysThreads = kKeysLaneThreads + 64;
constexpr int kKeysProducerWarp = 8, kKeysMmaWarp = 9;
constexpr int kKeysBlock = kKeysBlockKeys;   // keys per block (MMA M)
constexpr int kKeysRows = kKeysTileRows;     // query rows per CTA (MMA N)
constexpr int kKeysMaxTree = kKeysTileRows;  // n * G <= 64 implies n <= 64
constexpr float kKeysOverflow = 32.f;        // log2 units
constexpr int kBarKeysSetup = 1;             // key lanes + MMA warp
constexpr int kBarKeys = 2;                  // key lanes

template <int D>
struct KeysCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = 3;
  static constexpr int kQBytes = kKeysRows * D * 2;
  static constexpr int kKTile = kKeysBlock * D * 2;
  static constexpr int kVTile = kKeysBlock * 128 * 2;  // always 128 d: upper half zero when D = 64
  static constexpr int kStageBytes = kKTile + kVTile;
  static constexpr int kPBytes = kKeysBlock * kKeysRows * 2;  // P^T, written over the K tile
  static constexpr int kOnesBytes = 1024;  // one 8-row atom of bf16 ones, read by every row group
  static constexpr int kOffQ = 0;
  static constexpr int kOffStage = kOffQ + kQBytes;
  static constexpr int kOffOnes = kOffStage + kStages * kStageBytes;
  static constexpr int kOffDesc = kOffOnes + kOnesBytes;        // uint32 [64][2]
  static constexpr int kOffPar = kOffDesc + kKeysMaxTree * 8;   // int32 [64]
  static constexpr int kOffMref = kOffPar + kKeysMaxTree * 4;   // float [64]
  static constexpr int kOffAlpha = kOffMref + kKeysRows * 4;    // float [64]
  static constexpr int kOffWmax = kOffAlpha + kKeysRows * 4;    // float [4][64]
  static constexpr int kOffLse = kOffWmax + 4 * kKeysRows * 4;  // float [64]
  static constexpr int kOffWts = kOffLse + kKeysRows * 4;       // float [8][64] (spare)
  static constexpr int kOffBar = kOffWts + 8 * kKeysRows * 4;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done[2], mma_done
  static constexpr int kNumBars = 1 + 2 * kStages + 7;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 32 + 1024;
  static constexpr uint32_t kTmemCols = 256;  // S0 | S1 | O^T | L^T, 64 columns each
  static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0 && kOffOnes % 1024 == 0, "atoms");
  static_assert(kPBytes <= kKTile, "P^T fits in the K tile it replaces");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kKeysRows * D * 4 <= kStageBytes, "partial fits in a stage");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(kKeysThreads, 1)
    tree_attn_keys_kernel(const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v,
                          const __grid_constant__ AttnPlan plan, const int32_t* __restrict__ parent,
                          const uint32_t* __restrict__ anc, __nv_bfloat16* __restrict__ out,
                          int32_t* __restrict__ status) {
  using C = KeysCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sStage = smem + C::kOffStage;
  uint8_t* sOnes = smem + C::kOffOnes;
  uint32_t* sDesc = reinterpret_cast<uint32_t*>(smem + C::kOffDesc);
  int32_t* sPar = reinterpret_cast<int32_t*>(smem + C::kOffPar);
  float* sMref = reinterpret_cast<float*>(smem + C::kOffMref);
  float* sAlpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
  float* sWmax = reinterpret_cast<float*>(smem + C::kOffWmax);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
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
  int* req_slot = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  int* fail_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 12);
  volatile int* abort_v = abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- the unit
  const int unit = blockIdx.x;
  if (tid < plan.B && plan.unit_start[tid] <= unit && unit < plan.unit_start[tid + 1]) *req_slot = tid;
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], kKeysLaneThreads);
      mbar_init(&pv_done[x], 1);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    *fail_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const int b = plan.slot_req[*req_slot];
  const int local = unit - plan.unit_start[*req_slot];
  const int nch = plan.n_chunks[b];  // == cluster size
  const int mtiles = plan.mtiles[b];
  const int c = local % nch;
  const int gm = local / nch;
  const int mt = gm % mtiles;
  const int g = gm / mtiles;
  const int G = plan.G;
  const int P = plan.prefix[b], n = plan.nodes[b], off = plan.node_off[b];
  const int R = n * G;
  const int row0 = mt * kKeysRows;
  const int rows_valid = min(kKeysRows, R - row0);
  const int ngrp = (rows_valid + 15) >> 4;  // 16-row column groups holding valid rows
  const int clen = plan.chunk_len[b];
  const int k_begin = min(P + n, c * clen);
  const int k_end = min(P + n, k_begin + clen);
  const int nblk = (k_end - k_begin + kKeysBlock - 1) / kKeysBlock;
  // The unit comes from the plan alone, so when all units run in the first
  // wave the first ring's worth of K/V is pulled into L2 while the previous
  // kernel finishes.
  if (plan.prefetch_l2 && warp == kKeysProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    for (int j = 0; j < nblk && j < C::kStages; ++j)
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tma_prefetch_4d(&tmap_k, hf * 64, g, k_begin + j * kKeysBlock, b);
        tma_prefetch_4d(&tmap_v, hf * 64, g, k_begin + j * kKeysBlock, b);
      }
  }
  pdl_wait();  // the previous kernel's results are visible from here on

  if (warp == kKeysProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      const uint64_t pol = mtiles > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
      if (nblk > 0) {
        mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(sQ + hf * (kKeysRows * 128), &tmap_q, q_full, hf * 64, g * G, off + row0 / G, pol);
      }
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % S;
        if (j >= S && !mbar_wait(&kv_empty[st], ((j / S) - 1) & 1, abort_v)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kHalves * kKeysBlock * 128);
        const int key0 = k_begin + j * kKeysBlock;
        uint8_t* kt = sStage + st * C::kStageBytes;
        uint8_t* vt = kt + C::kKTile;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_4d(kt + hf * (kKeysBlock * 128), &tmap_k, &kv_full[st], hf * 64, g, key0, b, pol);
          tma_load_4d(vt + hf * (kKeysBlock * 128), &tmap_v, &kv_full[st], hf * 64, g, key0, b, pol);
        }
        ++issued;
      }
      if (*abort_v) {
        if (nblk > 0) mbar_wait(q_full, 0, nullptr);
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait(&kv_full[j % S], (j / S) & 1, nullptr);
      }
    }
  } else if (warp == kKeysMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
    named_bar(kBarKeysSetup, kKeysLaneThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32_ab(kKeysBlock, kKeysRows, 0, 0);
      constexpr uint32_t idO = idesc_bf16_f32_ab(128, kKeysRows, 1, 1);
      constexpr uint32_t idL = idesc_bf16_f32_ab(128, kKeysRows, 0, 1);
      const uint32_t tO = tmem + 2 * kKeysRows, tL = tmem + 3 * kKeysRows;
      const uint32_t qa = smem_u32(sQ), sa = smem_u32(sStage), oa = smem_u32(sOnes);
      auto issue_s = [&](int j) {
        const uint32_t ka = sa + (uint32_t)((j % S) * C::kStageBytes);
        const uint32_t dst = tmem + (uint32_t)((j & 1) * kKeysRows);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * (kKeysBlock * 128) + (kk & 3) * 32;
          const uint32_t bo = (kk >> 2) * (kKeysRows * 128) + (kk & 3) * 32;
          umma_bf16(dst, sdesc_sw128(ka + ao, 16, 1024), sdesc_sw128(qa + bo, 16, 1024), idS,
                    kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int j) {
        const uint32_t pb = sa + (uint32_t)((j % S) * C::kStageBytes);  // P^T over K(j)
        const uint32_t va = pb + (uint32_t)C::kKTile;
#pragma unroll
        for (int kk = 0; kk < kKeysBlock / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(pb + kk * 2048, kKeysBlock * 128, 1024);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          umma_bf16(tO, sdesc_sw128(va + kk * 2048, kKeysBlock * 128, 1024), bdesc, idO, acc);
          // Row-group stride 0: all 16 groups of 8 rows read the same atom of ones.
          umma_bf16(tL, sdesc_sw128(oa + (kk & 3) * 32, 16, 0), bdesc, idL, acc);
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
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ key-lane threads
    const int t = tid;              // 0 .. 255
    const int lg = warp & 3;        // TMEM lane group
    const int kl = lg * 32 + lane;  // key lane (and d for O^T)
    const int h = warp >> 2;        // which 8 of every 16 rows
    const uint32_t lane_base = (uint32_t)(lg * 32) << 16;
    // Tree of the request: parent[] (n <= 64) or the prepared ancestor words.
    int my_par = -1;
    uint32_t my_anc0 = 0u, my_anc1 = 0u;
    if (anc == nullptr) {
      if (t < n) my_par = __ldg(parent + off + t);
    } else if (t < rows_valid) {
      const uint2 a2 = __ldg(reinterpret_cast<const uint2*>(anc + (size_t)(off + (row0 + t) / G) * TSV_ANC_WORDS));
      my_anc0 = a2.x;
      my_anc1 = a2.y;
    }
    if (t < kKeysRows) {
      sMref[t] = t < rows_valid ? -INFINITY : INFINITY;  // rows past the tree never see a key
      sAlpha[t] = 1.f;
    }
    {
      const uint32_t one2 = 0x3F803F80u;  // two bf16 1.0
      const uint4 o4 = make_uint4(one2, one2, one2, one2);
      for (int i = t; i < C::kOnesBytes / 16; i += kKeysLaneThreads) reinterpret_cast<uint4*>(sOnes)[i] = o4;
      if (D == 64) {  // the upper half of every V stage stays zero
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int st = 0; st < S; ++st) {
          uint4* vh = reinterpret_cast<uint4*>(sStage + st * C::kStageBytes + C::kKTile + kKeysBlock * 128);
          for (int i = t; i < kKeysBlock * 128 / 16; i += kKeysLaneThreads) vh[i] = z;
        }
      }
    }
    if (anc == nullptr && t < n) sPar[t] = my_par;
    const bool bad = named_bar_or(kBarKeys, kKeysLaneThreads,
                                  anc == nullptr && t < n && (my_par < -1 || my_par >= t));
    if (anc == nullptr && local == 0 && t == 0) status[b] = bad ? TSV_ERR_BAD_TREE : TSV_OK;
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(kBarKeysSetup, kKeysLaneThreads + 32);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + lane_base + 2 * kKeysRows, tL = tmem + lane_base + 3 * kKeysRows;
    const float sl2 = plan.scale_log2;
    bool desc_ready = false;
    // A failed (timed-out) wait is made CTA-wide before anyone leaves the loop,
    // so every named barrier below is reached by all key-lane threads.
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int key0 = k_begin + j * kKeysBlock;
      const bool tail_block = key0 + kKeysBlock > P;  // uniform: the block reaches tree keys
      if (tail_block && !desc_ready) {
        // desc[jt] bit r <=> tree node jt is row r's node or one of its ancestors.
        if (t < 2 * kKeysMaxTree) sDesc[t] = 0u;
        named_bar(kBarKeys, kKeysLaneThreads);
        if (t < rows_valid && !bad) {
          const uint32_t rb = 1u << (t & 31);
          uint32_t* word = sDesc + (t >> 5);  // word (t>>5) of each 2-word row mask
          if (anc == nullptr) {
            for (int a = (row0 + t) / G; a >= 0; a = sPar[a]) atomicOr(word + 2 * a, rb);
          } else {
            for (uint32_t m = my_anc0; m; m &= m - 1) atomicOr(word + 2 * (__ffs(m) - 1), rb);
            for (uint32_t m = my_anc1; m; m &= m - 1) atomicOr(word + 2 * (32 + __ffs(m) - 1), rb);
          }
        }
        named_bar(kBarKeys, kKeysLaneThreads);
        desc_ready = true;
      }
      const bool okj = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_v));
      tc_fence_after();
      const int key = key0 + kl;
      const bool full_vis = key < P;
      uint64_t vis = 0ull;  // used only when !full_vis
      if (!full_vis && key < k_end)
        vis = (uint64_t)sDesc[2 * (key - P)] | ((uint64_t)sDesc[2 * (key - P) + 1] << 32);
      const uint32_t s_col = tmem + lane_base + (uint32_t)((j & 1) * kKeysRows);
      // The first block always moves the maxima (they start at -inf): skip the test.
      float over = j == 0 ? INFINITY : -INFINITY;
#pragma unroll 1
      for (int g16 = 0; j > 0 && g16 < ngrp; ++g16) {
        const int c0 = g16 * 16 + h * 8;
        float sv[8];
        tmem_ld8(s_col + c0, sv);
        const float4 ma = *reinterpret_cast<const float4*>(sMref + c0);
        const float4 mb = *reinterpret_cast<const float4*>(sMref + c0 + 4);
        const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        const uint32_t vm = full_vis ? 0xFFu : (uint32_t)(vis >> c0) & 0xFFu;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = fmaf(sv[e], sl2, -m[e]);
          over = fmaxf(over, ((vm >> e) & 1u) ? x : -INFINITY);
        }
      }
      if (!okj) *fail_flag = 1;
      const bool any_over = named_bar_or(kBarKeys, kKeysLaneThreads, over > kKeysOverflow || !okj);
      if (*fail_flag) {
        ok = false;
        break;
      }
      if (any_over) {
        // Move the reference maxima: per-row max over this block's visible keys.
        // Transposed warp reduction: each xor step halves the values a lane
        // keeps, so 8 rows x 32 lanes take 4 + 2 + 1 + 2 shuffles, after which
        // lane l holds the maximum of row c0 + ((l >> 2) & 7).
#pragma unroll 1
        for (int g16 = 0; g16 < ngrp; ++g16) {
          const int c0 = g16 * 16 + h * 8;
          float sv[8];
          tmem_ld8(s_col + c0, sv);
          const uint32_t vm = full_vis ? 0xFFu : (uint32_t)(vis >> c0) & 0xFFu;
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = ((vm >> e) & 1u) ? sv[e] * sl2 : -INFINITY;
          const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
          float w4[4], w2[2];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w4[i] = fmaxf(b4 ? v[i + 4] : v[i], __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 4], 16));
#pragma unroll
          for (int i = 0; i < 2; ++i)
            w2[i] = fmaxf(b3 ? w4[i + 2] : w4[i], __shfl_xor_sync(0xffffffffu, b3 ? w4[i] : w4[i + 2], 8));
          float w1 = fmaxf(b2 ? w2[1] : w2[0], __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4));
          w1 = fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, 2));
          w1 = fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, 1));
          if ((lane & 3) == 0) sWmax[lg * kKeysRows + c0 + (lane >> 2)] = w1;
        }
        named_bar(kBarKeys, kKeysLaneThreads);
        if (t < rows_valid) {
          const float m_old = sMref[t];
          const float bm = fmaxf(fmaxf(sWmax[t], sWmax[kKeysRows + t]),
                                 fmaxf(sWmax[2 * kKeysRows + t], sWmax[3 * kKeysRows + t]));
          const float m_new = fmaxf(m_old, bm);
          sAlpha[t] = m_new == -INFINITY ? 1.f : fast_exp2(m_old - m_new);
          sMref[t] = m_new;
        }
        named_bar(kBarKeys, kKeysLaneThreads);
        if (j > 0) {  // O^T and L^T hold PV(0..j-1): rescale this thread's columns
          if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_v)))
            *fail_flag = 1;  // seen by everyone at the next block's barrier
          tc_fence_after();
#pragma unroll 1
          for (int g16 = 0; g16 < ngrp; ++g16) {
            const int c0 = g16 * 16 + h * 8;
            float o[8], l8[8];
            tmem_ld8(tO + c0, o);
            tmem_ld8(tL + c0, l8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a = sAlpha[c0 + e];
              o[e] *= a;
              l8[e] *= a;
            }
            tmem_st8(tO + c0, o);
            tmem_st8(tL + c0, l8);
          }
        }
      }
      // P^T goes over the K tile of this block: S^T(j) has finished reading it.
      uint8_t* prow = sStage + (j % S) * C::kStageBytes + kl * 128;
#pragma unroll 1
      for (int g16 = 0; g16 < ngrp; ++g16) {
        const int c0 = g16 * 16 + h * 8;
        float sv[8];
        tmem_ld8(s_col + c0, sv);
        const float4 ma = *reinterpret_cast<const float4*>(sMref + c0);
        const float4 mb = *reinterpret_cast<const float4*>(sMref + c0 + 4);
        const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        const uint32_t vm = full_vis ? 0xFFu : (uint32_t)(vis >> c0) & 0xFFu;
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = fast_exp2(((vm >> e) & 1u) ? fmaf(sv[e], sl2, -m[e]) : -INFINITY);
        const int chunk = 2 * g16 + h;
        *reinterpret_cast<uint4*>(prow + ((chunk ^ (kl & 7)) << 4)) =
            make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                       pack_bf16x2(p[6], p[7]));
      }
      // A V row past the request's keys may hold anything (even NaN): zero it.
      if (key >= k_end && h < C::kHalves) {
        uint4* vrow = reinterpret_cast<uint4*>(sStage + (j % S) * C::kStageBytes + C::kKTile +
                                               h * (kKeysBlock * 128) + kl * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) vrow[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (ok && nblk > 0 &&
        !__all_sync(0xffffffffu, mbar_wait(&pv_done[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1, abort_v)))
      ok = false;
    pdl_trigger();  // the main loop is done: let the next kernel be scheduled
    // Epilogue: lane kl holds O^T[d = kl][rows] and L^T[.][rows] (the same on
    // every lane); this thread takes its 8 of every 16 rows.
    if (ok && nblk > 0) tc_fence_after();
    float* part = reinterpret_cast<float*>(sStage);  // the K/V stages are idle now
    const bool have = ok && nblk > 0;
#pragma unroll 1
    for (int g16 = 0; g16 < ngrp; ++g16) {
      const int c0 = g16 * 16 + h * 8;
      float o[8], l8[8];
      if (have) {
        tmem_ld8(tO + c0, o);
        tmem_ld8(tL + c0, l8);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = l8[e] = 0.f;
      }
      if (kl < D) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = c0 + e;
          if (r >= rows_valid) break;
          const float on = l8[e] > 0.f ? __fdividef(o[e], l8[e]) : 0.f;
          if (nch == 1) {
            const int gr = row0 + r, node = gr / G;
            out[((size_t)(off + node) * plan.Hq + g * G + (gr - node * G)) * D + kl] = __float2bfloat16_rn(on);
          } else {
            part[r * D + kl] = on;
          }
        }
      }
      if (nch > 1 && kl < 8 && c0 + kl < rows_valid) {
        float le = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e == kl) le = l8[e];
        sLse[c0 + kl] = le > 0.f ? sMref[c0 + kl] + __log2f(le) : -INFINITY;
      }
    }
  }

  // ---------------------------------------------------------------- cluster merge
  __syncwarp();
  if (nch > 1) {
    cluster_sync_all();  // every partial of the group is in its CTA's shared memory
    if (warp < 8) {
      // Rank c merges rows [r_lo, r_hi) of the tile.
      const int t = tid;
      const int r_lo = (c * rows_valid) / nch, r_hi = ((c + 1) * rows_valid) / nch;
      const int nr = r_hi - r_lo;
      // out[row][4 d] = sum over chunks of w_c x partial_c / sum of w_c with
      // w_c = 2^(lse_c - max lse): each item loads its row's log-sum-exps and
      // its 16 bytes of every partial in one round of remote loads, then
      // weighs them itself (no barrier between weights and sums).
      constexpr int D4 = D / 4;
      const uint32_t part_s = smem_u32(sStage);
      for (int i = t; i < nr * D4; i += kKeysLaneThreads) {
        const int r = r_lo + i / D4, d4 = i % D4;
        float lse[8];
        float4 v[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          if (cc < nch) {
            lse[cc] = ld_dsmem_f32(mapa_shared(smem_u32(sLse + r), cc));
            v[cc] = ld_dsmem_f32x4(mapa_shared(part_s + (uint32_t)(r * D + 4 * d4) * 4, cc));
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
            if (w > 0.f) {  // a chunk of weight 0 may hold anything
              acc.x += w * v[cc].x;
              acc.y += w * v[cc].y;
              acc.z += w * v[cc].z;
              acc.w += w * v[cc].w;
              wsum += w;
            }
          }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        const int gr = row0 + r, node = gr / G;
        __nv_bfloat16* o = out + ((size_t)(off + node) * plan.Hq + g * G + (gr - node * G)) * D + 4 * d4;
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
      }
    }
    cluster_sync_all();  // every CTA keeps its shared memory until its peers have read it
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_v) status[b] = TSV_ERR_TIMEOUT;
  if (warp == kKeysMmaWarp) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, C::kTmemCols);
  }
}

size_t attention_keys_smem_bytes(int D) {
  return D == 64 ? (size_t)KeysCfg<64>::kSmemBytes : (size_t)KeysCfg<128>::kSmemBytes;
}

cudaError_t attention_keys_set_attributes(int D) {
  if (D == 64)
    return cudaFuncSetAttribute(tree_attn_keys_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                KeysCfg<64>::kSmemBytes);
  return cudaFuncSetAttribute(tree_attn_keys_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              KeysCfg<128>::kSmemBytes);
}

cudaError_t launch_attention_keys(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                  const CUtensorMap& tmap_v, const AttnPlan& plan,
                                  const int32_t* parent, const uint32_t* anc, void* out,
                                  int32_t* status, cudaStream_t st) {
  if (plan.n_units == 0) return cudaSuccess;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
  const size_t smem = attention_keys_smem_bytes(plan.D);
  if (plan.D == 64)
    return launch_pdl(tree_attn_keys_kernel<64>, dim3(plan.n_units), dim3(kKeysThreads), smem, st,
                      (unsigned)plan.cluster, tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, status);
  return launch_pdl(tree_attn_keys_kernel<128>, dim3(plan.n_units), dim3(kKeysThreads), smem, st,
                    (unsigned)plan.cluster, tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, status);
}

}  // namespace tsv
