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
//   S^T = K Q^T      M = 128 keys, N = rows, K = D          (A = K tile, B = Q tile)
//   O^T += V^T P^T   M = 128 (d), N = rows, K = 128 keys    (A = V tile, M-major)
//
// N is the unit's row count rounded up to 16.  The softmax denominators are
// summed by the key-lane threads themselves, in registers, from the same
// bf16-rounded P that the PV MMA reads, and reduced over the 128 key lanes
// once per unit: each tcgen05.mma occupies the tensor pipe for about the same
// time whatever its N, so two MMA streams per block (S^T, PV) instead of
// three leave the pipe off the critical path.
//
// Eight key-lane warps: warps w and w+4 share TMEM lanes 32(w%4).. and split
// every 16-row column group into two halves of 8 rows.  Rows beyond the tree
// carry a reference maximum of +inf, so their probabilities are zero without
// any per-element test; only blocks that reach the tree part of the keys
// apply the ancestor mask, built per unit from parent[] (loaded one unit
// ahead) as "rows that see tree key j" bit masks.  A row's reference maximum
// moves only when a visible score exceeds it by more than 2^32 (always on its
// first visible block): one OR-reducing named barrier per block decides, and
// the rare move is a warp-shuffle maximum plus a rescale of O^T in TMEM and of
// the register row sums.
//
// Work units are (request, KV head, key chunk).  Each CTA writes the units it
// takes into a table in shared memory at entry, in one parallel round over
// the plan, so no role searches the kernel parameters on its critical path.
// A launch with more units than SMs and one chunk per request is persistent:
// one CTA per SM takes units i, 2G-1-i, 2G+i, ... of the longest-first order;
// its producer streams the next unit's K/V while the key lanes finish the
// previous one, O^T is double-buffered in TMEM, and four epilogue warps
// normalise and store a finished unit while the key lanes go on.
//
// When a request's keys are split into K chunks (K <= 8), the K CTAs of a
// chunk group form one cluster: each leaves its normalised partial and
// log2-sum-exp in its own shared memory, and CTA rank c merges the c-th
// share of the rows through distributed shared memory (weights first, then
// 16-byte loads kept in flight together) — no global partials, no atomics,
// no second kernel.
//
// Warp roles (448 threads): warps 0-7 key lanes (softmax, P^T, row sums, and
// the epilogue of a non-persistent launch), warp 8 TMA producer (K/V blocks of
// 128 keys into a 3-stage ring, each unit's Q tile after its first block),
// warp 9 tcgen05 issuer and TMEM owner, warps 10-13 epilogue of a persistent
// launch.  The issuer keeps two streams, S^T of the next block and PV of the
// oldest block whose P^T is in, and issues whichever is ready first, so a
// stage is released as soon as its own block is done.  P^T of a block is
// written over that block's K tile, which S^T has finished reading, so the
// ring needs no separate P buffers and three 64 KB stages fit next to Q.
#include "tsv_attention_common.cuh"

namespace tsv {

constexpr int kKeysLaneThreads = 256;
constexpr int kKeysEpiThreads = 128;  // epilogue warps of a persistent launch
constexpr int kKeysThreads = kKeysLaneThreads + 64 + kKeysEpiThreads;
constexpr int kKeysProducerWarp = 8, kKeysMmaWarp = 9;  // then the epilogue warps
constexpr int kKeysBlock = kKeysBlockKeys;   // keys per block (MMA M)
constexpr int kKeysRows = kKeysTileRows;     // query rows per CTA (MMA N)
constexpr int kKeysMaxTree = kKeysTileRows;  // n * G <= 64 implies n <= 64
constexpr float kKeysOverflow = 32.f;        // log2 units
constexpr int kBarKeysSetup = 1;             // key lanes + MMA warp + epilogue warps
constexpr int kBarKeys = 2;                  // key lanes
constexpr int kKeysMaxUnits = kKeysMaxUnitsPerCta;
constexpr int kKeysStages = 3;               // K/V ring depth

// One unit of work: (request b, KV head g, key chunk c, M-tile mt) and the
// key range it streams.  Each CTA writes the units it takes into a table in
// shared memory once, at entry, so that no role looks anything up in the
// kernel parameters on its critical path.
struct KeysUnit {
  int b, local, nch, mtiles, c, mt, g;
  int P, n, off, row0, rows_valid, ngrp;
  int k_begin, k_end, nblk;
};

// The k-th unit of this CTA, or -1 past the last.  One unit per CTA, except in
// a persistent launch (grid < units): CTA i then takes units i, 2G-1-i, 2G+i,
// 4G-1-i, ... of the longest-first unit order (G = grid), so every CTA gets
// one long and one short unit of each pair of rounds.
__device__ __forceinline__ int keys_unit_id(const AttnPlan& plan, int k) {
  if (!plan.persistent) return k == 0 ? (int)blockIdx.x : -1;
  const int G = (int)gridDim.x;
  const int u = k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
  return u < plan.n_units ? u : -1;
}

// Fills the unit table (all threads of the CTA take part): thread t < B owns
// slot t's unit range, so every unit is found in one round of parameter loads.
// Returns the number of units of this CTA.
__device__ __forceinline__ int keys_fill_units(const AttnPlan& plan, KeysUnit* table) {
  int n_my = 0;
  while (n_my < kKeysMaxUnits && keys_unit_id(plan, n_my) >= 0) ++n_my;
  const int t = threadIdx.x;
  if (t < plan.B) {
    const int lo = plan.unit_start[t], hi = plan.unit_start[t + 1];
    if (lo < hi) {
      const int b = plan.slot_req[t];
      const int nch = plan.n_chunks[b], mtiles = plan.mtiles[b], P = plan.prefix[b], n = plan.nodes[b];
      const int off = plan.node_off[b], clen = plan.chunk_len[b];
      for (int k = 0; k < n_my; ++k) {
        const int unit = keys_unit_id(plan, k);
        if (unit < lo || unit >= hi) continue;
        KeysUnit u;
        u.b = b;
        u.local = unit - lo;
        u.nch = nch;
        u.mtiles = mtiles;
        u.c = u.local % nch;
        const int gm = u.local / nch;
        u.mt = gm % mtiles;
        u.g = gm / mtiles;
        u.P = P;
        u.n = n;
        u.off = off;
        u.row0 = u.mt * kKeysRows;
        u.rows_valid = min(kKeysRows, n * plan.G - u.row0);
        u.ngrp = (u.rows_valid + 15) >> 4;  // 16-row column groups holding valid rows
        u.k_begin = min(P + n, u.c * clen);
        u.k_end = min(P + n, u.k_begin + clen);
        u.nblk = (u.k_end - u.k_begin + kKeysBlock - 1) / kKeysBlock;
        table[k] = u;
      }
    }
  }
  return n_my;
}

// Walks this CTA's K/V blocks in order across its units (the order in which
// the producer loads them and the MMA warp consumes them).  jg counts blocks
// over all units (the ring stage and barrier phases follow it); kq counts the
// units that have blocks (the Q buffer's phases follow it).
struct KeysCursor {
  int k, j, jg, kq, nblk;
  int st, ph;  // ring stage of block jg (jg % stages) and its use count parity ((jg / stages) & 1)
  bool valid;
};

__device__ __forceinline__ KeysCursor keys_cursor_first(const KeysUnit* table, int n_my) {
  KeysCursor c{0, 0, 0, 0, 0, 0, 0, false};
  for (; c.k < n_my; ++c.k) {
    c.nblk = table[c.k].nblk;
    if (c.nblk > 0) {
      c.valid = true;
      break;
    }
  }
  return c;
}

__device__ __forceinline__ KeysCursor keys_cursor_next(const KeysUnit* table, int n_my, KeysCursor c) {
  ++c.jg;
  if (++c.st == kKeysStages) {
    c.st = 0;
    c.ph ^= 1;
  }
  if (++c.j < c.nblk) return c;
  c.j = 0;
  ++c.kq;
  for (++c.k; c.k < n_my; ++c.k) {
    c.nblk = table[c.k].nblk;
    if (c.nblk > 0) return c;
  }
  c.valid = false;
  return c;
}

template <int D>
struct KeysCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = kKeysStages;
  static constexpr int kQBytes = kKeysRows * D * 2;
  static constexpr int kKTile = kKeysBlock * D * 2;
  static constexpr int kVTile = kKeysBlock * 128 * 2;  // always 128 d: upper half zero when D = 64
  static constexpr int kStageBytes = kKTile + kVTile;
  static constexpr int kPBytes = kKeysBlock * kKeysRows * 2;  // P^T, written over the K tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffStage = kOffQ + kQBytes;
  static constexpr int kOffDesc = kOffStage + kStages * kStageBytes;  // uint32 [64][2]
  static constexpr int kOffPar = kOffDesc + kKeysMaxTree * 8;   // int32 [64]
  static constexpr int kOffMref = kOffPar + kKeysMaxTree * 4;   // float [64]
  static constexpr int kOffAlpha = kOffMref + kKeysRows * 4;    // float [64]
  static constexpr int kOffWmax = kOffAlpha + kKeysRows * 4;    // float [4][64]
  static constexpr int kOffLse = kOffWmax + 4 * kKeysRows * 4;  // float [64]
  static constexpr int kOffLsum = kOffLse + kKeysRows * 4;     // float [2][64]: row sums of a unit
  static constexpr int kOffUnits = kOffLsum + 2 * kKeysRows * 4;  // KeysUnit [kKeysMaxUnits]
  static constexpr int kOffBar = kOffUnits + kKeysMaxUnits * 64;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done[2], mma_done, q_empty,
  // o_full[2], o_free[2]
  static constexpr int kNumBars = 1 + 2 * kStages + 12;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 32 + 1024;
  static_assert(sizeof(KeysUnit) == 64, "unit table entry");
  // S0 | S1 | O0 | O1, 64 columns each (O1: the second O^T buffer of a persistent launch).
  static constexpr uint32_t kTmemCols = 256;
  static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0, "atoms");
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
  uint32_t* sDesc = reinterpret_cast<uint32_t*>(smem + C::kOffDesc);
  int32_t* sPar = reinterpret_cast<int32_t*>(smem + C::kOffPar);
  float* sMref = reinterpret_cast<float*>(smem + C::kOffMref);
  float* sAlpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
  float* sWmax = reinterpret_cast<float*>(smem + C::kOffWmax);
  float* sLse = reinterpret_cast<float*>(smem + C::kOffLse);
  float* sLsum = reinterpret_cast<float*>(smem + C::kOffLsum);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + S;
  uint64_t* s_full = kv_empty + S;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* mma_done = pv_done + 2;
  uint64_t* q_empty = mma_done + 1;  // Q of a unit read by its last S^T MMA
  uint64_t* o_full = q_empty + 1;    // [2] a unit's last PV is done and its row sums are in (persistent)
  uint64_t* o_free = o_full + 2;     // [2] the epilogue warps have read that O^T and L^T
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  int* cur_req = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  int* fail_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 12);
  volatile int* abort_v = abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = plan.G;

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
    mbar_init(q_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&o_full[x], 2);  // the MMA warp's commit and one key-lane thread
      mbar_init(&o_free[x], kKeysEpiThreads);
    }
    *abort_flag = 0;
    *fail_flag = 0;
    *cur_req = -1;
    mbar_fence_init();
  }
  KeysUnit* sUnits = reinterpret_cast<KeysUnit*>(smem + C::kOffUnits);
  const int n_my = keys_fill_units(plan, sUnits);  // the same count in every thread
  __syncthreads();
  // The unit comes from the plan alone, so when all units run in the first
  // wave its Q tile and the first ring's worth of K/V are pulled into L2
  // while the previous kernel finishes.
  if (plan.prefetch_l2 && warp == kKeysProducerWarp && lane == 0) {
    const KeysUnit& U = sUnits[0];
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
#pragma unroll
    for (int hf = 0; hf < C::kHalves; ++hf) tma_prefetch_3d(&tmap_q, hf * 64, U.g * G, U.off + U.row0 / G);
    for (int j = 0; j < U.nblk && j < C::kStages; ++j)
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf) {
        tma_prefetch_4d(&tmap_k, hf * 64, U.g, U.k_begin + j * kKeysBlock, U.b);
        tma_prefetch_4d(&tmap_v, hf * 64, U.g, U.k_begin + j * kKeysBlock, U.b);
      }
  }
  pdl_wait();  // the previous kernel's results are visible from here on
  // The next kernel may be scheduled now: it waits for this one's completion
  // itself, and it is launched only once every CTA of this grid has started,
  // so it only takes SM room this grid leaves free (verification launched to
  // run beside this attention fills that room).
  pdl_trigger();

  if (warp == kKeysProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_q);
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
      // Blocks in order over the units.  A unit's Q tile goes right after its
      // first K/V block: the Q buffer is free only once the previous unit's
      // last S^T MMA has read it, and the ring should not stall behind that.
      int jg = 0, kq = 0;
      for (KeysCursor x = keys_cursor_first(sUnits, n_my); x.valid; x = keys_cursor_next(sUnits, n_my, x)) {
        const KeysUnit& U = sUnits[x.k];
        const uint64_t pol = U.mtiles > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
        const int st = x.st;
        if (x.jg >= S && !mbar_wait(&kv_empty[st], x.ph ^ 1, abort_v)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kHalves * kKeysBlock * 128);
        const int key0 = U.k_begin + x.j * kKeysBlock;
        uint8_t* kt = sStage + st * C::kStageBytes;
        uint8_t* vt = kt + C::kKTile;
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_load_4d(kt + hf * (kKeysBlock * 128), &tmap_k, &kv_full[st], hf * 64, U.g, key0, U.b, pol);
          tma_load_4d(vt + hf * (kKeysBlock * 128), &tmap_v, &kv_full[st], hf * 64, U.g, key0, U.b, pol);
        }
        jg = x.jg + 1;
        if (x.j == 0) {
          if (x.kq > 0 && !mbar_wait(q_empty, (x.kq - 1) & 1, abort_v)) break;
          mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(sQ + hf * (kKeysRows * 128), &tmap_q, q_full, hf * 64, U.g * G, U.off + U.row0 / G, pol);
          kq = x.kq + 1;
        }
      }
      if (*abort_v) {  // let the copies in flight land before the CTA leaves
        if (kq > 0) mbar_wait(q_full, (kq - 1) & 1, nullptr);
        for (int x = (jg > S ? jg - S : 0); x < jg; ++x) mbar_wait(&kv_full[x % S], (x / S) & 1, nullptr);
      }
    }
  } else if (warp == kKeysMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
    named_bar(kBarKeysSetup, kKeysLaneThreads + 32 + kKeysEpiThreads);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (lane == 0) {
      // N of every MMA = the unit's query rows rounded up to 16 (M = 128 takes
      // N = 16 .. 256 in steps of 16): a 16-row tree does a quarter of the
      // tensor work of a full 64-row tile.
      auto n_of = [&](const KeysCursor& x) { return 16 * sUnits[x.k].ngrp; };
      const uint32_t qa = smem_u32(sQ), sa = smem_u32(sStage);
      // Shared-memory descriptors are built once; a tile inside a stage, or a
      // K slice inside a tile, is the base descriptor plus its offset / 16 in
      // the start-address field (every address here is below 256 KB, so the
      // field never carries into the next one).  The issuing thread's work
      // per MMA is what bounds a block: one add per operand, no rebuild.
      const uint64_t dK0 = sdesc_sw128(sa, 16, 1024);                             // K tile, K-major
      const uint64_t dQ0 = sdesc_sw128(qa, 16, 1024);                             // Q tile, K-major
      const uint64_t dV0 = sdesc_sw128(sa + C::kKTile, kKeysBlock * 128, 1024);   // V^T, M-major
      const uint64_t dP0 = sdesc_sw128(sa, kKeysBlock * 128, 1024);               // P^T, N-major
      constexpr uint32_t kStageDesc = C::kStageBytes >> 4;
      auto issue_s = [&](const KeysCursor& x, int nN) {
        const uint32_t idS = idesc_bf16_f32_ab(kKeysBlock, nN, 0, 0);
        const uint64_t dk = dK0 + (uint64_t)(x.st * kStageDesc);
        const uint32_t dst = tmem + (uint32_t)((x.jg & 1) * kKeysRows);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr uint32_t kA = kKeysBlock * 128 / 16, kB = kKeysRows * 128 / 16;
          const uint32_t ao = (kk >> 2) * kA + (kk & 3) * 2;
          const uint32_t bo = (kk >> 2) * kB + (kk & 3) * 2;
          umma_bf16(dst, dk + ao, dQ0 + bo, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[x.jg & 1]);
      };
      // O^T of unit kq: columns 128.. (buffer 0) or 192.. (buffer 1, persistent only).
      auto issue_pv = [&](const KeysCursor& x, int nN) {
        const uint32_t idO = idesc_bf16_f32_ab(128, nN, 1, 1);
        const uint32_t tO = tmem + (uint32_t)((2 + (plan.persistent ? x.kq & 1 : 0)) * kKeysRows);
        const uint64_t dv = dV0 + (uint64_t)(x.st * kStageDesc);
        const uint64_t dp = dP0 + (uint64_t)(x.st * kStageDesc);  // P^T over K(jg)
        const uint32_t acc0 = x.j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kKeysBlock / 16; ++kk)
          umma_bf16(tO, dv + kk * (2048 / 16), dp + kk * (2048 / 16), idO, kk > 0 ? 1u : acc0);
        umma_commit(&pv_done[x.jg & 1]);
        umma_commit(&kv_empty[x.st]);
      };
      // Two independent streams of work, issued in whichever order their
      // inputs arrive: S^T of block xs (its unit's Q, first block only, and its
      // K/V tile have landed; the S buffer it writes was last read by block
      // xs - 2, whose P^T is in) and PV of block xp (its P^T is in; in a
      // persistent launch a unit's first PV overwrites the O^T | L^T buffer of
      // the unit two before it, which the epilogue warps must have read).
      // PV(j) never waits for block j+1's tile, so a stage is released as soon
      // as its own block is done.  The unit's last S^T releases the Q buffer;
      // its last PV hands O^T | L^T to the epilogue warps.
      KeysCursor xs = keys_cursor_first(sUnits, n_my), xp = xs;
      bool ok = true;
      // The time limit is checked once every 1024 idle polls: reading the
      // global timer on every poll would delay each issue by far more than
      // the poll itself.
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      while (xp.valid) {
        bool did = false;
        if (xs.valid && xs.jg <= xp.jg + 1 && (xs.j != 0 || mbar_test_wait(q_full, xs.kq & 1)) &&
            mbar_test_wait(&kv_full[xs.st], xs.ph)) {
          tc_fence_after();
          issue_s(xs, n_of(xs));
          if (xs.j == xs.nblk - 1) umma_commit(q_empty);
          xs = keys_cursor_next(sUnits, n_my, xs);
          did = true;
        }
        if (xp.jg < xs.jg && mbar_test_wait(&p_full[xp.jg & 1], (xp.jg >> 1) & 1) &&
            (xp.j != 0 || !plan.persistent || xp.kq < 2 ||
             mbar_test_wait(&o_free[xp.kq & 1], ((xp.kq >> 1) - 1) & 1))) {
          tc_fence_after();
          issue_pv(xp, n_of(xp));
          if (plan.persistent && xp.j == xp.nblk - 1) umma_commit(&o_full[xp.kq & 1]);
          xp = keys_cursor_next(sUnits, n_my, xp);
          did = true;
        }
        if (did) {
          t_idle = 0;
          idle_polls = 0;
        } else if ((++idle_polls & 1023u) == 0) {
          const uint64_t now = global_timer_ns();
          if (t_idle == 0) t_idle = now;
          if (*abort_v || now - t_idle > kWaitLimitNs) {
            *abort_v = 1;
            ok = false;
            break;
          }
        }
      }
      (void)ok;
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, nullptr);
    }
  } else if (warp < kKeysProducerWarp) {
    // ------------------------------------------------------------ key-lane threads
    const int t = tid;              // 0 .. 255
    const int lg = warp & 3;        // TMEM lane group
    const int kl = lg * 32 + lane;  // key lane (and d for O^T)
    const int h = warp >> 2;        // which 8 of every 16 rows
    const uint32_t lane_base = (uint32_t)(lg * 32) << 16;
    // Tree of a unit's request: parent[] (n <= 64) or the prepared ancestor
    // words of the thread's row.  Loaded one unit ahead, so that the global
    // load's latency hides behind the setup (first unit) or the previous unit.
    auto load_tree = [&](int k, int& par, uint32_t& a0, uint32_t& a1) {
      par = -1;
      a0 = a1 = 0u;
      if (k >= n_my) return;
      const KeysUnit& V = sUnits[k];
      if (anc == nullptr) {
        if (t < V.n) par = __ldg(parent + V.off + t);
      } else if (t < V.rows_valid) {
        const uint2 a2 =
            __ldg(reinterpret_cast<const uint2*>(anc + (size_t)(V.off + (V.row0 + t) / G) * TSV_ANC_WORDS));
        a0 = a2.x;
        a1 = a2.y;
      }
    };
    int nx_par;
    uint32_t nx_anc0, nx_anc1;
    load_tree(0, nx_par, nx_anc0, nx_anc1);
    {
      if (D == 64) {  // the upper half of every V stage stays zero
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        for (int st = 0; st < S; ++st) {
          uint4* vh = reinterpret_cast<uint4*>(sStage + st * C::kStageBytes + C::kKTile + kKeysBlock * 128);
          for (int i = t; i < kKeysBlock * 128 / 16; i += kKeysLaneThreads) vh[i] = z;
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar(kBarKeysSetup, kKeysLaneThreads + 32 + kKeysEpiThreads);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const float sl2 = plan.scale_log2;
    // A failed (timed-out) wait is made CTA-wide before anyone leaves the loop,
    // so every named barrier below is reached by all key-lane threads.
    bool ok = true;
    int jg = 0, kq = 0;
    int lst = 0;  // ring stage of block jg
    for (int k = 0; ok && k < n_my; ++k) {
      const KeysUnit U = sUnits[k];
      const int my_par = nx_par;
      const uint32_t my_anc0 = nx_anc0, my_anc1 = nx_anc1;
      load_tree(k + 1, nx_par, nx_anc0, nx_anc1);
      if (plan.persistent && U.nblk == 0) continue;
      const int P = U.P, n = U.n, off = U.off, row0 = U.row0, rows_valid = U.rows_valid, ngrp = U.ngrp;
      const int nblk = U.nblk, k_end = U.k_end;
      // This unit's O^T (buffer kq & 1 in a persistent launch).
      const int kq_unit = kq;
      const uint32_t tO = tmem + lane_base + (uint32_t)((2 + (plan.persistent ? kq & 1 : 0)) * kKeysRows);
      if (nblk > 0) ++kq;
      // Row sums of P over this thread's key, for its 8 of every 16 rows
      // (group g16 < ngrp), of the same bf16-rounded P the PV MMA reads.
      float lsum[4][8];
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) lsum[g][e] = 0.f;
      // The previous unit's readers of sMref, sDesc and sPar are done.
      if (k > 0) named_bar(kBarKeys, kKeysLaneThreads);
      if (t == 0) *cur_req = U.b;
      if (t < kKeysRows) {
        sMref[t] = t < rows_valid ? -INFINITY : INFINITY;  // rows past the tree never see a key
        sAlpha[t] = 1.f;
      }
      if (anc == nullptr && t < n) sPar[t] = my_par;
      const bool bad = named_bar_or(kBarKeys, kKeysLaneThreads,
                                    anc == nullptr && t < n && (my_par < -1 || my_par >= t));
      if (anc == nullptr && U.local == 0 && t == 0) status[U.b] = bad ? TSV_ERR_BAD_TREE : TSV_OK;
      bool desc_ready = false;
      for (int j = 0; j < nblk; ++j, ++jg) {
        const int key0 = U.k_begin + j * kKeysBlock;
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
        const bool okj = __all_sync(0xffffffffu, mbar_wait(&s_full[jg & 1], (jg >> 1) & 1, abort_v));
        tc_fence_after();
        const int key = key0 + kl;
        const bool full_vis = key < P;
        uint64_t vis = 0ull;  // used only when !full_vis
        if (!full_vis && key < k_end)
          vis = (uint64_t)sDesc[2 * (key - P)] | ((uint64_t)sDesc[2 * (key - P) + 1] << 32);
        const uint32_t s_col = tmem + lane_base + (uint32_t)((jg & 1) * kKeysRows);
        // P of this block against the current reference maxima, kept packed
        // in registers: if no visible score exceeds its row's reference by
        // more than 2^32 (the common case) these are the block's P; else the
        // maxima move and P is computed again.  The first block always moves
        // the maxima (they start at -inf): it skips the optimistic pass.
        uint32_t pk[4][4];
        float over = j == 0 ? INFINITY : -INFINITY;
        auto p_pass = [&](bool track) {
#pragma unroll
          for (int g16 = 0; g16 < 4; ++g16) {
            if (g16 >= ngrp) break;
            const int c0 = g16 * 16 + h * 8;
            float sv[8];
            tmem_ld8(s_col + c0, sv);
            const float4 ma = *reinterpret_cast<const float4*>(sMref + c0);
            const float4 mb = *reinterpret_cast<const float4*>(sMref + c0 + 4);
            const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
            const uint32_t vm = full_vis ? 0xFFu : (uint32_t)(vis >> c0) & 0xFFu;
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float x = ((vm >> e) & 1u) ? fmaf(sv[e], sl2, -m[e]) : -INFINITY;
              if (track) over = fmaxf(over, x);
              p[e] = fast_exp2(x);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) pk[g16][i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
          }
        };
        if (j > 0) p_pass(true);
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
#pragma unroll
          for (int g16 = 0; g16 < 4; ++g16)  // row sums of earlier blocks follow the new maxima
            if (g16 < ngrp)
#pragma unroll
              for (int e = 0; e < 8; ++e) lsum[g16][e] *= sAlpha[g16 * 16 + h * 8 + e];
          if (j > 0) {  // O^T holds PV(0..j-1): rescale this thread's columns
            if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(jg - 1) & 1], ((jg - 1) >> 1) & 1, abort_v)))
              *fail_flag = 1;  // seen by everyone at the next block's barrier
            tc_fence_after();
#pragma unroll 1
            for (int g16 = 0; g16 < ngrp; ++g16) {
              const int c0 = g16 * 16 + h * 8;
              float o[8];
              tmem_ld8(tO + c0, o);
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] *= sAlpha[c0 + e];
              tmem_st8(tO + c0, o);
            }
          }
          p_pass(false);  // against the moved maxima
        }
        // P^T goes over the K tile of this block: S^T(j) has finished reading it.
        uint8_t* prow = sStage + lst * C::kStageBytes + kl * 128;
#pragma unroll
        for (int g16 = 0; g16 < 4; ++g16) {
          if (g16 >= ngrp) break;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lsum[g16][2 * i] += __uint_as_float(pk[g16][i] << 16);
            lsum[g16][2 * i + 1] += __uint_as_float(pk[g16][i] & 0xFFFF0000u);
          }
          const int chunk = 2 * g16 + h;
          *reinterpret_cast<uint4*>(prow + ((chunk ^ (kl & 7)) << 4)) =
              make_uint4(pk[g16][0], pk[g16][1], pk[g16][2], pk[g16][3]);
        }
        // A V row past the request's keys may hold anything (even NaN): zero it.
        if (key >= k_end && h < C::kHalves) {
          uint4* vrow = reinterpret_cast<uint4*>(sStage + lst * C::kStageBytes + C::kKTile +
                                                 h * (kKeysBlock * 128) + kl * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) vrow[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[jg & 1]);
        lst = lst + 1 == S ? 0 : lst + 1;
      }
      // Row sums over the 128 key lanes: a transposed warp reduction (as for the
      // maxima) leaves lane l of each warp with row c0 + ((l >> 2) & 7) summed
      // over the warp's 32 keys; then the four lane-group warps' sums are added.
#pragma unroll
      for (int g16 = 0; g16 < 4; ++g16) {
        if (g16 >= ngrp) break;
        const int c0 = g16 * 16 + h * 8;
        const float* v = lsum[g16];
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
        float w4[4], w2[2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w4[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 4], 16);
#pragma unroll
        for (int i = 0; i < 2; ++i)
          w2[i] = (b3 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, b3 ? w4[i] : w4[i + 2], 8);
        float w1 = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
        if ((lane & 3) == 0) sWmax[lg * kKeysRows + c0 + (lane >> 2)] = w1;
      }
      // In a persistent launch the row-sum buffer of this unit was last read by
      // the epilogue of the unit two before it.
      float* lrow = sLsum + (plan.persistent ? (kq_unit & 1) * kKeysRows : 0);
      if (plan.persistent && kq_unit >= 2 && t < rows_valid &&
          !mbar_wait(&o_free[kq_unit & 1], ((kq_unit >> 1) - 1) & 1, abort_v))
        *fail_flag = 1;
      named_bar(kBarKeys, kKeysLaneThreads);
      if (t < rows_valid)
        lrow[t] = (sWmax[t] + sWmax[kKeysRows + t]) + (sWmax[2 * kKeysRows + t] + sWmax[3 * kKeysRows + t]);
      named_bar(kBarKeys, kKeysLaneThreads);
      if (*fail_flag) ok = false;
      // A persistent launch leaves the epilogue to the epilogue warps (the
      // unit's row sums are in, and the MMA warp's commit covers its O^T) and
      // goes straight on to its next unit.
      if (plan.persistent) {
        if (t == 0) mbar_arrive(&o_full[kq_unit & 1]);
        continue;
      }
      if (ok && nblk > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(&pv_done[(jg - 1) & 1], ((jg - 1) >> 1) & 1, abort_v)))
        ok = false;
      // Epilogue: lane kl holds O^T[d = kl][rows] and L^T[.][rows] (the same on
      // every lane); this thread takes its 8 of every 16 rows.
      if (ok && nblk > 0) tc_fence_after();
      float* part = reinterpret_cast<float*>(sStage);  // the K/V stages are idle now (clusters only)
      const bool have = ok && nblk > 0;
#pragma unroll 1
      for (int g16 = 0; g16 < ngrp; ++g16) {
        const int c0 = g16 * 16 + h * 8;
        float o[8], l8[8];
        if (have) {
          tmem_ld8(tO + c0, o);
#pragma unroll
          for (int e = 0; e < 8; ++e) l8[e] = lrow[c0 + e];
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
            if (U.nch == 1) {
              const int gr = row0 + r, node = gr / G;
              out[((size_t)(off + node) * plan.Hq + U.g * G + (gr - node * G)) * D + kl] =
                  __float2bfloat16_rn(on);
            } else {
              part[r * D + kl] = on;
            }
          }
        }
        if (U.nch > 1 && kl < 8 && c0 + kl < rows_valid) {
          float le = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e == kl) le = l8[e];
          sLse[c0 + kl] = le > 0.f ? sMref[c0 + kl] + __log2f(le) : -INFINITY;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    // Persistent launches only: for each unit, once its last PV is done and the
    // key lanes have left its row sums, lane d of O^T gives out[row][d] =
    // O^T[d][row] / sum[row] for every row; then the O^T buffer and the row sums
    // go back to the MMA warp and the key lanes (two units later).
    tc_fence_before();
    named_bar(kBarKeysSetup, kKeysLaneThreads + 32 + kKeysEpiThreads);
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (plan.persistent) {
      const int lq = warp & 3;        // TMEM lane quadrant of this warp
      const int d = lq * 32 + lane;   // its lane of O^T: the head dimension index
      const uint32_t lane_base = (uint32_t)(lq * 32) << 16;
      int kq = 0;
      for (int k = 0; k < n_my; ++k) {
        const KeysUnit& U = sUnits[k];
        if (U.nblk == 0) continue;
        const int ob = kq & 1;
        const bool okw = __all_sync(0xffffffffu, mbar_wait(&o_full[ob], (kq >> 1) & 1, abort_v));
        ++kq;
        if (!okw) break;
        tc_fence_after();
        const uint32_t tO = tmem + lane_base + (uint32_t)((2 + ob) * kKeysRows);
        const float* lrow = sLsum + ob * kKeysRows;
#pragma unroll 1
        for (int g16 = 0; g16 < U.ngrp; ++g16) {
          float o[16], l16[16];
          tmem_ld16(tO + g16 * 16, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) l16[e] = lrow[g16 * 16 + e];
          if (d < D) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int r = g16 * 16 + e;
              if (r >= U.rows_valid) break;
              const int gr = U.row0 + r, node = gr / G;
              const float on = l16[e] > 0.f ? __fdividef(o[e], l16[e]) : 0.f;
              out[((size_t)(U.off + node) * plan.Hq + U.g * G + (gr - node * G)) * D + d] = __float2bfloat16_rn(on);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&o_free[ob]);
      }
    }
  }

  // ---------------------------------------------------------------- cluster merge
  __syncwarp();
  const KeysUnit& U0 = sUnits[0];  // a non-persistent CTA's only unit
  const int nch = U0.nch;
  if (!plan.persistent && nch > 1) {
    cluster_sync_all();  // every partial of the group is in its CTA's shared memory
    if (warp < 8) {
      // Rank c merges rows [r_lo, r_hi) of the tile.
      const int t = tid;
      const int rows_valid = U0.rows_valid;
      const int r_lo = (U0.c * rows_valid) / nch, r_hi = ((U0.c + 1) * rows_valid) / nch;
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
        const int gr = U0.row0 + r, node = gr / G;
        __nv_bfloat16* o =
            out + ((size_t)(U0.off + node) * plan.Hq + U0.g * G + (gr - node * G)) * D + 4 * d4;
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
      }
    }
    cluster_sync_all();  // every CTA keeps its shared memory until its peers have read it
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_v && *cur_req >= 0) status[*cur_req] = TSV_ERR_TIMEOUT;
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
  const dim3 grid(plan.persistent ? plan.grid : plan.n_units);
  if (plan.D == 64)
    return launch_pdl(tree_attn_keys_kernel<64>, grid, dim3(kKeysThreads), smem, st, (unsigned)plan.cluster,
                      tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, status);
  return launch_pdl(tree_attn_keys_kernel<128>, grid, dim3(kKeysThreads), smem, st, (unsigned)plan.cluster,
                    tmap_q, tmap_k, tmap_v, plan, parent, anc, ob, status);
}

}  // namespace tsv
