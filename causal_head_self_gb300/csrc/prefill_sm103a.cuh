// prefill_sm103a.cuh -- fused causal / sliding-window / GQA attention forward
// for sm_103a: O = softmax(Q K^T * scale + M) V per (batch, query head).
//
// What it computes is the scaled dot-product attention of "Механизм внимания"
// (llm-arch-research.openidealab.com/textbook/attention), section "Scaled
// dot-product attention", with the mask of sections "Маскирование" (causal)
// and "Скользящее окно" (window, i - j < W form), and the head map
// g(h) = floor(h / (H/G)) of section "Виды по числу голов K/V: MHA, GQA, MQA".
// The score matrix never leaves the chip: scores are formed tile by tile and
// folded into the output with a running row maximum and running row sum (the
// online softmax that "多头注意力机制" (blog.euler0525.cn), section "Flash
// Attention", and the textbook's section "Эффективные реализации" describe).
//
// This kernel runs head size 64, and head size 128 beyond 1536 keys per
// head; shorter head-128 sequences and head size 256 run on the 64-key-tile
// kernel (prefill_k64_sm103a.cuh).
//
// The kernel is persistent: one CTA per SM walks a list of work items, each
// 256 query rows of one (b, h): two 128-row sub-tiles that take turns on the
// tensor core, so that the softmax of one overlaps the MMAs of the other.
// Items are handed out heaviest first (causal work grows with the query
// block) in "snake" order over the CTAs (a CTA with only two items takes the
// lighter one first), and the TMA producer runs ahead into the next item
// (its Q and K/V tiles) while the current one finishes.
// Roles (384 threads):
//   warps 0-3  softmax + epilogue of sub-tile 0 (thread t owns row t, TMEM lane t;
//              each warp writes its 32 output rows with bulk tensor stores)
//   warps 4-7  softmax + epilogue of sub-tile 1
//   warp  8    TMEM allocation; issues the MMAs of sub-tile 0
//   warp  9    one thread issues every TMA load (Q per item, then K/V tiles)
//   warp  10   issues the MMAs of sub-tile 1
// A tcgen05.mma is accepted only about as fast as the tensor core executes
// it, so time an issuing thread spends waiting on a barrier is tensor time
// lost.  Two issuers, each owning one sub-tile's chain S(j) -> softmax ->
// P.V(j) -> S(j+1), alternate MMA groups; in-order issue within a thread
// keeps S(j+1) from overwriting P(j) too early.
// With three warps on some SM sub-partitions, 168 registers per thread is the
// most an 11-warp CTA gets; the softmax keeps a 128-score row plus a few
// running values live within that.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+DH),
// O1 [384,384+DH).  P (bf16) is written over the first 64 columns of its S
// and fed to the P.V MMA straight from TMEM.
#pragma once

#include "sm103a_ptx.cuh"

namespace chs {

// Exact division of a non-negative int n < 2^31 by a fixed divisor d >= 1:
// n / d == (n * m) >> (31 + l) with l = ceil(log2 d) and m = ceil(2^(31+l) / d)
// (the rounding error n*(m*d - 2^(31+l)) / (d * 2^(31+l)) stays below 1/d).
// The multiplier is made on the host; the device pays one wide multiply
// instead of a division sequence.
struct FastDiv {
  uint32_t m, shift, d;
  __device__ __forceinline__ int div(int n) const {
    return (int)(((uint64_t)(uint32_t)n * m) >> shift);
  }
  __device__ __forceinline__ int mod(int n) const { return n - div(n) * (int)d; }
};

struct PrefillParams {
  int B, Hq, Hkv;
  int Sq;       // query rows per (b, h): the chunk
  int Skv;      // keys visible to the chunk's last query: start position + Sq
  int q_off;    // absolute position of query row 0 (the chunk's start position)
  int causal;   // 1: key j visible to query i only if j <= i
  int window;   // > 0: also only if i - j < window
  float scale_log2;   // softmax scale * log2(e)
  int num_qblocks;    // ceil(Sq / 256)
  int num_items;      // work items: num_qblocks * B * Hq
  float* lse;         // optional [B, Hq, Sq]: log sum_j exp(s_ij) per row (natural log)
  int* error_word;    // set to a nonzero status when a wait gives up
  int fault;          // test hook: 1 = the first K tile is never loaded
  FastDiv div_bh;     // by B * Hq (work items per query block)
  FastDiv div_hq;     // by Hq
  FastDiv div_group;  // by Hq / Hkv (query heads per K/V head)
};

template <int DH>
struct PrefillCfg {
  static_assert(DH == 64 || DH == 128, "head size 64 or 128");
  static constexpr int kRows = 128;                  // rows per sub-tile (MMA M)
  static constexpr int kKeys = 128;                  // keys per K/V tile
  static constexpr int kHalves = DH / 64;            // 128-byte swizzle boxes across DH
  static constexpr int kBoxBytes = 128 * 64 * 2;     // one 128 x 64 bf16 box
  static constexpr int kTileBytes = kHalves * kBoxBytes;
  static constexpr int kStagesK = DH == 128 ? 2 : 4;
  static constexpr int kStagesV = DH == 128 ? 2 : 4;
  static constexpr int kThreads = 384;   // 12 warps: three warpgroups
  // Registers per thread after the warpgroups rebalance (setmaxnreg): the
  // control warpgroup (warps 8-11) drops to kRegsControl, the two softmax
  // warpgroups rise to kRegsSoftmax.  The sum stays within the launch's
  // 384 x kRegsLaunch registers (the launcher checks the compiled count).
  static constexpr int kRegsLaunch = 168, kRegsControl = 80, kRegsSoftmax = 208;
  static_assert(4 * kRegsControl + 8 * kRegsSoftmax <= 12 * kRegsLaunch, "register split");
  static constexpr int kWarpProducer = 9;
  // warp issuing the MMAs of sub-tile s: 8 + 2 s (different sub-partitions)
  static constexpr int kWarpIssuer0 = 8, kWarpIssuer1 = 10;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
};

template <int DH>
struct __align__(1024) PrefillSmem {
  using Cfg = PrefillCfg<DH>;
  uint8_t q[2][Cfg::kTileBytes];          // Q sub-tiles of the current item
  uint8_t k[Cfg::kStagesK][Cfg::kTileBytes];
  uint8_t v[Cfg::kStagesV][Cfg::kTileBytes];
  // per softmax warp: its 32 output rows x 64 columns of bf16, 128-byte
  // swizzled (the layout of one box of the output's tensor map)
  uint8_t ostage[8][32 * 128];
  uint64_t q_full[2], q_empty[2];       // Q sub-tile s loaded / its last S MMA done
  uint64_t k_full[Cfg::kStagesK], k_empty[Cfg::kStagesK];
  uint64_t v_full[Cfg::kStagesV], v_empty[Cfg::kStagesV];
  uint64_t s_full[2], p_full[2], o_final[2], mma_done[2];
  uint32_t tmem_base;
  int abort_flag;
  int groups_done[2];   // MMA groups each issuer has issued (orders the two issuers)
};

// Geometry of one work item.  Query rows are counted within the chunk
// (0..Sq-1); their positions in the sequence, which the masks compare with
// key positions, are q_off higher.
struct PrefillTile {
  int q0;        // first query row of the item
  int lo, hi;    // K/V tile range loaded (union over the two sub-tiles)
  int Sq, Skv, q_off, causal, window;
  __device__ __forceinline__ int row_first(int s) const { return q0 + 128 * s; }
  __device__ __forceinline__ int pos_first(int s) const { return q_off + q0 + 128 * s; }
  __device__ __forceinline__ int pos_last(int s) const {
    return q_off + min(q0 + 128 * s + 127, Sq - 1);
  }
  __device__ __forceinline__ bool valid(int s) const { return q0 + 128 * s < Sq; }
  // does sub-tile s see any key of tile j?
  __device__ __forceinline__ bool active(int s, int j) const {
    if (!valid(s)) return false;
    const int c0 = 128 * j, c1 = min(128 * j + 127, Skv - 1);
    if (causal && c0 > pos_last(s)) return false;
    if (window > 0 && c1 < pos_first(s) - window + 1) return false;
    return true;
  }
  // offset from lo of the last tile sub-tile s sees (s must be valid)
  __device__ __forceinline__ int last_group(int s) const {
    return (causal ? min(hi, pos_last(s) / 128) : hi) - lo;
  }
  // is any (row, key) pair of sub-tile s x tile j masked?
  __device__ __forceinline__ bool needs_mask(int s, int j) const {
    const int c0 = 128 * j, c1 = 128 * j + 127;
    if (c1 >= Skv) return true;
    if (causal && c1 > pos_first(s)) return true;
    if (window > 0 && c0 < pos_last(s) - window + 1) return true;
    return false;
  }
};

__device__ __forceinline__ PrefillTile prefill_tile_of(const PrefillParams& p, int qb) {
  PrefillTile t;
  t.q0 = qb * 256;
  t.Sq = p.Sq;
  t.Skv = p.Skv;
  t.q_off = p.q_off;
  t.causal = p.causal;
  t.window = p.window;
  const int nkv = (p.Skv + 127) / 128;
  const int last_pos = p.q_off + min(t.q0 + 255, p.Sq - 1);
  t.hi = p.causal ? min(nkv - 1, last_pos / 128) : nkv - 1;
  t.lo = (p.causal && p.window > 0) ? max(0, p.q_off + t.q0 - p.window + 1) / 128 : 0;
  return t;
}

// Spin (bounded, abort-aware) until *p >= v; returns false on abort/timeout.
__device__ __forceinline__ bool spin_until_ge(volatile int* p, int v, volatile int* abort) {
  if (*p >= v) return true;
  const uint64_t t0 = globaltimer_ns();
  while (*p < v) {
    __nanosleep(20);   // leave issue slots to the softmax warps of this sub-partition
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Work item k of CTA c among G CTAs.  Items are numbered heaviest first
// (query block descending, then (b, h)); round k of the CTAs takes items
// [kG, (k+1)G) in forward order when k is even and backward when odd, so a
// CTA that drew a heavy item in one round draws a light one in the next.
__device__ __forceinline__ int prefill_item(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// The k-th work item of this CTA (num_items or more: none left).  When the
// CTAs have at most two items each (short sequences), a CTA takes its items
// lightest first: the short item's latency-bound chain (its loads, masked
// diagonal tiles and epilogue) then overlaps the start of the long one,
// instead of running alone at the end of the launch.  With more items per
// CTA the heaviest-first order is kept (its tail is the lightest items).
__device__ __forceinline__ int prefill_cta_item(int k, int num_items) {
  const int G = gridDim.x, c = blockIdx.x;
  if (num_items > 2 * G) return prefill_item(k, c, G);
  const int n = num_items > G ? 1 + (prefill_item(1, c, G) < num_items ? 1 : 0) : 1;
  return k < n ? prefill_item(n - 1 - k, c, G) : num_items;
}

struct PrefillItem {
  int b, h, bh, bh_kv;
  PrefillTile tile;
};

__device__ __forceinline__ PrefillItem prefill_item_of(const PrefillParams& p, int w) {
  PrefillItem it;
  const int blk = p.div_bh.div(w);
  const int qb = p.num_qblocks - 1 - blk;
  it.bh = w - blk * (int)p.div_bh.d;
  it.b = p.div_hq.div(it.bh);
  it.h = it.bh - it.b * p.Hq;
  it.bh_kv = it.b * p.Hkv + p.div_group.div(it.h);   // g(h) = floor(h / (H/G))
  it.tile = prefill_tile_of(p, qb);
  return it;
}

// Drain wait used at teardown: ignores the abort flag, bounded by time.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}


// One MMA issuer: the chain of sub-tile S (0 or 1) over all of the CTA's work
// items, run by a whole warp that stays converged; one elected lane issues
// each tcgen05 instruction.  Descriptors and tensor-memory addresses descend
// from compile-time constants, the CTA's shared-memory base and loop
// counters, so they stay in uniform registers: a tcgen05.mma is accepted
// only about as fast as the tensor core runs it, so every instruction
// between two of them is a bubble.  Wait results are made warp-uniform so
// the warp never diverges.
template <int DH, int S>
__device__ __forceinline__ void prefill_issuer(PrefillSmem<DH>& sm, const PrefillParams& p,
                                               volatile int* abort, int lane) {
  using Cfg = PrefillCfg<DH>;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, DH, false, true);
  // Descriptors are a fixed template OR'ed with (address >> 4); every
  // operand slice used below is that plus a compile-time offset, so an MMA
  // costs one 64-bit add and the issue itself.  Shared-memory addresses stay
  // below 2^18, so the offsets never carry out of the 14-bit address field.
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);                // Q, K
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kBoxBytes, 1024);   // V
  const uint64_t dq = kKmajor | (smem_u32(sm.q[S]) >> 4);
  const uint64_t dk = kKmajor | (smem_u32(sm.k[0]) >> 4);
  const uint64_t dv = kMnMajor | (smem_u32(sm.v[0]) >> 4);
  // the CTA owns all 512 columns, so its allocation starts at column 0
  constexpr uint32_t dS = S ? Cfg::kColS1 : Cfg::kColS0;
  constexpr uint32_t dO = S ? Cfg::kColO1 : Cfg::kColO0;
  // The work of each issuer is a sequence of groups: in an item with tiles
  // lo..hi, group g holds its P.V of tile lo+g-1 and its S of tile lo+g.
  // The tensor core runs
  //   S0(lo) | PV1(-) S1(lo) | PV0(lo) S0(lo+1) | PV1(lo) S1(lo+1) | ...
  // i.e. group g of sub-tile 0, then group g of sub-tile 1, then group g+1
  // of sub-tile 0, and on into the next item: each softmax runs while the
  // other sub-tile's two MMA groups keep the tensor core busy.  An issuer
  // first waits for everything of its own (V, K, then P), then for the other
  // issuer's previous group (a counter in shared memory), so the tensor core
  // idles only for that handover.  Group, K/V-ring and barrier-phase
  // counters run on across items.
  volatile int* mine = &sm.groups_done[S];
  volatile int* other = &sm.groups_done[1 - S];
  uint32_t kv_base = 0;   // K/V tiles of the earlier items
  int g_base = 0;         // groups of the earlier items
  uint32_t pph = 0, qph = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = prefill_cta_item(it, p.num_items);
    if (w >= p.num_items) break;
    const PrefillTile tile = prefill_item_of(p, w).tile;
    const int n_tiles = tile.hi - tile.lo + 1;
    const bool valid = tile.valid(S);
    // the group of this sub-tile's last S, after which its Q buffer is free
    const int last_s = valid ? tile.last_group(S) : -1;
    int n_active = 0;
    if (valid) {
      ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full[S], qph, abort));
      qph ^= 1;
      if (!ok) break;
    }
    for (int g = 0; g <= n_tiles; ++g) {
      const int gg = g_base + g;
      const bool do_pv = g >= 1 && tile.active(S, tile.lo + g - 1);
      const bool do_s = g < n_tiles && tile.active(S, tile.lo + g);
      const uint32_t vi = kv_base + (uint32_t)(g - 1), ki = kv_base + (uint32_t)g;
      const uint32_t vst = vi % Cfg::kStagesV, vph = (vi / Cfg::kStagesV) & 1u;
      const uint32_t kst = ki % Cfg::kStagesK, kph = (ki / Cfg::kStagesK) & 1u;
      // Waits ordered so that the one usually completing last (this
      // sub-tile's P, i.e. its softmax) comes last and the MMAs follow it at
      // once.  Every issuer waits for every tile before releasing it, so
      // neither can run a whole ring ahead of the other.
      if (g >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[vst], vph, abort))))
        break;
      if (g < n_tiles && !(ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[kst], kph, abort))))
        break;
      // sub-tile 0 waits for sub-tile 1's group gg-1, sub-tile 1 for sub-tile 0's group gg.
      // Sub-tile 0 starts an item's first S without waiting: it then runs on
      // the tensor core while sub-tile 1 finishes the previous item (its
      // last, masked softmax and P.V), instead of after it.
      if ((S == 1 || g > 0) &&
          !(ok = __all_sync(0xffffffffu, spin_until_ge(other, S ? gg + 1 : gg, abort))))
        break;
      if (do_pv) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_full[S], pph, abort)))) break;
        pph ^= 1;
      }
      tc_fence_after_sync();
      // The group is handed over to the other issuer two MMAs before its
      // end: the other issuer's waits and fences then overlap the last
      // MMAs of this group instead of leaving the tensor core idle.  (The
      // counter only paces the two issuers; no data passes through it.)
      auto publish = [&]() {
        if (lane == 0) *mine = gg + 1;
        __syncwarp();
      };
      if (g >= 1) {   // P.V of the previous tile
        if (do_pv) {
          // O_s (+)= P_s V: P from TMEM (8 columns = 16 keys per MMA), V MN-major.
          // The first P.V of an item overwrites O_s: the epilogue of the
          // previous item has read it, since these same softmax threads
          // published P only after that read completed.
          const uint64_t b = dv + (uint64_t)(vst * (Cfg::kTileBytes >> 4));
          mma_bf16_ts_warp(dO, dS, b, idesc_pv, n_active > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk) {
            if (kk == 6 && !do_s) publish();
            mma_bf16_ts_warp(dO, dS + kk * 8, b + kk * (2048 >> 4), idesc_pv, 1u);
          }
          ++n_active;
        }
        mma_commit_warp(&sm.v_empty[vst]);
      }
      if (g < n_tiles) {   // S of this tile
        if (do_s) {
          // S_s = Q_s K^T: K-major operands, 16 columns (32 bytes) of DH per MMA
          const uint64_t b = dk + (uint64_t)(kst * (Cfg::kTileBytes >> 4));
          mma_bf16_ss_warp(dS, dq, b, idesc_qk, 0u);
#pragma unroll
          for (int kk = 1; kk < DH / 16; ++kk) {
            if (kk == DH / 16 - 2) publish();
            const uint32_t off = ((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4;
            mma_bf16_ss_warp(dS, dq + off, b + off, idesc_qk, 1u);
          }
          mma_commit_warp(&sm.s_full[S]);
        }
        if (g == last_s) mma_commit_warp(&sm.q_empty[S]);
        mma_commit_warp(&sm.k_empty[kst]);
      }
      if (!do_s && !do_pv) publish();
    }
    if (!ok) break;
    if (n_active > 0) mma_commit_warp(&sm.o_final[S]);
    kv_base += (uint32_t)n_tiles;
    g_base += n_tiles + 1;
  }
  // nothing of this thread's may still run on the tensor core at teardown
  mma_commit_warp(&sm.mma_done[S]);
  mbar_wait_drain(&sm.mma_done[S], 0);
}

// TMA producer (one thread): per work item, Q sub-tile 0, the first K tile,
// Q sub-tile 1, then the K/V tiles in order.  A Q sub-tile is reloaded once
// its issuer's last S MMA of the previous item is done, so the next item's
// first tiles arrive while the current one finishes.
template <int DH>
__device__ __forceinline__ void prefill_producer(PrefillSmem<DH>& sm, const PrefillParams& p,
                                                 const CUtensorMap* map_q,
                                                 const CUtensorMap* map_k,
                                                 const CUtensorMap* map_v,
                                                 const PrefillItem& first,
                                                 volatile int* abort) {
  using Cfg = PrefillCfg<DH>;
  const uint64_t keep = policy_evict_last();   // K/V tiles are re-read by other CTAs
  uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
  uint32_t k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
  uint32_t nq0 = 0, nq1 = 0;   // Q loads per sub-tile so far
  bool ok = true;
  // the grid is no larger than the number of items, so every CTA has a first one
  PrefillItem item = first;
  for (int it = 0; ok; ++it) {
    const PrefillTile& tile = item.tile;
    auto load_q = [&](int s, uint32_t& n) {
      if (n > 0 && !mbar_wait(&sm.q_empty[s], (n - 1) & 1u, abort)) return false;
      // (checked builds: a query row of the chunk and a query head of the batch)
      const bool in_range = attn_check(tile.row_first(s) >= 0 && tile.row_first(s) < p.Sq &&
                                           item.bh >= 0 && item.bh < p.B * p.Hq,
                                       p.error_word);
      mbar_arrive_expect_tx(&sm.q_full[s], in_range ? (uint32_t)Cfg::kTileBytes : 0u);
      for (int hf = 0; in_range && hf < Cfg::kHalves; ++hf)
        // Q is read once: evict-first, so that it leaves the K/V tiles the
        // other query blocks of the head re-read in L2
        tma_load_3d_hint(sm.q[s] + hf * Cfg::kBoxBytes, map_q, &sm.q_full[s], hf * 64,
                         tile.row_first(s), item.bh, policy_evict_first());
      ++n;
      return true;
    };
    if (!(ok = load_q(0, nq0))) break;
    for (int j = tile.lo; j <= tile.hi; ++j) {
      // (checked builds: a key tile that starts inside the keys, of a K/V head of the batch)
      const bool in_range = attn_check(j >= 0 && 128 * j < tile.Skv && item.bh_kv >= 0 &&
                                           item.bh_kv < p.B * p.Hkv,
                                       p.error_word);
      const uint32_t bytes = in_range ? (uint32_t)Cfg::kTileBytes : 0u;
      if (!(ok = mbar_wait(&sm.k_empty[kst], kph ^ 1, abort))) break;
      if (p.fault != 1 || it != 0 || j != tile.lo) {   // (the test hook withholds one tile)
        mbar_arrive_expect_tx(&sm.k_full[kst], bytes);
        for (int hf = 0; in_range && hf < Cfg::kHalves; ++hf)
          tma_load_3d_hint(sm.k[kst] + hf * Cfg::kBoxBytes, map_k, &sm.k_full[kst], hf * 64,
                           128 * j, item.bh_kv, keep);
        k_loaded |= 1u << kst;
        k_par = (k_par & ~(1u << kst)) | (kph << kst);
      }
      if (++kst == Cfg::kStagesK) { kst = 0; kph ^= 1; }

      if (j == tile.lo && tile.valid(1) && !(ok = load_q(1, nq1))) break;

      if (!(ok = mbar_wait(&sm.v_empty[vst], vph ^ 1, abort))) break;
      mbar_arrive_expect_tx(&sm.v_full[vst], bytes);
      for (int hf = 0; in_range && hf < Cfg::kHalves; ++hf)
        tma_load_3d_hint(sm.v[vst] + hf * Cfg::kBoxBytes, map_v, &sm.v_full[vst], hf * 64,
                         128 * j, item.bh_kv, keep);
      v_loaded |= 1u << vst;
      v_par = (v_par & ~(1u << vst)) | (vph << vst);
      if (++vst == Cfg::kStagesV) { vst = 0; vph ^= 1; }
    }
    // decode the next item while this one's copies are in flight
    const int w = prefill_cta_item(it + 1, p.num_items);
    if (w >= p.num_items) break;
    item = prefill_item_of(p, w);
  }
  // every copy this thread started has landed before the CTA may exit
  if (nq0 > 0) mbar_wait_drain(&sm.q_full[0], (nq0 - 1) & 1u);
  if (nq1 > 0) mbar_wait_drain(&sm.q_full[1], (nq1 - 1) & 1u);
  for (int i = 0; i < Cfg::kStagesK; ++i)
    if (k_loaded & (1u << i)) mbar_wait_drain(&sm.k_full[i], (k_par >> i) & 1u);
  for (int i = 0; i < Cfg::kStagesV; ++i)
    if (v_loaded & (1u << i)) mbar_wait_drain(&sm.v_full[i], (v_par >> i) & 1u);
}

// Softmax and epilogue of sub-tile s: thread t owns query row t of the
// sub-tile (TMEM lane t) in every work item.  Per visible key tile: the
// online softmax of "Online normalizer calculation for softmax" with a lazy
// maximum; per item: O / l written straight from registers to global memory.
template <int DH>
__device__ __forceinline__ void prefill_softmax(PrefillSmem<DH>& sm, const PrefillParams& p,
                                                const CUtensorMap* map_o, uint32_t tbase,
                                                volatile int* abort, int warp, int lane) {
  using Cfg = PrefillCfg<DH>;
  const int s = warp / 4;                 // sub-tile
  const int wl = warp % 4;                // warp within the warpgroup = TMEM lane quarter
  const int t = wl * 32 + lane;           // row within the sub-tile = TMEM lane
  const uint32_t lane_addr = tbase + ((uint32_t)(wl * 32) << 16);
  const uint32_t colS = lane_addr + (s ? Cfg::kColS1 : Cfg::kColS0);
  const uint32_t colO = lane_addr + (s ? Cfg::kColO1 : Cfg::kColO0);
  const float sl2 = p.scale_log2;
  uint32_t ph = 0;   // bit 0: s_full phase, bit 1: o_final phase
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = prefill_cta_item(it, p.num_items);
    if (w >= p.num_items) break;
    const PrefillTile tile = prefill_item_of(p, w).tile;
    if (!tile.valid(s)) continue;           // a ragged last block: no rows here
    const int row = tile.pos_first(s) + t;  // this thread's query position

    float m_run = -INFINITY;   // running max of scale*log2e*score (lazily updated)
    float l_run = 0.f;         // running sum of exp2(x - m_run)
    for (int j = tile.lo; j <= tile.hi; ++j) {
      if (!tile.active(s, j)) continue;
      if (!(ok = mbar_wait(&sm.s_full[s], ph & 1u, abort))) break;
      ph ^= 1u;
      tc_fence_after_sync();

      if (tile.needs_mask(s, j)) {
        // A boundary crosses this tile: overwrite the scores of the keys this
        // row may not see with -inf in tensor memory, so the loads below and
        // everything after them are those of an unmasked tile.  Visible keys
        // of this row: [klo, khi] (absolute), as column offsets [clo, chi];
        // column c is kept iff c - clo, as unsigned, is <= chi - clo (an
        // empty range moves clo past every column).  A 32-column chunk that
        // every row of the warp sees is left alone, one that none sees is
        // filled without being read; only mixed chunks are read and masked
        // (a predicated select, never a branch).  A rolled loop keeps this
        // rarely run code small.
        const int kv0 = 128 * j;
        int khi = tile.Skv - 1;
        if (tile.causal) khi = min(khi, row);
        const int klo = tile.window > 0 ? row - tile.window + 1 : 0;
        int clo = klo - kv0;
        const int chi = khi - kv0;
        const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
        if (chi < clo) clo = 1 << 30;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          if (__all_sync(0xffffffffu, c0 >= clo && c0 + 31 <= chi)) continue;
          uint32_t y[32];
          if (__all_sync(0xffffffffu, c0 + 31 < clo || c0 > chi)) {
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = 0xff800000u;   // -inf
          } else {
            tmem_ld_32x32b_x32(colS + c0, y);
            tmem_ld_wait(y);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              y[e] = __float_as_uint(keep_if_le(__uint_as_float(y[e]), (uint32_t)(c0 + e - clo), span));
          }
          tmem_st_32x32b_x32(colS + c0, y);
        }
        tmem_st_wait();
      }

      // scores, with each 32-column chunk's maximum from the load itself
      uint32_t r0[32], r1[32], r2[32], r3[32];
      float mc0, mc1, mc2, mc3;
      tmem_ld_max_32x32b_x32(colS + 0, r0, mc0);
      tmem_ld_max_32x32b_x32(colS + 32, r1, mc1);
      tmem_ld_max_32x32b_x32(colS + 64, r2, mc2);
      tmem_ld_max_32x32b_x32(colS + 96, r3, mc3);
      tmem_ld_wait(r0, mc0);
      tmem_ld_wait(r1, mc1);
      tmem_ld_wait(r2, mc2);
      tmem_ld_wait(r3, mc3);
      float x[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(r0[c]);
        x[32 + c] = __uint_as_float(r1[c]);
        x[64 + c] = __uint_as_float(r2[c]);
        x[96 + c] = __uint_as_float(r3[c]);
      }
      const float mt = fmaxf(fmaxf(mc0, mc1), fmaxf(mc2, mc3));
      const float m_tile = mt * sl2;
      // lazy rescale: keep the old maximum unless the new one exceeds it by
      // more than 8 (weights stay <= 2^8); the result is exact either way
      // because O and l are divided by the same sum at the end.  While
      // m_run is -inf every weight so far was 0 (O and l are 0), so no
      // rescale is needed; that also covers the item's first tile, whose
      // first P.V overwrites O.
      const float m_new = fmaxf(m_run, m_tile);
      const bool fresh = m_run == -INFINITY;
      const bool upd = fresh || (m_new > m_run + 8.0f);
      const float m_use = upd ? m_new : m_run;
      const float corr = (upd && !fresh) ? ex2_approx(m_run - m_new) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      // P = exp2(x - m) as bf16 over the first 64 columns of S (the scores
      // die here, before O is touched, to keep register pressure down)
      // (pairs of columns go through packed f32x2 arithmetic)
      const float2 scale2 = make_float2(sl2, sl2), neg_m2 = make_float2(-msub, -msub);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // four partial sums
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 xs = __ffma2_rn(make_float2(x[32 * c4 + 2 * e], x[32 * c4 + 2 * e + 1]),
                                       scale2, neg_m2);
          const float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
          ls[e & 1] = __fadd2_rn(ls[e & 1], pp);
          pk[e] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st_32x32b_x16(colS + 16 * c4, pk);
      }
      const float lsum = (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
      // a raised maximum rescales this row's O (all earlier P.V are done:
      // the S MMA just waited for was issued after them)
      if (__any_sync(0xffffffffu, corr != 1.0f)) {
#pragma unroll 1
        for (int c = 0; c < DH / 16; ++c) {
          uint32_t o[16];
          tmem_ld_32x32b_x16(colO + 16 * c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st_32x32b_x16(colO + 16 * c, o);
        }
      }
      l_run = l_run * corr + lsum;
      m_run = m_use;
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sm.p_full[s]);
    }
    if (!ok) break;

    // ---- epilogue: O / l -> bf16 -> the output.  Each warp stages its 32
    // rows, 64 columns at a time, in shared memory in the 128-byte swizzled
    // layout of one box of the output's tensor map (16-byte stores, no bank
    // conflicts), and one lane writes the box with a bulk tensor store.  The
    // global write is then one asynchronous copy per warp and 64 columns
    // instead of 32-byte stores to 32 rows per instruction, which kept the
    // load/store pipeline (and the barrier waits of the other roles, which
    // go through it) busy for about a microsecond per item.
    if (!(ok = mbar_wait(&sm.o_final[s], (ph >> 1) & 1u, abort))) break;
    ph ^= 2u;
    tc_fence_after_sync();
    const float inv_l = 1.0f / l_run;
    const int bh = p.div_bh.mod(w);
    const int orow = tile.row_first(s) + t;  // output row within the chunk
    // sum_j exp(s_ij) = 2^m_run * l_run (m_run in units of log2)
    if (p.lse != nullptr && orow < p.Sq)
      p.lse[(size_t)bh * p.Sq + orow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
    const uint32_t stage = smem_u32(sm.ostage[warp]);
#pragma unroll
    for (int h = 0; h < Cfg::kHalves; ++h) {
      uint32_t o0[32], o1[32];
      tmem_ld_32x32b_x32(colO + 64 * h, o0);
      tmem_ld_32x32b_x32(colO + 64 * h + 32, o1);
      // the previous bulk store from this stage has read it
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
      tmem_ld_wait(o0);
      tmem_ld_wait(o1);
#pragma unroll
      for (int c = 0; c < 8; ++c) {   // 16-byte chunk c: columns 8c .. 8c+7 of these 64
        const uint32_t* x8 = c < 4 ? o0 + 8 * c : o1 + 8 * (c - 4);
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[e] = pack_bf16x2(__uint_as_float(x8[2 * e]) * inv_l,
                             __uint_as_float(x8[2 * e + 1]) * inv_l);
        st_shared_v4(stage + lane * 128 + ((c ^ (lane & 7)) << 4), v[0], v[1], v[2], v[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      // rows past the end of the chunk are clipped by the tensor map
      if (lane == 0) {
        // (evict-first: the output is not read again by this kernel)
        tma_store_3d_hint(map_o, sm.ostage[warp], 64 * h, tile.row_first(s) + 32 * wl, bh,
                          policy_evict_first());
        bulk_commit_group();
      }
    }
    // the next item's first P.V may overwrite O_s once these reads are done:
    // the arrive on p_full that allows it follows tcgen05.wait::ld above
  }
  // the staged rows must be written out before the CTA's shared memory goes
  if (lane == 0) bulk_wait_group0();
}

template <int DH>
__global__ void __launch_bounds__(384, 1)
    attn_prefill_sm103a(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_o, const PrefillParams p) {
  using Cfg = PrefillCfg<DH>;
  using Smem = PrefillSmem<DH>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  volatile int* abort = &sm.abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- setup (once per CTA; every barrier then runs on across work items)
  // The producer decodes its first item and prefetches the tensor maps
  // first: the parameter reads and the integer divisions then overlap the
  // barrier set-up and the tensor-memory allocation.
  PrefillItem first{};
  if (warp == Cfg::kWarpProducer && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_o);
    first = prefill_item_of(p, prefill_cta_item(0, p.num_items));
  }
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    sm.groups_done[0] = 0;
    sm.groups_done[1] = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], 128);
      mbar_init(&sm.o_final[s], 1);
      mbar_init(&sm.mma_done[s], 1);
    }
    // a K/V stage is free once both issuers' MMAs reading it are done
    for (int i = 0; i < Cfg::kStagesK; ++i) { mbar_init(&sm.k_full[i], 1); mbar_init(&sm.k_empty[i], 2); }
    for (int i = 0; i < Cfg::kStagesV; ++i) { mbar_init(&sm.v_full[i], 1); mbar_init(&sm.v_empty[i], 2); }
    fence_mbarrier_init();
  }
  if (warp == 8) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Set-up touched only shared memory, tensor memory and the parameters:
  // global memory waits for the previous kernel in the stream (a no-op
  // unless this launch is a programmatic dependent).  One CTA per SM holds
  // all of its registers and shared memory, so the next kernel, which may
  // now be launched, cannot take resources from this grid.
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tbase = sm.tmem_base;
  // all 512 columns are this CTA's, so the allocation starts at column 0;
  // the MMA issuers rely on that (compile-time tensor-memory addresses)
  // Warpgroup-wide register rebalance (every warp of a warpgroup executes
  // it), inside each role's branch so that the compiler gives the softmax
  // code the larger budget.
  if (tbase != 0 && threadIdx.x == 0) sm.abort_flag = 1;
  if (warp >= 8) {
    setmaxnreg_dec<Cfg::kRegsControl>();
    if (tbase == 0) {
      if (warp == Cfg::kWarpProducer) {
        if (lane == 0) prefill_producer<DH>(sm, p, &map_q, &map_k, &map_v, first, abort);
      } else if (warp == Cfg::kWarpIssuer0) {
        prefill_issuer<DH, 0>(sm, p, abort, lane);
      } else if (warp == Cfg::kWarpIssuer1) {
        prefill_issuer<DH, 1>(sm, p, abort, lane);
      }
    }
  } else {
    setmaxnreg_inc<Cfg::kRegsSoftmax>();
    if (tbase == 0) prefill_softmax<DH>(sm, p, &map_o, tbase, abort, warp, lane);
  }

  // ---- teardown (every thread gets here; all waits above are bounded)
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
}

template <int DH>
constexpr size_t prefill_smem_bytes() {
  return sizeof(PrefillSmem<DH>) + 1024;   // + alignment slack
}

}  // namespace chs
