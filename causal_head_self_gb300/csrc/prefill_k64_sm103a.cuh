// prefill_k64_sm103a.cuh -- causal prefill with one 128-row sub-tile per
// work item and 64-key tiles, on the 5th-generation tensor cores (sm_103a).
// Two instances:
//
//   Dh = 256 (the Gemma head size).  The accumulator O of one 128-row
//   sub-tile takes 256 of the 512 tensor-memory columns, so the two-sub-tile
//   ping-pong (prefill_sm103a.cuh) does not fit.  One CTA per SM: Q
//   (64 KiB), a two-stage K ring and a three-stage V ring of 32 KiB tiles
//   (224 KiB; the third V stage lets a V tile load while the two P.V before
//   it run); tensor memory S0 [0,64), S1 [64,128), Q [128,256), O [256,512).
//   Q is copied from shared into tensor memory once per item (tcgen05.cp)
//   and the S MMAs take it from there: with both operands in shared memory
//   an N = 64 MMA reads 6 KiB per 128 x 64 x 16 step, more than shared
//   memory delivers in the step's tensor-core time; with Q in tensor memory
//   it reads 2 KiB.
//
//   Dh = 128, short sequences.  Two CTAs per SM, each with half of the
//   shared memory (Q 32 KiB, two-stage K and V rings of 16 KiB tiles, a
//   4 KiB output staging tile per softmax warp) and half of the tensor
//   memory (S0 [0,64), S1 [64,128), O [128,256) from its allocation's base).
//   When every CTA has only one or two short items, the fixed cost of an
//   item (its first loads, the masked diagonal tiles, the epilogue)
//   dominates the ping-pong kernel's time; here the other CTA on the SM keeps
//   the tensor core busy through it.  The output leaves through bulk tensor
//   stores from the staging tiles.
//
// S is double-buffered, so the S MMA of the next key tile runs while the
// softmax works on the current one.  P (bf16) is written over the first 32
// columns of its S buffer and read from there by the P.V MMA.
//
// The kernel is persistent (CTAs walk 128-row items, heaviest first) with the
// roles of the ping-pong kernel (prefill_sm103a.cuh): one thread issues every
// TMA load, one warp issues every MMA, four warps run the softmax and the
// epilogue (thread t owns row t).  Masks, the lazy maximum and the
// chunked-prefill offset follow that kernel.  Every wait is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103a_ptx.cuh"

namespace chs {

struct PrefillK64Params {
  int B, Hq, Hkv;
  int Sq, Skv, q_off;   // as in the ping-pong kernel
  int causal, window;
  float scale_log2;
  int num_qblocks;      // ceil(Sq / 128)
  int num_items;        // num_qblocks * B * Hq
  int per_qb;           // B * Hq
  int group;            // Hq / Hkv
  __nv_bfloat16* o;     // [B, Hq, Sq, Dh]
  int o_wide;           // o is 32-byte aligned: 32-byte stores
  float* lse;           // optional [B, Hq, Sq]: log sum_j exp(s_ij) per row (natural log)
  int* error_word;
  int fault;            // test hook: 1 = the first K tile is never loaded
};

template <int DH_>
struct PrefillK64Cfg {
  static_assert(DH_ == 128 || DH_ == 256, "head size 128 or 256");
  static constexpr int DH = DH_;
  static constexpr int kBoxes = DH / 64;               // 64-column boxes per row
  static constexpr int kKeys = 64;                     // keys per tile
  static constexpr int kQBox = 128 * 64 * 2;           // Q box: 128 rows x 64 columns
  static constexpr int kKBox = kKeys * 64 * 2;         // K/V box: 64 rows x 64 columns
  static constexpr int kQBytes = kBoxes * kQBox;       // 32 / 64 KiB
  static constexpr int kTileBytes = kBoxes * kKBox;    // 16 / 32 KiB
  static constexpr int kStagesK = 2;   // K tiles: S(t) is issued two tiles ahead
  // V tiles: at Dh 256 a third stage hides the load behind two P.V
  static constexpr int kStagesV = DH == 256 ? 3 : 2;
  static constexpr int kCtasPerSm = DH == 256 ? 1 : 2;
  static constexpr uint32_t kTmemCols = DH == 256 ? 512 : 256;   // this CTA's allocation
  static constexpr int kThreads = 192;   // warps 0-3 softmax, 4 producer, 5 MMA issuer
  static constexpr int kWarpProducer = 4, kWarpIssuer = 5;
  // S buffer b at kColS + 64 b, O in the allocation's last DH columns
  static constexpr uint32_t kColS = 0, kColO = kTmemCols - DH;
  // Dh 128: the output goes through shared memory and bulk tensor stores
  // (32 rows x 64 columns per box and softmax warp).  Dh 256 has no shared
  // memory left for it and stores from registers.
  static constexpr bool kTmaStore = DH == 128;
  static constexpr int kStageBytes = kTmaStore ? 4 * 32 * 128 : 0;
  // Two CTAs and their shared memory fit an SM only without the 1 KiB
  // alignment slack: that instance takes the dynamic shared memory as placed
  // (1024-byte aligned, which the kernel checks).
  static constexpr int kAlignSlack = kTmaStore ? 0 : 1024;
  // Dh 256: Q is copied into tensor memory [128, 256) once per item and the S
  // MMAs read it there, so that they stream only K from shared memory
  static constexpr bool kQInTmem = DH == 256;
  static constexpr uint32_t kColQ = 128;
};

// Every array is a whole number of KiB, so each starts 1024-byte aligned once
// the structure does (the 128-byte swizzle repeats every 1024 bytes).
template <int DH>
struct PrefillK64Smem {
  using Cfg = PrefillK64Cfg<DH>;
  uint8_t q[Cfg::kQBytes];
  uint8_t k[Cfg::kStagesK][Cfg::kTileBytes];
  uint8_t v[Cfg::kStagesV][Cfg::kTileBytes];
  // per softmax warp (Dh 128): its 32 output rows x 64 columns of bf16,
  // 128-byte swizzled (the layout of one box of the output's tensor map)
  uint8_t ostage[Cfg::kStageBytes > 0 ? Cfg::kStageBytes : 1];
  uint64_t q_full, q_empty;
  uint64_t k_full[Cfg::kStagesK], k_empty[Cfg::kStagesK];
  uint64_t v_full[Cfg::kStagesV], v_empty[Cfg::kStagesV];
  uint64_t s_full[2], p_full[2], pv_done, o_final, mma_done;
  uint64_t qt_free;   // (Q in tensor memory) the item's last S MMA is done
  uint32_t tmem_base;
  int abort_flag;
};

// Geometry of one 128-row work item: query rows [q0, q0 + 128) of the chunk,
// at positions q_off + row; key tiles lo..hi of 64 keys.
struct PrefillK64Tile {
  int q0, lo, hi;
  int bh, bh_kv;
  __device__ __forceinline__ int pos_first(const PrefillK64Params& p) const { return p.q_off + q0; }
  __device__ __forceinline__ int pos_last(const PrefillK64Params& p) const {
    return p.q_off + min(q0 + 127, p.Sq - 1);
  }
  // is any (row, key) pair of tile j masked?
  __device__ __forceinline__ bool needs_mask(const PrefillK64Params& p, int j) const {
    const int c0 = 64 * j, c1 = 64 * j + 63;
    if (c1 >= p.Skv) return true;
    if (p.causal && c1 > pos_first(p)) return true;
    if (p.window > 0 && c0 < pos_last(p) - p.window + 1) return true;
    return false;
  }
};

// Item w: heaviest query blocks first (causal work grows with the block),
// dealt to the CTAs in snake order (see the ping-pong kernel).
__device__ __forceinline__ int prefill_k64_item(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// The k-th work item of this CTA (num_items or more: none left).  With at
// most two items per CTA the lighter one goes first, as in the ping-pong
// kernel: its latency-bound chain then overlaps the start of the long item.
__device__ __forceinline__ int prefill_k64_cta_item(int k, int num_items) {
  const int G = gridDim.x, c = blockIdx.x;
  if (num_items > 2 * G) return prefill_k64_item(k, c, G);
  const int n = num_items > G ? 1 + (prefill_k64_item(1, c, G) < num_items ? 1 : 0) : 1;
  return k < n ? prefill_k64_item(n - 1 - k, c, G) : num_items;
}

__device__ __forceinline__ PrefillK64Tile prefill_k64_tile_of(const PrefillK64Params& p, int w) {
  PrefillK64Tile t;
  const int blk = w / p.per_qb;
  const int qb = p.num_qblocks - 1 - blk;
  t.bh = w - blk * p.per_qb;
  const int b = t.bh / p.Hq, h = t.bh - (t.bh / p.Hq) * p.Hq;
  t.bh_kv = b * p.Hkv + h / p.group;   // g(h) = floor(h / (H/G))
  t.q0 = qb * 128;
  const int nkv = (p.Skv + 63) / 64;
  const int last_pos = p.q_off + min(t.q0 + 127, p.Sq - 1);
  t.hi = p.causal ? min(nkv - 1, last_pos / 64) : nkv - 1;
  t.lo = (p.causal && p.window > 0) ? max(0, p.q_off + t.q0 - p.window + 1) / 64 : 0;
  return t;
}

__device__ __forceinline__ void mbar_wait_drain_k64(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// TMA producer (one thread): per item, Q (Dh/64 boxes of 128 x 64) once its
// previous item's last S is done, then the item's K and V tiles (Dh/64 boxes
// of 64 x 64 each) through the K and V rings.
template <int DH>
__device__ __forceinline__ void prefill_k64_producer(PrefillK64Smem<DH>& sm, const PrefillK64Params& p,
                                                    const CUtensorMap* map_q,
                                                    const CUtensorMap* map_k,
                                                    const CUtensorMap* map_v,
                                                    volatile int* abort) {
  using Cfg = PrefillK64Cfg<DH>;
  const uint64_t keep = policy_evict_last();   // K/V tiles are re-read by other items
  uint32_t t = 0;                              // K/V tiles loaded so far
  uint32_t k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
  int nq = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = prefill_k64_cta_item(it, p.num_items);
    if (w >= p.num_items) break;
    const PrefillK64Tile tile = prefill_k64_tile_of(p, w);
    if (nq > 0 && !(ok = mbar_wait(&sm.q_empty, (uint32_t)(nq - 1) & 1u, abort))) break;
    // (checked builds: a query row of the chunk and a query head of the batch)
    const bool q_in_range = attn_check(tile.q0 >= 0 && tile.q0 < p.Sq && tile.bh >= 0 &&
                                           tile.bh < p.B * p.Hq,
                                       p.error_word);
    mbar_arrive_expect_tx(&sm.q_full, q_in_range ? (uint32_t)Cfg::kQBytes : 0u);
    for (int hf = 0; q_in_range && hf < Cfg::kBoxes; ++hf)
      // (read once: evict-first, leaving L2 to the K/V tiles that are re-read)
      tma_load_3d_hint(sm.q + hf * Cfg::kQBox, map_q, &sm.q_full, hf * 64, tile.q0, tile.bh,
                       policy_evict_first());
    ++nq;
    for (int j = tile.lo; j <= tile.hi; ++j, ++t) {
      const int st = (int)(t % Cfg::kStagesK);
      const uint32_t ph = (t / Cfg::kStagesK) & 1u;
      // (checked builds: a key tile that starts inside the keys, of a K/V head of the batch)
      const bool in_range = attn_check(j >= 0 && 64 * j < p.Skv && tile.bh_kv >= 0 &&
                                           tile.bh_kv < p.B * p.Hkv,
                                       p.error_word);
      const uint32_t bytes = in_range ? (uint32_t)Cfg::kTileBytes : 0u;
      if (!(ok = mbar_wait(&sm.k_empty[st], ph ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.k_full[st], bytes);
      if (p.fault != 1 || it != 0 || j != tile.lo) {   // (the test hook withholds one tile)
        for (int hf = 0; in_range && hf < Cfg::kBoxes; ++hf)
          tma_load_3d_hint(sm.k[st] + hf * Cfg::kKBox, map_k, &sm.k_full[st], hf * 64, 64 * j,
                           tile.bh_kv, keep);
      }
      k_loaded |= 1u << st;
      k_par = (k_par & ~(1u << st)) | (ph << st);
      const int sv = (int)(t % Cfg::kStagesV);
      const uint32_t pv = (t / Cfg::kStagesV) & 1u;
      if (!(ok = mbar_wait(&sm.v_empty[sv], pv ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.v_full[sv], bytes);
      for (int hf = 0; in_range && hf < Cfg::kBoxes; ++hf)
        tma_load_3d_hint(sm.v[sv] + hf * Cfg::kKBox, map_v, &sm.v_full[sv], hf * 64, 64 * j,
                         tile.bh_kv, keep);
      v_loaded |= 1u << sv;
      v_par = (v_par & ~(1u << sv)) | (pv << sv);
    }
  }
  // every copy this thread started has landed before the CTA may exit
  if (nq > 0) mbar_wait_drain_k64(&sm.q_full, (uint32_t)(nq - 1) & 1u);
  for (int i = 0; i < Cfg::kStagesK; ++i)
    if (k_loaded & (1u << i)) mbar_wait_drain_k64(&sm.k_full[i], (k_par >> i) & 1u);
  for (int i = 0; i < Cfg::kStagesV; ++i)
    if (v_loaded & (1u << i)) mbar_wait_drain_k64(&sm.v_full[i], (v_par >> i) & 1u);
}

// MMA issuer (one converged warp, one elected lane per instruction).  Per
// item: S of its first two tiles, then per tile t: P.V(t) once P(t) is
// written, and S(t+2) into the buffer P(t) lived in (the tensor core runs one
// thread's MMAs in order).  The first P.V of an item overwrites O: the
// softmax threads publish that P only after their epilogue has read O.  At
// Dh 256 an item starts with the copy of Q into tensor memory; a copy issued
// after an MMA is not ordered behind it, so the copy waits (qt_free) for the
// previous item's last S MMA, which is long done by then.
template <int DH>
__device__ __forceinline__ void prefill_k64_issuer(PrefillK64Smem<DH>& sm, const PrefillK64Params& p,
                                                   uint32_t tbase, volatile int* abort) {
  using Cfg = PrefillK64Cfg<DH>;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, Cfg::kKeys, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, Cfg::DH, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);            // Q, K
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kKBox, 1024);   // V: 64-column blocks kKBox apart
  const uint64_t dq = kKmajor | (smem_u32(sm.q) >> 4);
  const uint64_t dk = kKmajor | (smem_u32(sm.k[0]) >> 4);
  const uint64_t dv = kMnMajor | (smem_u32(sm.v[0]) >> 4);
  const uint32_t dO = tbase + Cfg::kColO;
  auto issue_s = [&](uint32_t t) -> bool {
    const int st = (int)(t % Cfg::kStagesK);
    const uint32_t ph = (t / Cfg::kStagesK) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.k_full[st], ph, abort))) return false;
    tc_fence_after_sync();
    const uint32_t dS = tbase + Cfg::kColS + 64u * (t & 1u);
    const uint64_t b = dk + (uint64_t)(st * (Cfg::kTileBytes >> 4));
#pragma unroll
    for (int kk = 0; kk < Cfg::DH / 16; ++kk) {
      // 16 columns (32 bytes) of Dh per MMA; a 64-column box holds 4 steps
      const uint32_t offq = ((kk / 4) * Cfg::kQBox + (kk % 4) * 32) >> 4;
      const uint32_t offk = ((kk / 4) * Cfg::kKBox + (kk % 4) * 32) >> 4;
      if constexpr (Cfg::kQInTmem)
        mma_bf16_ts_warp(dS, tbase + Cfg::kColQ + 8 * kk, b + offk, idesc_qk, kk > 0 ? 1u : 0u);
      else
        mma_bf16_ss_warp(dS, dq + offq, b + offk, idesc_qk, kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(&sm.s_full[t & 1u]);
    mma_commit_warp(&sm.k_empty[st]);
    return true;
  };
  uint32_t t = 0;   // global tile counter
  int nq = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = prefill_k64_cta_item(it, p.num_items);
    if (w >= p.num_items) break;
    const PrefillK64Tile tile = prefill_k64_tile_of(p, w);
    const int n = tile.hi - tile.lo + 1;
    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, (uint32_t)nq & 1u, abort)))) break;
    tc_fence_after_sync();
    uint64_t* q_done = &sm.q_empty;   // arrived on when the item's last S MMA is done
    if constexpr (Cfg::kQInTmem) {
      // the previous item's S MMAs read the tensor-memory copy of Q: the copy
      // of this item's Q waits for the last of them
      if (nq > 0 &&
          !(ok = __all_sync(0xffffffffu, mbar_wait(&sm.qt_free, (uint32_t)(nq - 1) & 1u, abort))))
        break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < Cfg::DH / 16; ++kk)
        tmem_cp_128x256b_warp(tbase + Cfg::kColQ + 8 * kk,
                              dq + (((kk / 4) * Cfg::kQBox + (kk % 4) * 32) >> 4));
      // the shared-memory Q is free once the copies are done
      mma_commit_warp(&sm.q_empty);
      q_done = &sm.qt_free;
    }
    ++nq;
    if (!(ok = issue_s(t))) break;
    if (n > 1 && !(ok = issue_s(t + 1))) break;
    if (n <= 2) mma_commit_warp(q_done);   // this item's last S is issued
    for (int i = 0; ok && i < n; ++i, ++t) {
      const int st = (int)(t % Cfg::kStagesV);
      const uint32_t ph = (t / Cfg::kStagesV) & 1u;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[st], ph, abort)))) break;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_full[t & 1u], (t >> 1) & 1u, abort))))
        break;
      tc_fence_after_sync();
      // O (+)= P V: P from TMEM (8 columns = 16 keys per MMA), V MN-major
      const uint32_t dP = tbase + Cfg::kColS + 64u * (t & 1u);
      const uint64_t b = dv + (uint64_t)(st * (Cfg::kTileBytes >> 4));
#pragma unroll
      for (int kk = 0; kk < Cfg::kKeys / 16; ++kk)
        mma_bf16_ts_warp(dO, dP + kk * 8, b + kk * (2048 >> 4), idesc_pv,
                         (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit_warp(&sm.pv_done);
      mma_commit_warp(&sm.v_empty[st]);
      if (i + 2 < n) {
        if (!(ok = issue_s(t + 2))) break;
        if (i + 2 == n - 1) mma_commit_warp(q_done);
      }
    }
    if (ok) mma_commit_warp(&sm.o_final);
  }
  // nothing of this warp's may still run on the tensor core at teardown
  mma_commit_warp(&sm.mma_done);
  mbar_wait_drain_k64(&sm.mma_done, 0);
}

// Softmax and epilogue (warps 0-3; thread t owns row t of the item, TMEM lane
// t): the online softmax of "Online normalizer calculation for softmax" with
// the lazy maximum of the ping-pong kernel, 64 scores per tile.
template <int DH>
__device__ __forceinline__ void prefill_k64_softmax(PrefillK64Smem<DH>& sm, const PrefillK64Params& p,
                                                    const CUtensorMap* map_o, uint32_t tbase,
                                                    volatile int* abort, int warp, int lane) {
  using Cfg = PrefillK64Cfg<DH>;
  const int t = warp * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
  const uint32_t colO = lane_addr + Cfg::kColO;
  const float sl2 = p.scale_log2;
  uint32_t tt = 0;      // global tile counter (the issuer's t)
  uint32_t items = 0;   // items finished (o_final phases)
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = prefill_k64_cta_item(it, p.num_items);
    if (w >= p.num_items) break;
    const PrefillK64Tile tile = prefill_k64_tile_of(p, w);
    const int row = tile.pos_first(p) + t;   // this thread's query position

    float m_run = -INFINITY, l_run = 0.f;
    for (int j = tile.lo; j <= tile.hi; ++j, ++tt) {
      const uint32_t b = tt & 1u;
      const uint32_t colS = lane_addr + Cfg::kColS + 64u * b;
      if (!(ok = mbar_wait(&sm.s_full[b], (tt >> 1) & 1u, abort))) break;
      tc_fence_after_sync();

      if (tile.needs_mask(p, j)) {
        // keys this row may not see become -inf in tensor memory (as in the
        // ping-pong kernel): visible keys [klo, khi] as column offsets
        // [clo, chi] of this 64-key tile
        const int kv0 = 64 * j;
        int khi = p.Skv - 1;
        if (p.causal) khi = min(khi, row);
        const int klo = p.window > 0 ? row - p.window + 1 : 0;
        int clo = klo - kv0;
        const int chi = khi - kv0;
        const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
        if (chi < clo) clo = 1 << 30;
#pragma unroll 1
        for (int c0 = 0; c0 < Cfg::kKeys; c0 += 32) {
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

      uint32_t r0[32], r1[32];
      float mc0, mc1;
      tmem_ld_max_32x32b_x32(colS + 0, r0, mc0);
      tmem_ld_max_32x32b_x32(colS + 32, r1, mc1);
      tmem_ld_wait(r0, mc0);
      tmem_ld_wait(r1, mc1);
      const float m_tile = fmaxf(mc0, mc1) * sl2;
      const float m_new = fmaxf(m_run, m_tile);
      const bool fresh = m_run == -INFINITY;
      const bool upd = fresh || (m_new > m_run + 8.0f);
      const float m_use = upd ? m_new : m_run;
      const float corr = (upd && !fresh) ? ex2_approx(m_run - m_new) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      // P = exp2(x - m) as bf16 over the first 32 columns of this S buffer
      const float2 scale2 = make_float2(sl2, sl2), neg_m2 = make_float2(-msub, -msub);
      float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const uint32_t* r = c2 ? r1 : r0;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 xs = __ffma2_rn(
              make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), scale2, neg_m2);
          const float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
          ls[e & 1] = __fadd2_rn(ls[e & 1], pp);
          pk[e] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st_32x32b_x16(colS + 16 * c2, pk);
      }
      const float lsum = (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
      // A raised maximum rescales O, once the previous tile's P.V (the only
      // one that can still run: this S was issued after the one before it)
      // has finished.  Never on an item's first tile (fresh), so tt >= 1.
      if (__any_sync(0xffffffffu, corr != 1.0f)) {
        if (!(ok = mbar_wait(&sm.pv_done, (tt - 1u) & 1u, abort))) break;
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < Cfg::DH / 16; ++c) {
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
      mbar_arrive(&sm.p_full[b]);
    }
    if (!ok) break;

    // ---- epilogue: O / l -> bf16 -> output rows
    if (!(ok = mbar_wait(&sm.o_final, items & 1u, abort))) break;
    ++items;
    tc_fence_after_sync();
    const float inv_l = 1.0f / l_run;
    const int orow = tile.q0 + t;   // output row within the chunk
    uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)tile.bh * p.Sq + orow) * Cfg::DH);
    const bool store = orow < p.Sq;
    // sum_j exp(s_ij) = 2^m_run * l_run (m_run in units of log2)
    if (p.lse != nullptr && store)
      p.lse[(size_t)tile.bh * p.Sq + orow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
    // (the output is not read again by this kernel: evict-first, leaving L2
    // to the K/V tiles the other query blocks re-read)
    const uint64_t out_policy = policy_evict_first();
    if constexpr (Cfg::kTmaStore) {
      // 64 columns per round: TMEM -> registers -> this warp's staging tile
      // -> one bulk tensor store (rows past the chunk's end are clipped by
      // the tensor map)
      uint8_t* stg = sm.ostage + warp * (32 * 128);
      const uint32_t stage = smem_u32(stg);
#pragma unroll
      for (int h = 0; h < Cfg::kBoxes; ++h) {
        uint32_t o0[32], o1[32];
        tmem_ld_32x32b_x32(colO + 64 * h, o0);
        tmem_ld_32x32b_x32(colO + 64 * h + 32, o1);
        // the previous bulk store from this tile has read it
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
        if (lane == 0) {
          tma_store_3d_hint(map_o, stg, 64 * h, tile.q0 + 32 * warp, tile.bh, out_policy);
          bulk_commit_group();
        }
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < Cfg::DH / 32; c += 2) {
        uint32_t o0[32], o1[32];
        tmem_ld_32x32b_x32(colO + 32 * c, o0);
        tmem_ld_32x32b_x32(colO + 32 * c + 32, o1);
        tmem_ld_wait(o0);
        tmem_ld_wait(o1);
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // 16 columns each
          const uint32_t* o = q < 2 ? o0 + 16 * q : o1 + 16 * (q - 2);
          uint32_t v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            v[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
          if (store) {
            uint4* d = dst + 2 * (2 * c + q);
            if (p.o_wide) {
              st_global_v8_hint(d, v, out_policy);
            } else {
              d[0] = make_uint4(v[0], v[1], v[2], v[3]);
              d[1] = make_uint4(v[4], v[5], v[6], v[7]);
            }
          }
        }
      }
    }
    // the next item's first P.V overwrites O only after the arrive on p_full
    // that follows these loads (tcgen05.wait::ld above)
  }
  // the staged rows must be written out before the CTA's shared memory goes
  if constexpr (Cfg::kTmaStore) {
    if (lane == 0) bulk_wait_group0();
  }
}

template <int DH>
__global__ void __launch_bounds__(PrefillK64Cfg<DH>::kThreads, PrefillK64Cfg<DH>::kCtasPerSm)
    attn_prefill_k64_sm103a(const __grid_constant__ CUtensorMap map_q,
                            const __grid_constant__ CUtensorMap map_k,
                            const __grid_constant__ CUtensorMap map_v,
                            const __grid_constant__ CUtensorMap map_o,   // Dh 128 only
                            const PrefillK64Params p) {
  using Cfg = PrefillK64Cfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  if (Cfg::kAlignSlack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
    // no room to align: refuse before any barrier, copy or allocation
    if (threadIdx.x == 0) atomicExch(p.error_word, 3);   // ATTN_ERR_CUDA
    return;
  }
  PrefillK64Smem<DH>& sm = *reinterpret_cast<PrefillK64Smem<DH>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  volatile int* abort = &sm.abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (warp == Cfg::kWarpProducer && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    if (Cfg::kTmaStore) prefetch_tensormap(&map_o);
  }
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int i = 0; i < Cfg::kStagesK; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < Cfg::kStagesV; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_full[b], 128);
    }
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.o_final, 1);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.qt_free, 1);
    fence_mbarrier_init();
  }
  if (warp == Cfg::kWarpProducer) {
    tmem_alloc(&sm.tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // global memory only after the previous kernel in the stream is complete;
  // this grid (its CTAs take nearly all of the shared memory of their SMs)
  // leaves the next kernel little to take, so it may be launched now
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  // every tensor-memory address is relative to this CTA's allocation (at
  // Dh 128 two CTAs share an SM's 512 columns)
  const uint32_t tbase = sm.tmem_base;
  if (warp == Cfg::kWarpProducer) {
    if (lane == 0) prefill_k64_producer<DH>(sm, p, &map_q, &map_k, &map_v, abort);
  } else if (warp == Cfg::kWarpIssuer) {
    prefill_k64_issuer<DH>(sm, p, tbase, abort);
  } else {
    prefill_k64_softmax<DH>(sm, p, &map_o, tbase, abort, warp, lane);
  }

  // ---- teardown (every wait above is bounded)
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kWarpProducer) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
}

template <int DH>
constexpr size_t prefill_k64_smem_bytes() {
  return sizeof(PrefillK64Smem<DH>) + PrefillK64Cfg<DH>::kAlignSlack;
}

// two CTAs per SM at Dh 128 in the SM's 228 KiB (1 KiB of it reserved per CTA)
static_assert(2 * (prefill_k64_smem_bytes<128>() + 1024) <= 228 * 1024, "Dh 128: two CTAs per SM");
static_assert(prefill_k64_smem_bytes<256>() <= 227 * 1024, "Dh 256: one CTA per SM");

}  // namespace chs
