// backward256_sm103a.cuh -- backward pass of causal self-attention at head
// size 256 (the Gemma head size) on the 5th-generation tensor cores.
//
// The gradients are those of the Dh <= 128 kernels (backward_sm103a.cuh):
//     dV = P^T dO,   dS = P o (dP - D),   dK = scale dS^T Q,   dQ = scale dS K,
// with P recomputed from the saved log-sum-exp ("Механизм внимания",
// sections "Почему делить на корень из d_h" and "Эффективные реализации").
// What changes at Dh = 256 is the budget.  A 256-column accumulator takes
// half of the 512 tensor-memory columns, so dK and dV of one key block no
// longer fit beside the score and dP tiles, and a 128 x 256 bf16 tile is
// 64 KiB, so a key block, its value block and one 128-row query block with
// its dO already fill the 227 KiB of shared memory.  Hence four kernels:
//   attn_bwd_prep<256>   D and lse2 per row (the Dh <= 128 prep kernel);
//   attn_bwd256_kv<0>    dV: per 128-key block (which stays in shared
//                        memory), 64-row query blocks of every query head of
//                        the group stream past; S^T = K Q^T (M = 128 keys,
//                        N = 64 queries, K = 256), P^T written as bf16 over
//                        it, dV += P^T dO (N = 256, K = 64);
//   attn_bwd256_kv<1>    dK: K and V stay, the 64-row query blocks stream;
//                        S^T = K Q^T and dP^T = V dO^T, dS^T over dP^T,
//                        dK += dS^T Q;
//   attn_bwd256_dq       dQ: per 128-row query block (Q and dO stay),
//                        64-key blocks stream; S = Q K^T, dP = dO V^T, dS
//                        over dP, dQ += dS K.
// S (or S^T) and dP are recomputed in the passes that need them (5 MMA
// units per block pair against the 4 of a fused pass); there are no atomics
// and the result is deterministic.  Tensor memory: two score buffers
// [0, 64) and [64, 128), two dP buffers [128, 192) and [192, 256) (the dQ
// pass uses one score buffer), the accumulator [256, 512).  Columns a pass
// leaves free hold an MMA operand copied from shared memory (tcgen05.cp)
// once per item, so that its N = 64 score MMAs read less shared memory: K in
// the dV pass (at [128, 256)), the first 128 columns of Q in the dQ pass (at
// [64, 128)).  A copy is not ordered behind an MMA issued before it, so each
// copy waits for the previous item's last reader of the old copy.  Roles as in the
// Dh <= 128 kernels: two element-wise warpgroups on the two 32-column halves
// of every 64-column tile (thread t owns tensor-memory lane t), one TMA
// thread, one MMA warp.  Every wait is bounded.
#pragma once

#include "backward_sm103a.cuh"

namespace chs {

struct Bwd256Cfg {
  static constexpr int DH = 256;
  static constexpr int kBig = 128;                     // rows of an item's resident block (MMA M)
  static constexpr int kSmall = 64;                    // rows of a streamed block
  static constexpr int kBigBox = kBig * 64 * 2;        // one 128-row x 64-column box (16 KiB)
  static constexpr int kSmallBox = kSmall * 64 * 2;    // one 64-row x 64-column box (8 KiB)
  static constexpr int kBigTile = 4 * kBigBox;         // 128 x 256 (64 KiB)
  static constexpr int kSmallTile = 4 * kSmallBox;     // 64 x 256 (32 KiB)
  static constexpr int kWG = 2;                        // element-wise warpgroups
  static constexpr int kCols = kSmall / kWG;           // 32 columns of a 64-column tile each
  static constexpr int kEW = 128 * kWG;                // element-wise threads
  static constexpr int kThreads = 32 * (4 * kWG + 2);
  static constexpr int kWarpProducer = 4 * kWG, kWarpIssuer = 4 * kWG + 1;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256;   // + 64 b for buffer b
  // dV pass: K (128 keys x 256, bf16 pairs) in the unused dP columns [128, 256)
  static constexpr uint32_t kColKt = 128;
  // dQ pass: Q's first 128 columns (bf16 pairs) in the unused second score
  // buffer [64, 128)
  static constexpr uint32_t kColQt = 64;
};

// Columns of a 64-column tile hold each warpgroup's bf16 pairs in the first
// half of its own 32 columns; the pairs of columns 16 kk .. 16 kk + 15 start
// at this column (the A operand of the accumulation MMAs, read from tensor
// memory).
__host__ __device__ constexpr uint32_t bwd256_packed_col(int kk) {
  return (uint32_t)(32 * (16 * kk / 32) + (16 * kk % 32) / 2);
}

// 64-row query blocks [lo, hi] that see some key of 128-key block kb.
__device__ __forceinline__ void bwd256_qblocks_of(const BwdParams& p, int kb, int& lo, int& hi) {
  const int nq = (p.S + 63) / 64;
  lo = 0;
  hi = nq - 1;
  if (!p.causal) return;
  lo = 2 * kb;   // query i sees key j only if j <= i
  if (p.window > 0) hi = min(hi, (128 * kb + 127 + p.window - 1) / 64);   // i - j < W
}

// 64-key blocks [lo, hi] that 128-row query block qb sees.
__device__ __forceinline__ void bwd256_kblocks_of(const BwdParams& p, int qb, int& lo, int& hi) {
  const int nk = (p.S + 63) / 64;
  lo = 0;
  hi = nk - 1;
  if (!p.causal) return;
  hi = min(hi, (128 * qb + 127) / 64);
  if (p.window > 0) lo = max(0, 128 * qb - p.window + 1) / 64;
}

// ============================================================ dV and dK passes

// Stages: in the dV pass Q is read by S^T(n) alone and released after it, so
// three Q stages keep S^T two steps ahead of its loads, and the per-row
// statistics (read by the element-wise warps until P^T(n) is written) travel
// with dO, released after dV(n).  In the dK pass Q is read by S^T(n) and
// dK(n), dO by dP^T(n) alone; the statistics travel with Q.
template <bool DK>
struct __align__(1024) Bwd256KvSmem {
  using Cfg = Bwd256Cfg;
  static constexpr int kStagesQ = DK ? 2 : 3;
  static constexpr int kStagesDO = DK ? 1 : 2;
  static constexpr int kStagesStat = DK ? kStagesQ : kStagesDO;
  uint8_t k[Cfg::kBigTile];                     // this item's key block (stays)
  uint8_t q[kStagesQ][Cfg::kSmallTile];         // query blocks
  uint8_t dO[kStagesDO][Cfg::kSmallTile];       // their output gradients
  uint8_t v[DK ? Cfg::kBigTile : 16];           // the value block (dK pass; stays)
  float lse2[kStagesStat][64];                  // the blocks' log-sum-exps (log2 units)
  float dlt[kStagesStat][64];                   // their D_i
  uint64_t kv_full, kv_empty;
  uint64_t kt_free;   // (dV pass) the item's last S^T MMA, the last reader of K in tensor memory, is done
  uint64_t q_full[kStagesQ], q_empty[kStagesQ];
  uint64_t do_full[kStagesDO], do_empty[kStagesDO];
  uint64_t s_full[2], dp_full[2], p_full[2], ds_full[2], acc_final, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Item w: 128-key block kb (earliest, i.e. heaviest under a causal mask,
// first) of K/V head bkv = b * Hkv + g.
__device__ __forceinline__ BwdKvItem bwd256_kv_item_of(const BwdParams& p, int w) {
  BwdKvItem r;
  const int per = p.B * p.Hkv;
  r.kb = w / per;
  r.bkv = w - r.kb * per;
  r.b = r.bkv / p.Hkv;
  r.g = r.bkv - r.b * p.Hkv;
  bwd256_qblocks_of(p, r.kb, r.lo, r.hi);
  return r;
}

template <bool DK>
__device__ __forceinline__ void bwd256_kv_producer(Bwd256KvSmem<DK>& sm, const BwdParams& p,
                                                   const CUtensorMap* map_q,
                                                   const CUtensorMap* map_k,
                                                   const CUtensorMap* map_v,
                                                   const CUtensorMap* map_do,
                                                   volatile int* abort) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256KvSmem<DK>;
  const uint64_t keep = policy_evict_last();   // query blocks are re-read by other key blocks
  uint32_t u = 0, q_loaded = 0, q_par = 0, d_loaded = 0, d_par = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd256_kv_item_of(p, w);
    if (items > 0 && !(ok = mbar_wait(&sm.kv_empty, (uint32_t)(items - 1) & 1u, abort))) break;
    // (checked builds: a key block of the sequence, of a K/V head of the batch)
    const bool kv_in_range = attn_check(I.kb >= 0 && 128 * I.kb < p.S && I.bkv >= 0 &&
                                            I.bkv < p.B * p.Hkv,
                                        p.error_word);
    mbar_arrive_expect_tx(&sm.kv_full, kv_in_range ? (DK ? 2u : 1u) * Cfg::kBigTile : 0u);
    if (kv_in_range && (p.fault != 4 || it != 0)) {   // (the test hook withholds one K/V block)
      for (int hf = 0; hf < 4; ++hf) {
        tma_load_3d(sm.k + hf * Cfg::kBigBox, map_k, &sm.kv_full, 64 * hf, 128 * I.kb, I.bkv);
        if (DK)
          tma_load_3d(sm.v + hf * Cfg::kBigBox, map_v, &sm.kv_full, 64 * hf, 128 * I.kb, I.bkv);
      }
    }
    ++items;
    for (int hh = 0; ok && hh < p.group; ++hh) {
      const int bh = I.b * p.Hq + I.g * p.group + hh;
      for (int qb = I.lo; qb <= I.hi; ++qb, ++u) {
        const uint32_t st = u % Smem::kStagesQ, ph = (u / Smem::kStagesQ) & 1u;
        const uint32_t ds = u % Smem::kStagesDO, dph = (u / Smem::kStagesDO) & 1u;
        const size_t row0 = (size_t)bh * p.S_pad + 64 * qb;
        // (checked builds: a query block of the sequence, of a query head of
        // the batch, whose per-row statistics lie inside the workspace)
        const bool in_range = attn_check(qb >= 0 && 64 * qb < p.S && bh >= 0 && bh < p.B * p.Hq &&
                                             row0 + 64 <= (size_t)p.B * p.Hq * p.S_pad,
                                         p.error_word);
        // the per-row statistics ride with Q (dK pass) or dO (dV pass)
        constexpr uint32_t kStatBytes = 2u * 256u;
        if (!(ok = mbar_wait(&sm.q_empty[st], ph ^ 1u, abort))) break;
        mbar_arrive_expect_tx(&sm.q_full[st],
                              in_range ? Cfg::kSmallTile + (DK ? kStatBytes : 0u) : 0u);
        for (int hf = 0; in_range && hf < 4; ++hf)
          tma_load_3d_hint(sm.q[st] + hf * Cfg::kSmallBox, map_q, &sm.q_full[st], 64 * hf,
                           64 * qb, bh, keep);
        if (DK && in_range) {
          bulk_load(sm.lse2[st], p.lse2 + row0, 256, &sm.q_full[st], keep);
          bulk_load(sm.dlt[st], p.delta + row0, 256, &sm.q_full[st], keep);
        }
        q_loaded |= 1u << st;
        q_par = (q_par & ~(1u << st)) | (ph << st);
        if (!(ok = mbar_wait(&sm.do_empty[ds], dph ^ 1u, abort))) break;
        mbar_arrive_expect_tx(&sm.do_full[ds],
                              in_range ? Cfg::kSmallTile + (DK ? 0u : kStatBytes) : 0u);
        for (int hf = 0; in_range && hf < 4; ++hf)
          tma_load_3d_hint(sm.dO[ds] + hf * Cfg::kSmallBox, map_do, &sm.do_full[ds], 64 * hf,
                           64 * qb, bh, keep);
        if (!DK && in_range) {
          bulk_load(sm.lse2[ds], p.lse2 + row0, 256, &sm.do_full[ds], keep);
          bulk_load(sm.dlt[ds], p.delta + row0, 256, &sm.do_full[ds], keep);
        }
        d_loaded |= 1u << ds;
        d_par = (d_par & ~(1u << ds)) | (dph << ds);
      }
    }
  }
  // every copy this thread started has landed before the CTA may exit
  if (items > 0) bwd_wait_drain(&sm.kv_full, (uint32_t)(items - 1) & 1u);
  for (int i = 0; i < Smem::kStagesQ; ++i)
    if (q_loaded & (1u << i)) bwd_wait_drain(&sm.q_full[i], (q_par >> i) & 1u);
  for (int i = 0; i < Smem::kStagesDO; ++i)
    if (d_loaded & (1u << i)) bwd_wait_drain(&sm.do_full[i], (d_par >> i) & 1u);
}

// MMA issue order per item of N steps (one step = one 64-row query block of
// one query head; u counts steps across items).  dV pass: S^T(0), then per
// step n: S^T(n+1) into the other score buffer, then dV(n) once P^T(n) is
// written.  dK pass: S^T(0), dP^T(0), then per step n: S^T(n+1), dP^T(n+1)
// into the other buffers, then dK(n) once dS^T(n) is written.  A buffer is
// overwritten two steps later, after the accumulation MMA that read it
// (issued before, in order) and after the element-wise warps are done with
// it (the accumulation waited for them).
template <bool DK>
__device__ __forceinline__ void bwd256_kv_issuer(Bwd256KvSmem<DK>& sm, const BwdParams& p,
                                                 volatile int* abort) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256KvSmem<DK>;
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t idesc_acc = idesc_bf16_f32(128, 256, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kSmallBox, 1024);
  const uint64_t dk_ = kKmajor | (smem_u32(sm.k) >> 4);
  const uint64_t dv_ = kKmajor | (smem_u32(sm.v) >> 4);
  const uint64_t dq_k = kKmajor | (smem_u32(sm.q[0]) >> 4);
  const uint64_t ddo_k = kKmajor | (smem_u32(sm.dO[0]) >> 4);
  const uint64_t dq_mn = kMnMajor | (smem_u32(sm.q[0]) >> 4);
  const uint64_t ddo_mn = kMnMajor | (smem_u32(sm.dO[0]) >> 4);
  constexpr uint64_t kStage = Cfg::kSmallTile >> 4;   // one stage in descriptor units
  // D (128 x 64) = A (128 x 256, stays) B^T (64 x 256, a stage), both K-major
  auto mma_s = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t offa = ((kk / 4) * Cfg::kBigBox + (kk % 4) * 32) >> 4;
      const uint32_t offb = ((kk / 4) * Cfg::kSmallBox + (kk % 4) * 32) >> 4;
      mma_bf16_ss_warp(d, a + offa, b + offb, idesc_s, kk > 0 ? 1u : 0u);
    }
  };
  // Acc (128 x 256) (+)= A (tensor memory, 128 x 64 bf16 pairs) B (64 x 256, MN-major)
  auto mma_acc = [&](uint32_t a, uint64_t b, bool first) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16_ts_warp(Cfg::kColAcc, a + bwd256_packed_col(kk), b + kk * (2048 >> 4), idesc_acc,
                       (!first || kk > 0) ? 1u : 0u);
  };
  auto wait_all = [&](uint64_t* bar, uint32_t ph) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort));
  };
  auto qst = [](uint32_t x) { return x % (uint32_t)Smem::kStagesQ; };
  auto qph = [](uint32_t x) { return (x / (uint32_t)Smem::kStagesQ) & 1u; };
  auto dst = [](uint32_t x) { return x % (uint32_t)Smem::kStagesDO; };
  auto dph = [](uint32_t x) { return (x / (uint32_t)Smem::kStagesDO) & 1u; };
  // S^T(x) into score buffer x & 1; (dK pass) dP^T(x) into dP buffer x & 1
  auto issue_scores = [&](uint32_t x) -> bool {
    if (!wait_all(&sm.q_full[qst(x)], qph(x))) return false;
    tc_fence_after_sync();
    if (!DK) {
      // S^T = K Q^T with K from tensor memory: only Q streams from shared memory
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint32_t offb = ((kk / 4) * Cfg::kSmallBox + (kk % 4) * 32) >> 4;
        mma_bf16_ts_warp(Cfg::kColS + 64 * (x & 1u), Cfg::kColKt + 8 * kk,
                         dq_k + qst(x) * kStage + offb, idesc_s, kk > 0 ? 1u : 0u);
      }
    } else {
      mma_s(Cfg::kColS + 64 * (x & 1u), dk_, dq_k + qst(x) * kStage);
    }
    mma_commit_warp(&sm.s_full[x & 1u]);
    if (!DK) mma_commit_warp(&sm.q_empty[qst(x)]);   // (dV pass: S^T is Q's only reader)
    if (DK) {
      if (!wait_all(&sm.do_full[dst(x)], dph(x))) return false;
      tc_fence_after_sync();
      mma_s(Cfg::kColDP + 64 * (x & 1u), dv_, ddo_k + dst(x) * kStage);
      mma_commit_warp(&sm.dp_full[x & 1u]);
      mma_commit_warp(&sm.do_empty[dst(x)]);
    }
    return true;
  };
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd256_kv_item_of(p, w);
    const int N = p.group * (I.hi - I.lo + 1);
    if (!(ok = wait_all(&sm.kv_full, (uint32_t)items & 1u))) break;
    tc_fence_after_sync();
    // the barrier the item's last S^T commits: kv_empty (K read from shared
    // memory), or in the dV pass kt_free (K read from tensor memory)
    uint64_t* k_done = &sm.kv_empty;
    if (!DK) {
      // copy K into tensor memory once the previous item's S^T MMAs, which
      // read the previous copy, are done (a copy is not ordered behind an
      // MMA issued before it); the shared-memory K is then free
      if (items > 0 &&
          !(ok = wait_all(&sm.kt_free, (uint32_t)(items - 1) & 1u)))
        break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        tmem_cp_128x256b_warp(Cfg::kColKt + 8 * kk,
                              dk_ + (((kk / 4) * Cfg::kBigBox + (kk % 4) * 32) >> 4));
      mma_commit_warp(&sm.kv_empty);
      k_done = &sm.kt_free;
    }
    ++items;
    if (!(ok = issue_scores(u))) break;
    if (N == 1) mma_commit_warp(k_done);
    for (int n = 0; n < N; ++n, ++u) {
      if (n + 1 < N) {
        if (!(ok = issue_scores(u + 1))) break;
        if (n + 2 == N) mma_commit_warp(k_done);   // the item's last read of K (and V)
      }
      if (DK) {
        if (!(ok = wait_all(&sm.ds_full[u & 1u], (u >> 1) & 1u))) break;
        tc_fence_after_sync();
        mma_acc(Cfg::kColDP + 64 * (u & 1u), dq_mn + qst(u) * kStage, n == 0);   // dK += dS^T Q
        mma_commit_warp(&sm.q_empty[qst(u)]);
      } else {
        if (!(ok = wait_all(&sm.p_full[u & 1u], (u >> 1) & 1u))) break;
        if (!(ok = wait_all(&sm.do_full[dst(u)], dph(u)))) break;
        tc_fence_after_sync();
        mma_acc(Cfg::kColS + 64 * (u & 1u), ddo_mn + dst(u) * kStage, n == 0);   // dV += P^T dO
        mma_commit_warp(&sm.do_empty[dst(u)]);
      }
    }
    if (ok) mma_commit_warp(&sm.acc_final);
  }
  mma_commit_warp(&sm.mma_done);
  bwd_wait_drain(&sm.mma_done, 0);
}

// Element-wise work of the dV / dK passes (warps 0-7; thread t of warpgroup
// wg owns key row 128 kb + t, tensor-memory lane t, and query columns
// 32 wg .. 32 wg + 31 of each 64-row query block).  Per step:
// P^T = exp2(S^T * scale*log2e - lse2[query]) (0 where masked); the dV pass
// writes it as bf16 pairs over S^T, the dK pass keeps it in fp32 and writes
// dS^T = P^T o (dP^T - D[query]) as bf16 pairs over dP^T.  Per item: dV, or
// scale * dK, out (the two warpgroups take alternate 32-column chunks).
template <bool DK>
__device__ __forceinline__ void bwd256_kv_softmax(Bwd256KvSmem<DK>& sm, const BwdParams& p,
                                                  uint32_t tbase, volatile int* abort, int warp,
                                                  int lane) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256KvSmem<DK>;
  const int wg = warp / 4;
  const int t = (warp % 4) * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)((warp % 4) * 32) << 16);
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd256_kv_item_of(p, w);
    const int j = 128 * I.kb + t;   // this thread's key
    for (int hh = 0; ok && hh < p.group; ++hh) {
      for (int qb = I.lo; qb <= I.hi; ++qb, ++u) {
        const uint32_t st = u % Smem::kStagesStat;
        const uint32_t b = u & 1u;   // this step's score (and dP) buffer
        // the step's lse2 / D (bulk copies counted on the Q or the dO stage)
        uint64_t* stat_full = DK ? &sm.q_full[st] : &sm.do_full[st];
        if (!(ok = mbar_wait(stat_full, (u / Smem::kStagesStat) & 1u, abort))) break;
        if (!(ok = mbar_wait(&sm.s_full[b], (u >> 1) & 1u, abort))) break;
        tc_fence_after_sync();
        // visible query columns of key j: c in [clo, chi] (query i = 64 qb + 32 wg + c)
        const int i0 = 64 * qb + Cfg::kCols * wg;
        int clo = 0, chi = Cfg::kCols - 1;
        if (p.causal) clo = j - i0;                                     // i >= j
        if (p.window > 0) chi = min(chi, j - i0 + p.window - 1);        // i - j < W
        chi = min(chi, p.S - 1 - i0);                                   // i < S
        const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
        if (chi < clo) clo = 1 << 30;
        const bool msk = clo > 0 || chi < Cfg::kCols - 1;
        const float4* L4 = reinterpret_cast<const float4*>(sm.lse2[st] + Cfg::kCols * wg);
        const float4* D4 = reinterpret_cast<const float4*>(sm.dlt[st] + Cfg::kCols * wg);
        const uint32_t colS = lane_addr + Cfg::kColS + 64 * b + Cfg::kCols * wg;
        uint32_t x[32];
        tmem_ld_32x32b_x32(colS, x);
        tmem_ld_wait(x);
        float pf[Cfg::kCols];
        uint32_t w16[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l = L4[e4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = 2 * e4 + h, col = 2 * e;
            const float2 xs = __ffma2_rn(
                make_float2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])), sl2,
                h ? make_float2(-l.z, -l.w) : make_float2(-l.x, -l.y));
            float a = ex2_approx(xs.x), c = ex2_approx(xs.y);
            if (msk) {
              a = zero_unless_le(a, (uint32_t)(col - clo), span);
              c = zero_unless_le(c, (uint32_t)(col + 1 - clo), span);
            }
            pf[col] = a;
            pf[col + 1] = c;
            w16[e] = pack_bf16x2(a, c);
          }
        }
        if (!DK) {
          tmem_st_32x32b_x16(colS, w16);   // P^T pairs over this warpgroup's S^T columns
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&sm.p_full[b]);
          continue;
        }
        if (!(ok = mbar_wait(&sm.dp_full[b], (u >> 1) & 1u, abort))) break;
        tc_fence_after_sync();
        const uint32_t colDP = lane_addr + Cfg::kColDP + 64 * b + Cfg::kCols * wg;
        uint32_t y[32];
        tmem_ld_32x32b_x32(colDP, y);
        tmem_ld_wait(y);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 d = D4[e4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e = 2 * e4 + h, col = 2 * e;
            const float2 dd = __fadd2_rn(
                make_float2(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1])),
                h ? make_float2(-d.z, -d.w) : make_float2(-d.x, -d.y));
            const float2 dsv = __fmul2_rn(make_float2(pf[col], pf[col + 1]), dd);
            w16[e] = pack_bf16x2(dsv.x, dsv.y);
          }
        }
        tmem_st_32x32b_x16(colDP, w16);   // dS^T pairs over this warpgroup's dP^T columns
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sm.ds_full[b]);
      }
    }
    if (!ok) break;

    // ---- epilogue: dV, or scale * dK, of key j
    if (!(ok = mbar_wait(&sm.acc_final, (uint32_t)items & 1u, abort))) break;
    ++items;
    tc_fence_after_sync();
    const bool store = j < p.S;
    __nv_bfloat16* dst = (DK ? p.dk : p.dv) + ((size_t)I.bkv * p.S + j) * Cfg::DH;
    const float mul = DK ? p.scale : 1.0f;
#pragma unroll 1
    for (int c = wg; c < Cfg::DH / 32; c += Cfg::kWG) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(lane_addr + Cfg::kColAcc + 32 * c, r);
      tmem_ld_wait(r);
      if (store) bwd_store32(dst + 32 * c, r, mul);
    }
    // the next item's first accumulation overwrites the accumulator only
    // after this thread's next arrive on p_full / ds_full, which follows
    // these loads
  }
}

template <bool DK>
__global__ void __launch_bounds__(Bwd256Cfg::kThreads, 1)
    attn_bwd256_kv(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256KvSmem<DK>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  volatile int* abort = &sm.abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (warp == Cfg::kWarpProducer && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    if (DK) prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_do);
  }
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    mbar_init(&sm.kt_free, 1);
    for (int i = 0; i < Smem::kStagesQ; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    for (int i = 0; i < Smem::kStagesDO; ++i) {
      mbar_init(&sm.do_full[i], 1);
      mbar_init(&sm.do_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.dp_full[i], 1);
      mbar_init(&sm.p_full[i], Cfg::kEW);
      mbar_init(&sm.ds_full[i], Cfg::kEW);
    }
    mbar_init(&sm.acc_final, 1);
    mbar_init(&sm.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == Cfg::kWarpProducer) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // the dV pass follows the prep kernel (it waits for it before reading
  // D and lse2); the dK pass reads nothing the dV pass writes, only the
  // inputs and the prep's output, complete before any dV CTA let this grid
  // be scheduled, so it starts at once and waits for the dV pass only
  // before it ends (below)
  if (!DK) griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tbase = sm.tmem_base;
  // compile-time tensor-memory columns: the allocation must start at column 0
  if (tbase != 0 && threadIdx.x == 0) sm.abort_flag = 1;
  if (tbase == 0) {
    if (warp == Cfg::kWarpProducer) {
      if (lane == 0) bwd256_kv_producer<DK>(sm, p, &map_q, &map_k, &map_v, &map_do, abort);
    } else if (warp == Cfg::kWarpIssuer) {
      bwd256_kv_issuer<DK>(sm, p, abort);
    } else {
      bwd256_kv_softmax<DK>(sm, p, tbase, abort, warp, lane);
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kWarpProducer) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
  // (dK pass) not finished before the dV pass is, so that the next kernel in
  // the stream sees dV as well
  if (DK && threadIdx.x == 0) griddep_wait();
}

// ============================================================ dQ pass

struct __align__(1024) Bwd256QSmem {
  using Cfg = Bwd256Cfg;
  static constexpr int kStagesK = 2, kStagesV = 1;
  uint8_t q[Cfg::kBigTile];                 // this item's query block (stays)
  uint8_t dO[Cfg::kBigTile];                // and its output gradient
  uint8_t k[kStagesK][Cfg::kSmallTile];     // key blocks: read by S(n) and dQ(n)
  uint8_t v[kStagesV][Cfg::kSmallTile];     // value blocks: read by dP(n) only
  uint64_t q_full, q_empty;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full, s_free, acc_final, mma_done;
  uint64_t dp_full[2], ds_full[2];   // per dP / dS buffer
  uint64_t qt_free;                  // the item's last S MMA (reader of Q in tensor memory) is done
  uint32_t tmem_base;
  int abort_flag;
};

// Item w: 128-row query block qb (latest, i.e. heaviest under a causal
// mask, first) of query head bh.
__device__ __forceinline__ BwdQItem bwd256_q_item_of(const BwdParams& p, int w) {
  BwdQItem r;
  const int per = p.B * p.Hq;
  const int blk = w / per;
  r.qb = p.nblk - 1 - blk;
  r.bh = w - blk * per;
  const int b = r.bh / p.Hq;
  r.bkv = b * p.Hkv + (r.bh - b * p.Hq) / p.group;   // g(h) = floor(h / (H/G))
  bwd256_kblocks_of(p, r.qb, r.lo, r.hi);
  return r;
}

__device__ __forceinline__ void bwd256_dq_producer(Bwd256QSmem& sm, const BwdParams& p,
                                                   const CUtensorMap* map_q,
                                                   const CUtensorMap* map_k,
                                                   const CUtensorMap* map_v,
                                                   const CUtensorMap* map_do,
                                                   volatile int* abort) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256QSmem;
  const uint64_t keep = policy_evict_last();   // key blocks are re-read by other query blocks
  uint32_t u = 0, k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd256_q_item_of(p, w);
    if (items > 0 && !(ok = mbar_wait(&sm.q_empty, (uint32_t)(items - 1) & 1u, abort))) break;
    // (checked builds: a query block of the sequence, of a query head of the batch)
    const bool q_in_range = attn_check(I.qb >= 0 && 128 * I.qb < p.S && I.bh >= 0 &&
                                           I.bh < p.B * p.Hq,
                                       p.error_word);
    mbar_arrive_expect_tx(&sm.q_full, q_in_range ? 2u * Cfg::kBigTile : 0u);
    for (int hf = 0; q_in_range && hf < 4; ++hf) {
      tma_load_3d(sm.q + hf * Cfg::kBigBox, map_q, &sm.q_full, 64 * hf, 128 * I.qb, I.bh);
      tma_load_3d(sm.dO + hf * Cfg::kBigBox, map_do, &sm.q_full, 64 * hf, 128 * I.qb, I.bh);
    }
    ++items;
    for (int kb = I.lo; kb <= I.hi; ++kb, ++u) {
      // (checked builds: a key block of the sequence, of a K/V head of the batch)
      const bool in_range = attn_check(kb >= 0 && 64 * kb < p.S && I.bkv >= 0 &&
                                           I.bkv < p.B * p.Hkv,
                                       p.error_word);
      const uint32_t bytes = in_range ? (uint32_t)Cfg::kSmallTile : 0u;
      const uint32_t ks = u % Smem::kStagesK, kph = (u / Smem::kStagesK) & 1u;
      if (!(ok = mbar_wait(&sm.k_empty[ks], kph ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.k_full[ks], bytes);
      for (int hf = 0; in_range && hf < 4; ++hf)
        tma_load_3d_hint(sm.k[ks] + hf * Cfg::kSmallBox, map_k, &sm.k_full[ks], 64 * hf, 64 * kb,
                         I.bkv, keep);
      k_loaded |= 1u << ks;
      k_par = (k_par & ~(1u << ks)) | (kph << ks);
      const uint32_t vs = u % Smem::kStagesV, vph = (u / Smem::kStagesV) & 1u;
      if (!(ok = mbar_wait(&sm.v_empty[vs], vph ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.v_full[vs], bytes);
      for (int hf = 0; in_range && hf < 4; ++hf)
        tma_load_3d_hint(sm.v[vs] + hf * Cfg::kSmallBox, map_v, &sm.v_full[vs], 64 * hf, 64 * kb,
                         I.bkv, keep);
      v_loaded |= 1u << vs;
      v_par = (v_par & ~(1u << vs)) | (vph << vs);
    }
  }
  if (items > 0) bwd_wait_drain(&sm.q_full, (uint32_t)(items - 1) & 1u);
  for (int i = 0; i < Smem::kStagesK; ++i)
    if (k_loaded & (1u << i)) bwd_wait_drain(&sm.k_full[i], (k_par >> i) & 1u);
  for (int i = 0; i < Smem::kStagesV; ++i)
    if (v_loaded & (1u << i)) bwd_wait_drain(&sm.v_full[i], (v_par >> i) & 1u);
}

// MMA issue order per item of N key blocks: S(0), dP(0), then per block n:
// S(n+1) once the element-wise warps have read S(n), dP(n+1) into the other
// dP buffer, then dQ(n) once dS(n) is written over dP(n) (as in the Dh <= 128
// dQ pass).  A key block is released after dQ, a value block after its dP.
__device__ __forceinline__ void bwd256_dq_issuer(Bwd256QSmem& sm, const BwdParams& p,
                                                 volatile int* abort) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256QSmem;
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t idesc_acc = idesc_bf16_f32(128, 256, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kSmallBox, 1024);
  const uint64_t dq_ = kKmajor | (smem_u32(sm.q) >> 4);
  const uint64_t ddo_ = kKmajor | (smem_u32(sm.dO) >> 4);
  const uint64_t dk_k = kKmajor | (smem_u32(sm.k[0]) >> 4);
  const uint64_t dv_k = kKmajor | (smem_u32(sm.v[0]) >> 4);
  const uint64_t dk_mn = kMnMajor | (smem_u32(sm.k[0]) >> 4);
  constexpr uint64_t kStage = Cfg::kSmallTile >> 4;
  // D (128 x 64) = A (128 x 256, stays) B^T (64 x 256, a stage), both K-major
  auto mma_s = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t offa = ((kk / 4) * Cfg::kBigBox + (kk % 4) * 32) >> 4;
      const uint32_t offb = ((kk / 4) * Cfg::kSmallBox + (kk % 4) * 32) >> 4;
      mma_bf16_ss_warp(d, a + offa, b + offb, idesc_s, kk > 0 ? 1u : 0u);
    }
  };
  // S = Q K^T with Q's first 128 columns from tensor memory, the rest from
  // shared memory
  auto mma_qk = [&](uint32_t d, uint64_t b) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t offa = ((kk / 4) * Cfg::kBigBox + (kk % 4) * 32) >> 4;
      const uint32_t offb = ((kk / 4) * Cfg::kSmallBox + (kk % 4) * 32) >> 4;
      if (kk < 8)
        mma_bf16_ts_warp(d, Cfg::kColQt + 8 * kk, b + offb, idesc_s, kk > 0 ? 1u : 0u);
      else
        mma_bf16_ss_warp(d, dq_ + offa, b + offb, idesc_s, 1u);
    }
  };
  auto wait_all = [&](uint64_t* bar, uint32_t ph) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort));
  };
  auto kst = [](uint32_t x) { return x % (uint32_t)Smem::kStagesK; };
  auto kph = [](uint32_t x) { return (x / (uint32_t)Smem::kStagesK) & 1u; };
  auto vst = [](uint32_t x) { return x % (uint32_t)Smem::kStagesV; };
  auto vph = [](uint32_t x) { return (x / (uint32_t)Smem::kStagesV) & 1u; };
  auto issue_dp = [&](uint32_t x) -> bool {
    if (!wait_all(&sm.v_full[vst(x)], vph(x))) return false;
    tc_fence_after_sync();
    mma_s(Cfg::kColDP + 64 * (x & 1u), ddo_, dv_k + vst(x) * kStage);   // dP = dO V^T
    mma_commit_warp(&sm.dp_full[x & 1u]);
    mma_commit_warp(&sm.v_empty[vst(x)]);
    return true;
  };
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd256_q_item_of(p, w);
    const int N = I.hi - I.lo + 1;
    if (!(ok = wait_all(&sm.q_full, (uint32_t)items & 1u))) break;
    // Q's first half into tensor memory, once the previous item's S MMAs
    // (which read the previous copy) are done
    if (items > 0 && !(ok = wait_all(&sm.qt_free, (uint32_t)(items - 1) & 1u))) break;
    tc_fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      tmem_cp_128x256b_warp(Cfg::kColQt + 8 * kk,
                            dq_ + (((kk / 4) * Cfg::kBigBox + (kk % 4) * 32) >> 4));
    ++items;
    if (!(ok = wait_all(&sm.k_full[kst(u)], kph(u)))) break;
    tc_fence_after_sync();
    mma_qk(Cfg::kColS, dk_k + kst(u) * kStage);                          // S = Q K^T
    mma_commit_warp(&sm.s_full);
    if (!(ok = issue_dp(u))) break;
    if (N == 1) {
      mma_commit_warp(&sm.q_empty);
      mma_commit_warp(&sm.qt_free);
    }
    for (int n = 0; n < N; ++n, ++u) {
      if (n + 1 < N) {
        if (!(ok = wait_all(&sm.s_free, u & 1u))) break;
        if (!(ok = wait_all(&sm.k_full[kst(u + 1)], kph(u + 1)))) break;
        tc_fence_after_sync();
        mma_qk(Cfg::kColS, dk_k + kst(u + 1) * kStage);
        mma_commit_warp(&sm.s_full);
        if (!(ok = issue_dp(u + 1))) break;
        if (n + 2 == N) {
          mma_commit_warp(&sm.q_empty);
          mma_commit_warp(&sm.qt_free);
        }
      }
      if (!(ok = wait_all(&sm.ds_full[u & 1u], (u >> 1) & 1u))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)                                       // dQ += dS K
        mma_bf16_ts_warp(Cfg::kColAcc, Cfg::kColDP + 64 * (u & 1u) + bwd256_packed_col(kk),
                         dk_mn + kst(u) * kStage + kk * (2048 >> 4), idesc_acc,
                         (n > 0 || kk > 0) ? 1u : 0u);
      mma_commit_warp(&sm.k_empty[kst(u)]);
    }
    if (ok) mma_commit_warp(&sm.acc_final);
  }
  mma_commit_warp(&sm.mma_done);
  bwd_wait_drain(&sm.mma_done, 0);
}

// Element-wise work of the dQ pass (warps 0-7; thread t of warpgroup wg owns
// query row 128 qb + t and key columns 32 wg .. 32 wg + 31 of each 64-key
// block): P = exp2(S * scale*log2e - lse2_i) (0 where masked), kept in fp32;
// dS = P o (dP - D_i) as bf16 pairs over dP.  Per item: scale * dQ out.
__device__ __forceinline__ void bwd256_dq_softmax(Bwd256QSmem& sm, const BwdParams& p,
                                                  uint32_t tbase, volatile int* abort, int warp,
                                                  int lane) {
  using Cfg = Bwd256Cfg;
  const int wg = warp / 4;
  const int t = (warp % 4) * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)((warp % 4) * 32) << 16);
  const uint32_t colS = lane_addr + Cfg::kColS + Cfg::kCols * wg;
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd256_q_item_of(p, w);
    const int i = 128 * I.qb + t;   // this thread's query
    const float L = p.lse2[(size_t)I.bh * p.S_pad + i];
    const float Di = p.delta[(size_t)I.bh * p.S_pad + i];
    const float2 negL = make_float2(-L, -L), negD = make_float2(-Di, -Di);
    for (int kb = I.lo; kb <= I.hi; ++kb, ++u) {
      if (!(ok = mbar_wait(&sm.s_full, u & 1u, abort))) break;
      tc_fence_after_sync();
      // visible keys of query i: [klo, khi], as columns [clo, chi] of this warpgroup's
      const int j0 = 64 * kb + Cfg::kCols * wg;
      int khi = p.S - 1;
      if (p.causal) khi = min(khi, i);
      const int klo = p.window > 0 ? i - p.window + 1 : 0;
      int clo = klo - j0;
      const int chi = khi - j0;
      const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
      if (chi < clo) clo = 1 << 30;
      const bool msk = clo > 0 || chi < Cfg::kCols - 1;
      uint32_t x[32];
      tmem_ld_32x32b_x32(colS, x);
      tmem_ld_wait(x);
      // S is in registers: the next S may overwrite it
      tc_fence_before_sync();
      mbar_arrive(&sm.s_free);
      float pf[Cfg::kCols];
#pragma unroll
      for (int e = 0; e < Cfg::kCols / 2; ++e) {
        const int col = 2 * e;
        const float2 xs = __ffma2_rn(make_float2(__uint_as_float(x[col]), __uint_as_float(x[col + 1])),
                                     sl2, negL);
        float a = ex2_approx(xs.x), c = ex2_approx(xs.y);
        if (msk) {
          a = zero_unless_le(a, (uint32_t)(col - clo), span);
          c = zero_unless_le(c, (uint32_t)(col + 1 - clo), span);
        }
        pf[col] = a;
        pf[col + 1] = c;
      }
      const uint32_t b = u & 1u;   // this block's dP buffer
      const uint32_t colDP = lane_addr + Cfg::kColDP + 64 * b + Cfg::kCols * wg;
      if (!(ok = mbar_wait(&sm.dp_full[b], (u >> 1) & 1u, abort))) break;
      tc_fence_after_sync();
      uint32_t y[32];
      tmem_ld_32x32b_x32(colDP, y);
      tmem_ld_wait(y);
      uint32_t w16[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int col = 2 * e;
        const float2 dd = __fadd2_rn(
            make_float2(__uint_as_float(y[col]), __uint_as_float(y[col + 1])), negD);
        const float2 dsv = __fmul2_rn(make_float2(pf[col], pf[col + 1]), dd);
        w16[e] = pack_bf16x2(dsv.x, dsv.y);
      }
      tmem_st_32x32b_x16(colDP, w16);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sm.ds_full[b]);
    }
    if (!ok) break;

    // ---- epilogue: scale * dQ of query i (the warpgroups take alternate chunks)
    if (!(ok = mbar_wait(&sm.acc_final, (uint32_t)items & 1u, abort))) break;
    ++items;
    tc_fence_after_sync();
    const bool store = i < p.S;
    const size_t row = ((size_t)I.bh * p.S + i) * Cfg::DH;
#pragma unroll 1
    for (int c = wg; c < Cfg::DH / 32; c += Cfg::kWG) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(lane_addr + Cfg::kColAcc + 32 * c, r);
      tmem_ld_wait(r);
      if (store) bwd_store32(p.dq + row + 32 * c, r, p.scale);
    }
  }
}

__global__ void __launch_bounds__(Bwd256Cfg::kThreads, 1)
    attn_bwd256_dq(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using Cfg = Bwd256Cfg;
  using Smem = Bwd256QSmem;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  volatile int* abort = &sm.abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (warp == Cfg::kWarpProducer && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_do);
  }
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int i = 0; i < Smem::kStagesK; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < Smem::kStagesV; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, Cfg::kEW);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.dp_full[i], 1);
      mbar_init(&sm.ds_full[i], Cfg::kEW);
    }
    mbar_init(&sm.acc_final, 1);
    mbar_init(&sm.qt_free, 1);
    mbar_init(&sm.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == Cfg::kWarpProducer) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Launched as a programmatic dependent of the dK pass: like that pass it
  // reads only the inputs and the prep kernel's output (complete before this
  // grid could be scheduled), so it starts at once, and it waits for the dK
  // pass only before it ends (below)
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tbase = sm.tmem_base;
  if (tbase != 0 && threadIdx.x == 0) sm.abort_flag = 1;
  if (tbase == 0) {
    if (warp == Cfg::kWarpProducer) {
      if (lane == 0) bwd256_dq_producer(sm, p, &map_q, &map_k, &map_v, &map_do, abort);
    } else if (warp == Cfg::kWarpIssuer) {
      bwd256_dq_issuer(sm, p, abort);
    } else {
      bwd256_dq_softmax(sm, p, tbase, abort, warp, lane);
    }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kWarpProducer) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
  // not finished before the dK pass (and through it the dV pass) is, so that
  // the next kernel in the stream sees dK and dV as well
  if (threadIdx.x == 0) griddep_wait();
}

template <bool DK>
constexpr size_t bwd256_kv_smem_bytes() { return sizeof(Bwd256KvSmem<DK>) + 1024; }
constexpr size_t bwd256_dq_smem_bytes() { return sizeof(Bwd256QSmem) + 1024; }

}  // namespace chs
