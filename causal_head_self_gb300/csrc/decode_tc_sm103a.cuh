// decode_tc_sm103a.cuh -- the decode step for query-head groups (GQA, MQA)
// on the 5th-generation tensor cores (sm_103a).
//
// When several query heads share one K/V head, every cached byte meets
// Hq / Hkv query rows (64 FLOP per byte for a group of 32), and the
// CUDA-core decode kernel's per-key softmax work, done for every head of the
// group, becomes its bound (at Dh 64 it held a group of 4 to 55 % of the HBM
// bandwidth; this path runs it at 82 %).  Packed together,
// the group's query rows form a real contraction: S = Q K^T with the group's
// heads as the M dimension (up to 128 per CTA; fewer rows leave the rest of
// the tile unused), 128 keys (64 at Dh = 256) as N, Dh as K, and O = P V.  So this path is the
// prefill pipeline reduced to one 128-row sub-tile without a causal mask: a
// TMA producer streams 128-key K and V tiles of one split of the cache, one
// warp issues tcgen05.mma (S and P.V accumulate in tensor memory), and the
// softmax warps (only those holding real rows) run the online softmax with a
// lazy maximum.  Each CTA writes fp32 partials (o unnormalised, m, l) of its
// split; a small combine kernel merges the splits per (b, query head) with
// the same log-sum-exp algebra as the CUDA-core decode.
//
// Key tiles are placed so that the split's last tile ends at its last key:
// tile j starts at position k_end - kKeys * (n - j), and only the first tile
// can reach below k_begin (into earlier, valid cache rows, or below 0 where
// the copy fills zeros).  Those columns are masked to -inf, so their weights
// are exactly 0 and every V row the MMA reads is a written cache row (or a
// zero row): rows past seqlens[b] are never read.
//
// Every wait is bounded (sm103a_ptx.cuh): a lost arrival ends the CTA with
// ATTN_ERR_TIMEOUT latched instead of a hang.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103a_ptx.cuh"

namespace chs {

struct DecodeTcParams {
  int B, Hq, Hkv, G, Tmax, window;
  int ring;                 // 1: position t of a sequence sits at cache row t % Tmax
  int nsplit, chunk;        // chunk: keys per split, a multiple of 128
  int row_blocks;           // ceil(G / 128): CTAs per (b, K/V head, split)
  float scale_log2;
  const int* seqlens;       // [B], device
  float* o_part;            // [B, Hq, nsplit, DH]  unnormalised
  float* m_part;            // [B, Hq, nsplit]      (log2 domain)
  float* l_part;            // [B, Hq, nsplit]
  __nv_bfloat16* o;         // [B, Hq, 1, DH]
  int* error_word;
  int fault;                // test hook: 3 = the first K tile is never loaded
};

template <int DH>
struct DecodeTcCfg {
  // keys per K/V tile: 128, or 64 at Dh = 256 so that Q (64 KiB) and the two
  // two-stage rings (32 KiB tiles) fit in shared memory
  static constexpr int kKeys = DH <= 128 ? 128 : 64;
  static constexpr int kHalves = DH / 64;
  static constexpr int kQBoxBytes = 128 * 64 * 2;    // Q box: 128 rows x 64 columns
  static constexpr int kBoxBytes = kKeys * 64 * 2;   // K/V box: kKeys rows x 64 columns
  static constexpr int kQBytes = kHalves * kQBoxBytes;
  static constexpr int kTileBytes = kHalves * kBoxBytes;
  static constexpr int kStages = DH <= 128 ? 3 : 2;  // K ring and V ring (smem: 224 KiB at Dh 128)
  static constexpr int kThreads = 192;               // warps 0-3 softmax, 4 producer, 5 MMA
  static constexpr int kWarpProducer = 4, kWarpIssuer = 5;
  static constexpr uint32_t kCols = 512;             // S0, S1 (kKeys each), O [256, 256 + DH)
  static constexpr uint32_t kColS = 0, kColO = 256;  // S buffer b at kColS + kKeys b
  static_assert(2 * kKeys <= (int)kColO && kColO + DH <= kCols, "tensor-memory columns");
};

template <int DH>
struct __align__(1024) DecodeTcSmem {
  using Cfg = DecodeTcCfg<DH>;
  uint8_t q[Cfg::kQBytes];
  uint8_t k[Cfg::kStages][Cfg::kTileBytes];
  uint8_t v[Cfg::kStages][Cfg::kTileBytes];
  uint64_t q_full;
  uint64_t k_full[Cfg::kStages], k_empty[Cfg::kStages];
  uint64_t v_full[Cfg::kStages], v_empty[Cfg::kStages];
  uint64_t s_full[2], p_full[2], pv_done, o_final, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// The first visible position of a sequence of L keys.  In ring mode the
// cache holds the last Tmax positions, and window <= 0 means a window of Tmax.
__device__ __forceinline__ int decode_tc_lo(const DecodeTcParams& p, int L) {
  const int w = p.window > 0 ? p.window : (p.ring ? p.Tmax : 0);
  return w > 0 ? max(0, L - w) : 0;
}

// The key positions of split `split` of a sequence of L keys: [k_begin, k_end).
// Linear caches: splits at multiples of chunk; ring caches: counted from the
// first visible position.
__device__ __forceinline__ void decode_tc_range(const DecodeTcParams& p, int L, int split,
                                                int& k_begin, int& k_end) {
  // (64-bit: positions may come within a chunk of 2^31)
  const long long lo = decode_tc_lo(p, L), c = p.chunk;
  const long long b = p.ring ? lo + split * c : max(split * c, lo);
  const long long e = p.ring ? b + c : (split + 1) * c;
  k_begin = (int)min(b, (long long)L);
  k_end = (int)min(e, (long long)L);
}

// Where a split's keys sit in the cache, as at most two runs of contiguous
// rows (a ring wraps at most once within a split: its visible positions
// span at most Tmax), each cut into tiles that end at the run's last row.
// Tile j < n1 starts at row origin1 + kKeys j, tile j >= n1 at row
// origin2 + kKeys (j - n1).  Only each run's first tile reaches below the
// run (rows of other positions, or below row 0 where the copy fills zeros):
// its first clo1 (resp. clo2) columns are masked.
struct DecodeTcSpan {
  int n1, origin1, clo1;
  int ntiles, origin2, clo2;
};

template <int KEYS>
__device__ __forceinline__ DecodeTcSpan decode_tc_span(const DecodeTcParams& p, int k_begin,
                                                       int k_end) {
  DecodeTcSpan sp;
  int r_begin = k_begin, r_end1 = k_end, len2 = 0;
  if (p.ring) {
    r_begin = k_begin % p.Tmax;                            // row of the first key
    // first position back at row 0 (64-bit: it may lie past 2^31 - 1)
    const long long wrap = (long long)k_begin - r_begin + p.Tmax;
    const int e1 = (int)min((long long)k_end, wrap);
    r_end1 = r_begin + (e1 - k_begin);
    len2 = k_end - e1;
  }
  sp.n1 = (r_end1 - r_begin + KEYS - 1) / KEYS;
  sp.origin1 = r_end1 - KEYS * sp.n1;
  sp.clo1 = r_begin - sp.origin1;
  const int n2 = (len2 + KEYS - 1) / KEYS;
  sp.origin2 = len2 - KEYS * n2;
  sp.clo2 = -sp.origin2;
  sp.ntiles = sp.n1 + n2;
  return sp;
}

// Drain wait used at teardown: ignores the abort flag, bounded by time.
__device__ __forceinline__ void mbar_wait_drain_tc(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// TMA producer (one thread): the CTA's 128 query rows once, then the split's
// K and V tiles through two-stage rings.
template <int DH>
__device__ __forceinline__ void decode_tc_producer(DecodeTcSmem<DH>& sm, const DecodeTcParams& p,
                                                   const CUtensorMap* map_q,
                                                   const CUtensorMap* map_k,
                                                   const CUtensorMap* map_v, int bg, int rb,
                                                   const DecodeTcSpan& sp, volatile int* abort) {
  using Cfg = DecodeTcCfg<DH>;
  const uint64_t once = policy_evict_first();   // each cached row is read by one CTA
  mbar_arrive_expect_tx(&sm.q_full, Cfg::kQBytes);
  for (int hf = 0; hf < Cfg::kHalves; ++hf)
    tma_load_3d(sm.q + hf * Cfg::kQBoxBytes, map_q, &sm.q_full, hf * 64, 128 * rb, bg);
  uint32_t k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
  for (int j = 0; j < sp.ntiles; ++j) {
    const int st = j % Cfg::kStages;
    const uint32_t ph = (uint32_t)(j / Cfg::kStages) & 1u;
    // may be negative for a run's first tile: zeros
    const int row = j < sp.n1 ? sp.origin1 + Cfg::kKeys * j : sp.origin2 + Cfg::kKeys * (j - sp.n1);
    // (checked builds: a tile ends inside the cache and starts less than a
    // tile below row 0)
    const bool in_range = attn_check(row > -Cfg::kKeys && row + Cfg::kKeys <= p.Tmax, p.error_word);
    const uint32_t bytes = in_range ? (uint32_t)Cfg::kTileBytes : 0u;
    if (!mbar_wait(&sm.k_empty[st], ph ^ 1u, abort)) break;
    if (p.fault != 3 || j != 0) {   // (the test hook withholds one tile)
      mbar_arrive_expect_tx(&sm.k_full[st], bytes);
      for (int hf = 0; in_range && hf < Cfg::kHalves; ++hf)
        tma_load_3d_hint(sm.k[st] + hf * Cfg::kBoxBytes, map_k, &sm.k_full[st], hf * 64, row, bg,
                         once);
      k_loaded |= 1u << st;
      k_par = (k_par & ~(1u << st)) | (ph << st);
    }
    if (!mbar_wait(&sm.v_empty[st], ph ^ 1u, abort)) break;
    mbar_arrive_expect_tx(&sm.v_full[st], bytes);
    for (int hf = 0; in_range && hf < Cfg::kHalves; ++hf)
      tma_load_3d_hint(sm.v[st] + hf * Cfg::kBoxBytes, map_v, &sm.v_full[st], hf * 64, row, bg,
                       once);
    v_loaded |= 1u << st;
    v_par = (v_par & ~(1u << st)) | (ph << st);
  }
  // every copy this thread started has landed before the CTA may exit
  mbar_wait_drain_tc(&sm.q_full, 0);
  for (int i = 0; i < Cfg::kStages; ++i) {
    if (k_loaded & (1u << i)) mbar_wait_drain_tc(&sm.k_full[i], (k_par >> i) & 1u);
    if (v_loaded & (1u << i)) mbar_wait_drain_tc(&sm.v_full[i], (v_par >> i) & 1u);
  }
}

// MMA issuer (one converged warp, one elected lane per instruction).  S is
// double-buffered in tensor memory: S(j+1) is computed while the softmax
// works on S(j), so the softmax warps go from one tile to the next without
// waiting for the tensor core.  Order: S(0), S(1), then per tile j: P.V(j)
// once P(j) is written, and S(j+2) into the buffer P(j) lived in (the tensor
// core runs one thread's MMAs in order, so S(j+2) follows P.V(j)).
template <int DH>
__device__ __forceinline__ void decode_tc_issuer(DecodeTcSmem<DH>& sm, uint32_t tbase, int ntiles,
                                                 volatile int* abort) {
  using Cfg = DecodeTcCfg<DH>;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, Cfg::kKeys, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, DH, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);                // Q, K
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kBoxBytes, 1024);   // V
  const uint64_t dq = kKmajor | (smem_u32(sm.q) >> 4);
  const uint64_t dk = kKmajor | (smem_u32(sm.k[0]) >> 4);
  const uint64_t dv = kMnMajor | (smem_u32(sm.v[0]) >> 4);
  const uint32_t dO = tbase + Cfg::kColO;
  auto issue_s = [&](int j) -> bool {
    const int st = j % Cfg::kStages;
    const uint32_t ph = (uint32_t)(j / Cfg::kStages) & 1u;
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.k_full[st], ph, abort))) return false;
    tc_fence_after_sync();
    const uint32_t dS = tbase + Cfg::kColS + (uint32_t)Cfg::kKeys * (uint32_t)(j & 1);
    const uint64_t b = dk + (uint64_t)(st * (Cfg::kTileBytes >> 4));
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      // 16 columns (32 bytes) of Dh per MMA; a 64-column box holds 4 steps
      const uint32_t offq = ((kk / 4) * Cfg::kQBoxBytes + (kk % 4) * 32) >> 4;
      const uint32_t offk = ((kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32) >> 4;
      mma_bf16_ss_warp(dS, dq + offq, b + offk, idesc_qk, kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(&sm.s_full[j & 1]);
    mma_commit_warp(&sm.k_empty[st]);
    return true;
  };
  bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, abort));
  if (ok) ok = issue_s(0);
  if (ok && ntiles > 1) ok = issue_s(1);
  for (int j = 0; ok && j < ntiles; ++j) {
    const int st = j % Cfg::kStages;
    const uint32_t ph = (uint32_t)(j / Cfg::kStages) & 1u;
    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[st], ph, abort)))) break;
    if (!(ok = __all_sync(0xffffffffu,
                          mbar_wait(&sm.p_full[j & 1], (uint32_t)(j >> 1) & 1u, abort))))
      break;
    tc_fence_after_sync();
    // O (+)= P V: P from TMEM (8 columns = 16 keys per MMA), V MN-major
    const uint32_t dP = tbase + Cfg::kColS + (uint32_t)Cfg::kKeys * (uint32_t)(j & 1);
    const uint64_t b = dv + (uint64_t)(st * (Cfg::kTileBytes >> 4));
#pragma unroll
    for (int kk = 0; kk < Cfg::kKeys / 16; ++kk)
      mma_bf16_ts_warp(dO, dP + kk * 8, b + kk * (2048 >> 4), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
    mma_commit_warp(&sm.pv_done);
    mma_commit_warp(&sm.v_empty[st]);
    if (j + 2 < ntiles) ok = issue_s(j + 2);
  }
  if (ok) mma_commit_warp(&sm.o_final);
  // nothing of this warp's may still run on the tensor core at teardown
  mma_commit_warp(&sm.mma_done);
  mbar_wait_drain_tc(&sm.mma_done, 0);
}

// Softmax of the CTA's query rows (thread t owns row t, TMEM lane t): per
// 128-key tile the online softmax of "Online normalizer calculation for
// softmax" with a lazy maximum, as in the prefill; at the end, the row's
// unnormalised o, its maximum m and sum l go to the split's partials.
template <int DH>
__device__ __forceinline__ void decode_tc_softmax(DecodeTcSmem<DH>& sm, const DecodeTcParams& p,
                                                  uint32_t tbase, int warp, int lane, int b,
                                                  int head0, int rows, int split,
                                                  const DecodeTcSpan& sp, volatile int* abort) {
  using Cfg = DecodeTcCfg<DH>;
  const int t = warp * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
  const uint32_t colO = lane_addr + Cfg::kColO;
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int j = 0; j < sp.ntiles; ++j) {
    if (!(ok = mbar_wait(&sm.s_full[j & 1], (uint32_t)(j >> 1) & 1u, abort))) break;
    tc_fence_after_sync();
    const uint32_t colS = lane_addr + Cfg::kColS + (uint32_t)Cfg::kKeys * (uint32_t)(j & 1);
    const int clo0 = j == 0 ? sp.clo1 : (j == sp.n1 ? sp.clo2 : 0);
    if (clo0 > 0) {
      // a run's first tile reaches below the run: its first clo0 columns are
      // not this split's keys (a whole-warp chunk below them is filled
      // without being read; the chunk that straddles is read and masked)
#pragma unroll 1
      for (int c0 = 0; c0 < Cfg::kKeys; c0 += 32) {
        if (c0 >= clo0) break;
        uint32_t y[32];
        if (c0 + 31 < clo0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) y[e] = 0xff800000u;   // -inf
        } else {
          tmem_ld_32x32b_x32(colS + c0, y);
          tmem_ld_wait(y);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            y[e] = __float_as_uint(keep_if_le(__uint_as_float(y[e]), (uint32_t)(c0 + e - clo0),
                                              (uint32_t)(Cfg::kKeys - 1 - clo0)));
        }
        tmem_st_32x32b_x32(colS + c0, y);
      }
      tmem_st_wait();
    }
    constexpr int kChunks = Cfg::kKeys / 32;
    uint32_t r[kChunks][32];
    float mc[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) tmem_ld_max_32x32b_x32(colS + 32 * c, r[c], mc[c]);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) tmem_ld_wait(r[c], mc[c]);
    float x[Cfg::kKeys];
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(r[c][e]);
    float mt = mc[0];
#pragma unroll
    for (int c = 1; c < kChunks; ++c) mt = fmaxf(mt, mc[c]);
    const float m_tile = mt * sl2;
    // lazy maximum (raised only past +8 in log2 units; exact either way)
    const float m_new = fmaxf(m_run, m_tile);
    const bool fresh = m_run == -INFINITY;
    const bool upd = fresh || (m_new > m_run + 8.0f);
    const float m_use = upd ? m_new : m_run;
    const float corr = (upd && !fresh) ? ex2_approx(m_run - m_new) : 1.0f;
    const float msub = (m_use == -INFINITY) ? 0.f : m_use;
    const float2 scale2 = make_float2(sl2, sl2), neg_m2 = make_float2(-msub, -msub);
    float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int c4 = 0; c4 < kChunks; ++c4) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 xs = __ffma2_rn(make_float2(x[32 * c4 + 2 * e], x[32 * c4 + 2 * e + 1]),
                                     scale2, neg_m2);
        const float2 pp = make_float2(ex2_approx(xs.x), ex2_approx(xs.y));
        ls[e & 1] = __fadd2_rn(ls[e & 1], pp);
        pk[e] = pack_bf16x2(pp.x, pp.y);
      }
      tmem_st_32x32b_x16(colS + 16 * c4, pk);   // P over the first kKeys / 2 columns of S
    }
    const float lsum = (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
    // a raised maximum rescales the row's O, once P.V of the previous tile
    // has written it (S(j) was issued before P.V(j-1): wait for it; P.V(j)
    // cannot run before this tile's P is published below)
    if (__any_sync(0xffffffffu, corr != 1.0f)) {
      if (j > 0 && !(ok = mbar_wait(&sm.pv_done, (uint32_t)(j - 1) & 1u, abort))) break;
      tc_fence_after_sync();
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
    mbar_arrive(&sm.p_full[j & 1]);
  }
  if (!ok || !mbar_wait(&sm.o_final, 0, abort)) return;
  tc_fence_after_sync();
  const bool real = t < rows;
  const size_t ps = ((size_t)b * p.Hq + head0 + t) * p.nsplit + split;
  float4* dst = reinterpret_cast<float4*>(p.o_part + ps * DH);
#pragma unroll 1
  for (int c = 0; c < DH / 32; ++c) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(colO + 32 * c, o);
    tmem_ld_wait(o);
    if (real) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        dst[8 * c + e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                     __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
    }
  }
  if (real) {
    p.m_part[ps] = m_run;
    p.l_part[ps] = l_run;
  }
}

// grid (nsplit, B * Hkv * row_blocks): one split of one (b, K/V head) for up
// to 128 of its group's query heads.
template <int DH>
__global__ void __launch_bounds__(192, 1)
    attn_decode_tc_sm103a(const __grid_constant__ CUtensorMap map_q,
                          const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v, const DecodeTcParams p) {
  using Cfg = DecodeTcCfg<DH>;
  using Smem = DecodeTcSmem<DH>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  volatile int* abort = &sm.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the lengths and the cache may come from the previous kernel in the
  // stream: wait for it before the first global read (a no-op unless this
  // launch is a programmatic dependent)
  griddep_wait();

  const int split = blockIdx.x;
  const int rb = blockIdx.y % p.row_blocks;
  const int bg = blockIdx.y / p.row_blocks;   // b * Hkv + g
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int L = p.seqlens[b];
  if (L < 1 || (!p.ring && L > p.Tmax)) return;   // the combine kernel reports it
  int k_begin, k_end;
  decode_tc_range(p, L, split, k_begin, k_end);
  if (k_begin >= k_end) return;               // no visible key in this split
  const DecodeTcSpan sp = decode_tc_span<Cfg::kKeys>(p, k_begin, k_end);
  const int ntiles = sp.ntiles;
  const int rows = min(128, p.G - 128 * rb);  // real query rows of this CTA
  const int active_warps = (rows + 31) / 32;

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < Cfg::kStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 32 * active_warps);
    }
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.o_final, 1);
    mbar_init(&sm.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == Cfg::kWarpIssuer) {
    tmem_alloc(&sm.tmem_base, Cfg::kCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = sm.tmem_base;

  if (warp == Cfg::kWarpProducer) {
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      decode_tc_producer<DH>(sm, p, &map_q, &map_k, &map_v, bg, rb, sp, abort);
    }
  } else if (warp == Cfg::kWarpIssuer) {
    decode_tc_issuer<DH>(sm, tbase, ntiles, abort);
  } else if (warp < active_warps) {
    decode_tc_softmax<DH>(sm, p, tbase, warp, lane, b, g * p.G + 128 * rb, rows, split, sp,
                          abort);
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kWarpIssuer) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, Cfg::kCols);
  }
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
  // this CTA's partials are written: the combine grid may be scheduled (it
  // still waits for this whole grid to finish before reading them)
  if (threadIdx.x == 0) griddep_launch_dependents();
}

// Merge the splits of one (b, query head): o = sum_s 2^(m_s - M) o_s /
// sum_s 2^(m_s - M) l_s with M the largest m_s (the online-softmax merge),
// in split order.  One block of DH threads per (b, query head).
template <int DH>
__global__ void __launch_bounds__(DH) attn_decode_tc_combine(const DecodeTcParams p) {
  // launched as a programmatic dependent of attn_decode_tc_sm103a: wait until
  // that grid has completed and its writes are visible
  griddep_wait();
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int d = threadIdx.x;
  const int L = p.seqlens[b];
  if (L < 1 || (!p.ring && L > p.Tmax)) {
    // a sequence length outside [1, Tmax] (ring: below 1): zero output, latch the error
    p.o[(size_t)bh * DH + d] = __float2bfloat16(0.f);
    if (d == 0) atomicExch(p.error_word, 1);   // ATTN_ERR_INVALID_ARG
    return;
  }
  const int lo = decode_tc_lo(p, L);
  const int s_first = p.ring ? 0 : lo / p.chunk;
  const int s_last = p.ring ? (L - 1 - lo) / p.chunk : (L - 1) / p.chunk;
  const float* mp = p.m_part + (size_t)bh * p.nsplit;
  const float* lp = p.l_part + (size_t)bh * p.nsplit;
  const float* op = p.o_part + (size_t)bh * p.nsplit * DH;
  // splits in groups of 8, every load of a group issued before any is used
  // (one round of L2 latency per group), merged with a running maximum in
  // split order
  constexpr int kG = 8;
  float M = -INFINITY, o = 0.f, l = 0.f;
  for (int s0 = s_first; s0 <= s_last; s0 += kG) {
    float mv[kG], lv[kG], ov[kG];
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const bool in = s0 + e <= s_last;
      mv[e] = in ? __ldcg(mp + s0 + e) : -INFINITY;
      lv[e] = in ? __ldcg(lp + s0 + e) : 0.f;
      ov[e] = in ? __ldcg(op + (size_t)(s0 + e) * DH + d) : 0.f;
    }
    float Mg = M;
#pragma unroll
    for (int e = 0; e < kG; ++e) Mg = fmaxf(Mg, mv[e]);
    const float c = (M == -INFINITY) ? 0.f : ex2_approx(M - Mg);
    o *= c;
    l *= c;
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const float f = (mv[e] == -INFINITY) ? 0.f : ex2_approx(mv[e] - Mg);
      o = fmaf(f, ov[e], o);
      l = fmaf(f, lv[e], l);
    }
    M = Mg;
  }
  p.o[(size_t)bh * DH + d] = __float2bfloat16(o / l);
}

template <int DH>
constexpr size_t decode_tc_smem_bytes() {
  return sizeof(DecodeTcSmem<DH>) + 1024;   // + alignment slack
}

}  // namespace chs
