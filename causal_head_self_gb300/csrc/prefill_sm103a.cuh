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
// One CTA owns 256 query rows of one (b, h): two 128-row sub-tiles that take
// turns on the tensor core, so that the softmax of one overlaps the MMAs of
// the other.  Roles (320 threads):
//   warps 0-3  softmax + epilogue of sub-tile 0 (thread t owns row t, TMEM lane t)
//   warps 4-7  softmax + epilogue of sub-tile 1
//   warp  8    TMEM allocation; one thread issues every tcgen05.mma
//   warp  9    one thread issues every TMA load (Q once, then K/V tiles)
// With three warps on some SM sub-partitions, 168 registers per thread is the
// most a 10-warp CTA gets; the softmax keeps a 128-score row plus a few
// running values live within that.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+DH),
// O1 [384,384+DH).  P (bf16) is written over the first 64 columns of its S
// and fed to the P.V MMA straight from TMEM.
#pragma once

#include "sm103a_ptx.cuh"

namespace chs {

struct PrefillParams {
  int B, Hq, Hkv, S;
  int causal;   // 1: key j visible to query i only if j <= i
  int window;   // > 0: also only if i - j < window
  float scale_log2;   // softmax scale * log2(e)
  int num_qblocks;    // ceil(S / 256)
  int* error_word;    // set to a nonzero status when a wait gives up
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
  static constexpr int kThreads = 320;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
};

template <int DH>
struct __align__(1024) PrefillSmem {
  using Cfg = PrefillCfg<DH>;
  uint8_t q[2][Cfg::kTileBytes];          // Q sub-tiles; reused as output staging
  uint8_t k[Cfg::kStagesK][Cfg::kTileBytes];
  uint8_t v[Cfg::kStagesV][Cfg::kTileBytes];
  uint64_t q_full;
  uint64_t k_full[Cfg::kStagesK], k_empty[Cfg::kStagesK];
  uint64_t v_full[Cfg::kStagesV], v_empty[Cfg::kStagesV];
  uint64_t s_full[2], p_full[2], o_final[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Geometry of one CTA's work item.
struct PrefillTile {
  int q0;        // first query row of the CTA
  int lo, hi;    // K/V tile range loaded (union over the two sub-tiles)
  int S, causal, window;
  __device__ __forceinline__ int row_first(int s) const { return q0 + 128 * s; }
  __device__ __forceinline__ int row_last(int s) const { return min(q0 + 128 * s + 127, S - 1); }
  __device__ __forceinline__ bool valid(int s) const { return q0 + 128 * s < S; }
  // does sub-tile s see any key of tile j?
  __device__ __forceinline__ bool active(int s, int j) const {
    if (!valid(s)) return false;
    const int c0 = 128 * j, c1 = min(128 * j + 127, S - 1);
    if (causal && c0 > row_last(s)) return false;
    if (window > 0 && c1 < row_first(s) - window + 1) return false;
    return true;
  }
  // is any (row, key) pair of sub-tile s x tile j masked?
  __device__ __forceinline__ bool needs_mask(int s, int j) const {
    const int c0 = 128 * j, c1 = 128 * j + 127;
    if (c1 >= S) return true;
    if (causal && c1 > row_first(s)) return true;
    if (window > 0 && c0 < row_last(s) - window + 1) return true;
    return false;
  }
};

__device__ __forceinline__ PrefillTile prefill_tile_of(const PrefillParams& p, int qb) {
  PrefillTile t;
  t.q0 = qb * 256;
  t.S = p.S;
  t.causal = p.causal;
  t.window = p.window;
  const int nkv = (p.S + 127) / 128;
  const int last_row = min(t.q0 + 255, p.S - 1);
  t.hi = p.causal ? min(nkv - 1, last_row / 128) : nkv - 1;
  t.lo = (p.causal && p.window > 0) ? max(0, t.q0 - p.window + 1) / 128 : 0;
  return t;
}

// Drain wait used at teardown: ignores the abort flag, bounded by time.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

template <int DH>
__global__ void __launch_bounds__(320, 1)
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

  // ---- work item: heaviest query blocks first (causal work grows with qb)
  const int per_qb = p.B * p.Hq;
  const int qb = p.num_qblocks - 1 - (int)(blockIdx.x / per_qb);
  const int bh = (int)(blockIdx.x % per_qb);
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int g = h / (p.Hq / p.Hkv);          // g(h) = floor(h / (H/G))
  const int bh_kv = b * p.Hkv + g;
  const PrefillTile tile = prefill_tile_of(p, qb);

  // ---- setup
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    mbar_init(&sm.q_full, 1);
    for (int i = 0; i < Cfg::kStagesK; ++i) { mbar_init(&sm.k_full[i], 1); mbar_init(&sm.k_empty[i], 1); }
    for (int i = 0; i < Cfg::kStagesV; ++i) { mbar_init(&sm.v_full[i], 1); mbar_init(&sm.v_empty[i], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], 128);
      mbar_init(&sm.o_final[s], 1);
    }
    mbar_init(&sm.mma_done, 1);
    fence_mbarrier_init();
  }
  if (warp == 8) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 9) {
    // =================================================================== TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const int nsub = tile.valid(1) ? 2 : 1;
      mbar_arrive_expect_tx(&sm.q_full, nsub * Cfg::kTileBytes);
      for (int s = 0; s < nsub; ++s)
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_3d(sm.q[s] + hf * Cfg::kBoxBytes, &map_q, &sm.q_full, hf * 64,
                      tile.row_first(s), bh);
      const uint64_t keep = policy_evict_last();   // K/V tiles are re-read by other CTAs
      uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
      uint32_t k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
      for (int j = tile.lo; j <= tile.hi; ++j) {
        if (!mbar_wait(&sm.k_empty[kst], kph ^ 1, abort)) break;
        mbar_arrive_expect_tx(&sm.k_full[kst], Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_3d_hint(sm.k[kst] + hf * Cfg::kBoxBytes, &map_k, &sm.k_full[kst], hf * 64,
                           128 * j, bh_kv, keep);
        k_loaded |= 1u << kst;
        k_par = (k_par & ~(1u << kst)) | (kph << kst);
        if (++kst == Cfg::kStagesK) { kst = 0; kph ^= 1; }

        if (!mbar_wait(&sm.v_empty[vst], vph ^ 1, abort)) break;
        mbar_arrive_expect_tx(&sm.v_full[vst], Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_3d_hint(sm.v[vst] + hf * Cfg::kBoxBytes, &map_v, &sm.v_full[vst], hf * 64,
                           128 * j, bh_kv, keep);
        v_loaded |= 1u << vst;
        v_par = (v_par & ~(1u << vst)) | (vph << vst);
        if (++vst == Cfg::kStagesV) { vst = 0; vph ^= 1; }
      }
      // every copy this thread started has landed before the CTA may exit
      mbar_wait_drain(&sm.q_full, 0);
      for (int i = 0; i < Cfg::kStagesK; ++i)
        if (k_loaded & (1u << i)) mbar_wait_drain(&sm.k_full[i], (k_par >> i) & 1u);
      for (int i = 0; i < Cfg::kStagesV; ++i)
        if (v_loaded & (1u << i)) mbar_wait_drain(&sm.v_full[i], (v_par >> i) & 1u);
    }
  } else if (warp == 8) {
    // =================================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, DH, false, true);
      // S_s = Q_s K^T: K-major operands, 16 columns (32 bytes) of DH per MMA
      auto issue_qk = [&](int s, int kst) {
        const uint32_t d = tbase + (s ? Cfg::kColS1 : Cfg::kColS0);
        const uint32_t qa = smem_u32(sm.q[s]), ka = smem_u32(sm.k[kst]);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
          mma_bf16_ss(d, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                      idesc_qk, kk > 0);
        }
      };
      // O_s (+)= P_s V: P from TMEM (8 columns = 16 keys per MMA), V MN-major
      auto issue_pv = [&](int s, int vst, bool acc) {
        const uint32_t d = tbase + (s ? Cfg::kColO1 : Cfg::kColO0);
        const uint32_t a = tbase + (s ? Cfg::kColS1 : Cfg::kColS0);
        const uint32_t va = smem_u32(sm.v[vst]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(d, a + kk * 8, smem_desc_sw128(va + kk * 2048, Cfg::kBoxBytes, 1024),
                      idesc_pv, (acc || kk > 0) ? 1u : 0u);
      };
      int n_active[2] = {0, 0};
      uint32_t kst = 0, kph = 0, vst = 0, vph = 0, pph0 = 0, pph1 = 0;
      bool pend1 = false, pend_ready = false;
      uint32_t pend_vst = 0, pend_vph = 0;
      bool ok = mbar_wait(&sm.q_full, 0, abort);
      tc_fence_after_sync();
      for (int j = tile.lo; ok && j <= tile.hi; ++j) {
        const bool a0 = tile.active(0, j), a1 = tile.active(1, j);
        if (!(ok = mbar_wait(&sm.k_full[kst], kph, abort))) break;
        tc_fence_after_sync();
        if (a0) {
          issue_qk(0, kst);
          mma_commit(&sm.s_full[0]);
        }
        if (pend1) {   // P.V of sub-tile 1 for the previous tile
          if (!(ok = mbar_wait(&sm.p_full[1], pph1, abort))) break;
          pph1 ^= 1;
          if (!pend_ready && !(ok = mbar_wait(&sm.v_full[pend_vst], pend_vph, abort))) break;
          tc_fence_after_sync();
          issue_pv(1, pend_vst, n_active[1] > 0);
          ++n_active[1];
          mma_commit(&sm.v_empty[pend_vst]);
          pend1 = false;
        }
        if (a1) {
          issue_qk(1, kst);
          mma_commit(&sm.s_full[1]);
        }
        mma_commit(&sm.k_empty[kst]);
        if (++kst == Cfg::kStagesK) { kst = 0; kph ^= 1; }
        bool vready = false;
        if (a0) {
          if (!(ok = mbar_wait(&sm.p_full[0], pph0, abort))) break;
          pph0 ^= 1;
          if (!(ok = mbar_wait(&sm.v_full[vst], vph, abort))) break;
          vready = true;
          tc_fence_after_sync();
          issue_pv(0, vst, n_active[0] > 0);
          ++n_active[0];
        }
        if (a1) {
          pend1 = true;
          pend_vst = vst;
          pend_vph = vph;
          pend_ready = vready;
        } else {
          if (!vready && !(ok = mbar_wait(&sm.v_full[vst], vph, abort))) break;
          mma_commit(&sm.v_empty[vst]);
        }
        if (++vst == Cfg::kStagesV) { vst = 0; vph ^= 1; }
      }
      if (ok && pend1) {
        ok = mbar_wait(&sm.p_full[1], pph1, abort);
        if (ok && !pend_ready) ok = mbar_wait(&sm.v_full[pend_vst], pend_vph, abort);
        if (ok) {
          tc_fence_after_sync();
          issue_pv(1, pend_vst, n_active[1] > 0);
          ++n_active[1];
          mma_commit(&sm.v_empty[pend_vst]);
        }
      }
      if (ok) {
        if (n_active[0] > 0) mma_commit(&sm.o_final[0]);
        if (n_active[1] > 0) mma_commit(&sm.o_final[1]);
      }
      // nothing may still be running on the tensor core at teardown
      mma_commit(&sm.mma_done);
      mbar_wait_drain(&sm.mma_done, 0);
    }
  } else {
    // =================================================================== softmax + epilogue
    const int s = warp / 4;                 // sub-tile
    const int wl = warp % 4;                // warp within the warpgroup = TMEM lane quarter
    const int t = wl * 32 + lane;           // row within the sub-tile = TMEM lane
    const int row = tile.row_first(s) + t;  // absolute query row
    const uint32_t lane_addr = tbase + ((uint32_t)(wl * 32) << 16);
    const uint32_t colS = lane_addr + (s ? Cfg::kColS1 : Cfg::kColS0);
    const uint32_t colO = lane_addr + (s ? Cfg::kColO1 : Cfg::kColO0);
    const float sl2 = p.scale_log2;

    float m_run = -INFINITY;   // running max of scale*log2e*score (lazily updated)
    float l_run = 0.f;         // running sum of exp2(x - m_run)
    int n_done = 0;
    uint32_t sph = 0;
    for (int j = tile.lo; j <= tile.hi; ++j) {
      if (!tile.active(s, j)) continue;
      if (!mbar_wait(&sm.s_full[s], sph, abort)) break;
      sph ^= 1;
      tc_fence_after_sync();

      uint32_t r0[32], r1[32], r2[32], r3[32];
      tmem_ld_32x32b_x32(colS + 0, r0);
      tmem_ld_32x32b_x32(colS + 32, r1);
      tmem_ld_32x32b_x32(colS + 64, r2);
      tmem_ld_32x32b_x32(colS + 96, r3);
      tmem_ld_wait(r0);
      tmem_ld_wait(r1);
      tmem_ld_wait(r2);
      tmem_ld_wait(r3);
      float x[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = __uint_as_float(r0[c]);
        x[32 + c] = __uint_as_float(r1[c]);
        x[64 + c] = __uint_as_float(r2[c]);
        x[96 + c] = __uint_as_float(r3[c]);
      }
      if (tile.needs_mask(s, j)) {
        // visible keys of this row: [klo, khi] (absolute), as column offsets
        const int kv0 = 128 * j;
        int khi = tile.S - 1;
        if (tile.causal) khi = min(khi, row);
        const int klo = tile.window > 0 ? row - tile.window + 1 : 0;
        const int clo = klo - kv0, chi = khi - kv0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < clo || c > chi) x[c] = -INFINITY;
      }
      // row maximum as four independent chains of three-input max
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmax3(x[i], x[4 + i], x[8 + i]);
#pragma unroll
      for (int c = 12; c < 124; c += 8)
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = fmax3(mx[i], x[c + i], x[c + 4 + i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], x[124 + i]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_tile = mt * sl2;
      // lazy rescale: keep the old maximum unless the new one exceeds it by
      // more than 8 (weights stay <= 2^8); the result is exact either way
      // because O and l are divided by the same sum at the end.
      const float m_new = fmaxf(m_run, m_tile);
      const bool upd = (n_done == 0) || (m_new > m_run + 8.0f);
      const float m_use = upd ? m_new : m_run;
      const float corr = (upd && n_done > 0) ? ex2_approx(m_run - m_new) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      // P = exp2(x - m) as bf16 over the first 64 columns of S (the scores
      // die here, before O is touched, to keep register pressure down)
      float ls[4] = {0.f, 0.f, 0.f, 0.f};   // independent partial sums
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2_approx(fmaf(x[32 * c4 + 2 * e], sl2, -msub));
          const float p1 = ex2_approx(fmaf(x[32 * c4 + 2 * e + 1], sl2, -msub));
          ls[e & 3] += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st_32x32b_x16(colS + 16 * c4, pk);
      }
      const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
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
      ++n_done;
    }

    if (n_done > 0 && !*abort && mbar_wait(&sm.o_final[s], 0, abort)) {
      tc_fence_after_sync();
      // O / l -> bf16 -> this warp's 32 rows of the staging tile (Q buffer,
      // 128-byte swizzled like the TMA box) -> TMA store
      const float inv_l = 1.0f / l_run;
      uint8_t* stg = sm.q[s];
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(colO + 32 * c, o);
        tmem_ld_wait(o);
        const int hf = (32 * c) / 64;
        const int chunk0 = ((32 * c) % 64) / 8;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv_l, __uint_as_float(o[8 * q4 + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv_l, __uint_as_float(o[8 * q4 + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv_l, __uint_as_float(o[8 * q4 + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv_l, __uint_as_float(o[8 * q4 + 7]) * inv_l);
          const int chunk = (chunk0 + q4) ^ (t & 7);
          *reinterpret_cast<uint4*>(stg + hf * Cfg::kBoxBytes + t * 128 + chunk * 16) = w;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && tile.row_first(s) + wl * 32 < p.S) {   // boxes wholly past S: nothing to store
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_store_3d(&map_o, stg + hf * Cfg::kBoxBytes + wl * 32 * 128, hf * 64,
                       tile.row_first(s) + wl * 32, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      __syncwarp();
    }
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
