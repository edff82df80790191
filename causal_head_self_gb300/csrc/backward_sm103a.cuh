// backward_sm103a.cuh -- backward pass of causal self-attention on the
// 5th-generation tensor cores (sm_103a), Dh = 64 or 128.
//
// Given q, k, v, the forward output o, its row log-sum-exps and the upstream
// gradient dO, the gradients follow from the chain rule through
// o_i = sum_j p_ij v_j, p_i = softmax(s_i) and s_ij = scale q_i . k_j, with
// the softmax derivative dp_i/dz_j = p_i (delta_ij - p_j) of "Механизм
// внимания", section "Почему делить на корень из d_h":
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),  D_i = dO_i . o_i,
//     dK = scale dS^T Q,   dQ = scale dS K.
// (D_i = sum_j p_ij dp_ij, the contraction of that Jacobian, because
// o_i = sum_j p_ij v_j.)  As section "Эффективные реализации" of the same
// page describes for FlashAttention, the weights P are recomputed block by
// block from the saved log-sum-exp, never stored.
//
// Three kernels, all deterministic (no atomics anywhere):
//   attn_bwd_prep      D_i and the log-sum-exp in units of log2, per row;
//   attn_bwd_dkdv      one CTA per 128-key block of one K/V head: K and V
//                      stay in shared memory while the query blocks of every
//                      query head of the group stream past; S^T = K Q^T and
//                      dP^T = V dO^T land in tensor memory, the softmax
//                      warps turn them into P^T and dS^T (bf16, written over
//                      them), and dV += P^T dO, dK += dS^T Q accumulate in
//                      tensor memory (M = 128 keys);
//   attn_bwd_dq        one CTA per 128-row query block: Q and dO stay, the
//                      key blocks stream past; S = Q K^T and dP = dO V^T
//                      (two dP buffers, so the next block's S and dP run
//                      while dS is formed), dS as above, dQ += dS K
//                      (M = 128 queries).
// dQ is computed by its own pass (recomputing S and dP) instead of being
// reduced across key blocks with atomics: 7 MMAs per block pair instead of 5,
// in exchange for a deterministic result.
//
// Roles: the first 4 kWG warps run the element-wise work and the epilogues,
// kWG warpgroups on kWG column ranges of the same 128 rows (thread t of each
// owns tensor-memory lane t), so each does a share of every step's
// exponentials and the shares run side by side (kWG = 2: two halves); the
// next warp's lane 0 issues every TMA copy, the last warp every MMA (one
// elected lane).  Every wait is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103a_ptx.cuh"

namespace chs {

struct BwdParams {
  int B, Hq, Hkv, S;
  int causal, window;     // as in the forward (window > 0 only with causal)
  float scale_log2;       // scale * log2(e)
  float scale;            // applied to dK and dQ
  int S_pad;              // S rounded up to 128: row stride of lse2 and delta
  int nblk;               // ceil(S / 128)
  int group;              // Hq / Hkv
  int num_items;
  const float* lse2;      // [B * Hq, S_pad] log2 of sum_j 2^(s_ij log2 e); +inf past S
  const float* delta;     // [B * Hq, S_pad] D_i = dO_i . o_i; 0 past S
  __nv_bfloat16* dq;      // [B, Hq, S, DH]
  __nv_bfloat16* dk;      // [B, Hkv, S, DH]
  __nv_bfloat16* dv;      // [B, Hkv, S, DH]
  int* error_word;
  int fault;              // test hook: 4 = the dK/dV pass never loads its first K/V block
};

template <int DH>
struct BwdCfg {
  static constexpr int kBox = 128 * 64 * 2;         // one 128-row x 64-column box
  static constexpr int kTile = (DH / 64) * kBox;    // a 128 x DH tile
  // warps 0 .. 4 kWG - 1: element-wise work (warp w: tensor-memory lanes
  // 32 (w % 4) .., columns kCols (w / 4) .. + kCols - 1 of S and dP); then one
  // TMA warp and one MMA warp
  static constexpr int kWG = 2;                 // element-wise warpgroups
  static constexpr int kCols = 128 / kWG;       // columns of S / dP per warpgroup
  static constexpr int kChunks = kCols / 32;    // 32-column tensor-memory loads per row
  static constexpr int kEW = 128 * kWG;         // element-wise threads
  static constexpr int kThreads = 32 * (4 * kWG + 2);
  static constexpr int kWarpProducer = 4 * kWG, kWarpIssuer = 4 * kWG + 1;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColA0 = 256, kColA1 = 384;
  // the dQ pass has one accumulator (dQ at kColA0): its second dP buffer
  // takes the columns of the dK/dV pass's second accumulator
  static constexpr uint32_t kColDP1 = kColA1;
  static_assert(kColA0 + DH <= kColDP1, "dQ accumulator and the second dP buffer");
};

// Where the bf16 pairs of columns 16 kk .. 16 kk + 15 of a 128-column S or dP
// buffer are written (P over S, dS over dP): each warpgroup's pairs go to the
// first half of its own kCols columns, so that one warpgroup's stores never
// land on columns another warpgroup has still to load.
__host__ __device__ constexpr uint32_t bwd_packed_col(int kk) {
  constexpr int cols = BwdCfg<64>::kCols;
  return (uint32_t)(cols * (16 * kk / cols) + (16 * kk % cols) / 2);
}

// D_i = sum_d dO[i, d] o[i, d] (fp32 products of the bf16 values) and
// lse2_i = lse_i * log2(e) for every row of [B * Hq, S_pad]; rows past S get
// D = 0 and lse2 = +inf (their weights exp2(x - lse2) are then 0).  DH / 8
// lanes per row, 16 bytes of o and of dO each; a block covers kPrepRowSets
// row sets, all of whose loads are issued before the first is used.
constexpr int kPrepRowSets = 4;
template <int DH>
constexpr int bwd_prep_rows_per_block() { return kPrepRowSets * 256 / (DH / 8); }

template <int DH>
__global__ void __launch_bounds__(256)
    attn_bwd_prep(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                  const float* __restrict__ lse, float* __restrict__ lse2,
                  float* __restrict__ delta, long long rows, int S, int S_pad) {
  constexpr int kLanes = DH / 8;                // 16 or 8 lanes per row
  constexpr int kRowsPerSet = 256 / kLanes;
  // o, dO and lse may come from the previous kernel in the stream
  griddep_wait();
  griddep_launch_dependents();
  const int sub = threadIdx.x % kLanes;
  long long r[kPrepRowSets];
  bool valid[kPrepRowSets];
  uint4 a[kPrepRowSets], b[kPrepRowSets];
#pragma unroll
  for (int k = 0; k < kPrepRowSets; ++k) {
    r[k] = (long long)blockIdx.x * bwd_prep_rows_per_block<DH>() + k * kRowsPerSet +
           threadIdx.x / kLanes;
    const long long bh = r[k] / S_pad;
    const int i = (int)(r[k] - bh * S_pad);
    valid[k] = r[k] < rows && i < S;
    a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
    if (valid[k]) {
      const size_t base = ((size_t)bh * S + i) * DH + 8 * sub;
      a[k] = *reinterpret_cast<const uint4*>(o + base);
      b[k] = *reinterpret_cast<const uint4*>(dout + base);
    }
  }
#pragma unroll
  for (int k = 0; k < kPrepRowSets; ++k) {
    const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
    const uint32_t wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
      acc = fmaf(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wb[e] & 0xffff0000u), acc);
    }
#pragma unroll
    for (int m = kLanes / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (sub == 0 && r[k] < rows) {
      const long long bh = r[k] / S_pad;
      const int i = (int)(r[k] - bh * S_pad);
      delta[r[k]] = valid[k] ? acc : 0.f;
      lse2[r[k]] = valid[k] ? lse[(size_t)bh * S + i] * 1.4426950408889634f
                            : __int_as_float(0x7f800000);
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// x if off <= span (unsigned), else 0 (a predicated select; see keep_if_le)
__device__ __forceinline__ float zero_unless_le(float x, uint32_t off, uint32_t span) {
  float d;
  asm("{\n .reg .pred p;\n setp.le.u32 p, %1, %2;\n selp.f32 %0, %3, 0f00000000, p;\n}"
      : "=f"(d) : "r"(off), "r"(span), "f"(x));
  return d;
}

__device__ __forceinline__ void bwd_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Heaviest-first snake order over the CTAs (as in the forward kernels).
__device__ __forceinline__ int bwd_item(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Query blocks [lo, hi] that see some key of key block kb (128-row blocks).
__device__ __forceinline__ void bwd_qblocks_of(const BwdParams& p, int kb, int& lo, int& hi) {
  if (!p.causal) {
    lo = 0;
    hi = p.nblk - 1;
    return;
  }
  lo = kb;   // query i sees key j only if j <= i
  hi = p.nblk - 1;
  if (p.window > 0) hi = min(hi, (128 * kb + 127 + p.window - 1) / 128);   // i - j < W
}

// Key blocks [lo, hi] that query block qb sees.
__device__ __forceinline__ void bwd_kblocks_of(const BwdParams& p, int qb, int& lo, int& hi) {
  if (!p.causal) {
    lo = 0;
    hi = p.nblk - 1;
    return;
  }
  hi = qb;
  lo = p.window > 0 ? max(0, 128 * qb - p.window + 1) / 128 : 0;
}

// Does some (query, key) pair of query block qb x key block kb fall outside
// the mask (or past S)?
__device__ __forceinline__ bool bwd_needs_mask(const BwdParams& p, int qb, int kb) {
  if (128 * kb + 127 >= p.S || 128 * qb + 127 >= p.S) return true;
  if (!p.causal) return false;
  if (128 * kb + 127 > 128 * qb) return true;                                  // j > i somewhere
  if (p.window > 0 && 128 * qb + 127 - 128 * kb >= p.window) return true;      // i - j >= W somewhere
  return false;
}

// ============================================================ dK, dV pass

template <int DH>
struct __align__(1024) BwdKvSmem {
  using Cfg = BwdCfg<DH>;
  uint8_t k[Cfg::kTile];           // this item's key block (stays)
  uint8_t v[Cfg::kTile];           // this item's value block (stays)
  uint8_t q[2][Cfg::kTile];        // query blocks, two stages
  uint8_t dO[2][Cfg::kTile];       // their output gradients
  float lse2[2][128];              // their log-sum-exps (log2 units)
  float dlt[2][128];               // their D_i
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, acc_final, mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Item w of the dK/dV pass: key block kb (heaviest, i.e. earliest, first
// under a causal mask) of K/V head bkv = b * Hkv + g.
struct BwdKvItem {
  int kb, bkv, b, g, lo, hi;
};

__device__ __forceinline__ BwdKvItem bwd_kv_item_of(const BwdParams& p, int w) {
  BwdKvItem r;
  const int per = p.B * p.Hkv;
  r.kb = w / per;
  r.bkv = w - r.kb * per;
  r.b = r.bkv / p.Hkv;
  r.g = r.bkv - r.b * p.Hkv;
  bwd_qblocks_of(p, r.kb, r.lo, r.hi);
  return r;
}

template <int DH>
__device__ __forceinline__ void bwd_dkdv_producer(BwdKvSmem<DH>& sm, const BwdParams& p,
                                                  const CUtensorMap* map_q,
                                                  const CUtensorMap* map_k,
                                                  const CUtensorMap* map_v,
                                                  const CUtensorMap* map_do, volatile int* abort) {
  using Cfg = BwdCfg<DH>;
  constexpr int kBoxes = DH / 64;
  const uint64_t keep = policy_evict_last();   // query blocks are re-read by other key blocks
  uint32_t u = 0, loaded = 0, par = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd_kv_item_of(p, w);
    if (items > 0 && !(ok = mbar_wait(&sm.kv_empty, (uint32_t)(items - 1) & 1u, abort))) break;
    // (checked builds: a key block of the sequence, of a K/V head of the batch)
    const bool kv_in_range = attn_check(I.kb >= 0 && 128 * I.kb < p.S && I.bkv >= 0 &&
                                            I.bkv < p.B * p.Hkv,
                                        p.error_word);
    mbar_arrive_expect_tx(&sm.kv_full, kv_in_range ? 2u * Cfg::kTile : 0u);
    if (kv_in_range && (p.fault != 4 || it != 0)) {   // (the test hook withholds one K/V block)
      for (int hf = 0; hf < kBoxes; ++hf) {
        tma_load_3d(sm.k + hf * Cfg::kBox, map_k, &sm.kv_full, 64 * hf, 128 * I.kb, I.bkv);
        tma_load_3d(sm.v + hf * Cfg::kBox, map_v, &sm.kv_full, 64 * hf, 128 * I.kb, I.bkv);
      }
    }
    ++items;
    for (int hh = 0; ok && hh < p.group; ++hh) {
      const int bh = I.b * p.Hq + I.g * p.group + hh;
      for (int qb = I.lo; qb <= I.hi; ++qb, ++u) {
        const int st = (int)(u & 1u);
        const uint32_t ph = (u >> 1) & 1u;
        if (!(ok = mbar_wait(&sm.q_empty[st], ph ^ 1u, abort))) break;
        const size_t row0 = (size_t)bh * p.S_pad + 128 * qb;
        // (checked builds: a query block of the sequence, of a query head of
        // the batch, whose per-row statistics lie inside the workspace)
        const bool in_range = attn_check(qb >= 0 && 128 * qb < p.S && bh >= 0 && bh < p.B * p.Hq &&
                                             row0 + 128 <= (size_t)p.B * p.Hq * p.S_pad,
                                         p.error_word);
        mbar_arrive_expect_tx(&sm.q_full[st], in_range ? 2u * Cfg::kTile + 2u * 512u : 0u);
        for (int hf = 0; in_range && hf < kBoxes; ++hf) {
          tma_load_3d_hint(sm.q[st] + hf * Cfg::kBox, map_q, &sm.q_full[st], 64 * hf, 128 * qb, bh,
                           keep);
          tma_load_3d_hint(sm.dO[st] + hf * Cfg::kBox, map_do, &sm.q_full[st], 64 * hf, 128 * qb,
                           bh, keep);
        }
        if (in_range) {
          bulk_load(sm.lse2[st], p.lse2 + row0, 512, &sm.q_full[st], keep);
          bulk_load(sm.dlt[st], p.delta + row0, 512, &sm.q_full[st], keep);
        }
        loaded |= 1u << st;
        par = (par & ~(1u << st)) | (ph << st);
      }
    }
  }
  // every copy this thread started has landed before the CTA may exit
  if (items > 0) bwd_wait_drain(&sm.kv_full, (uint32_t)(items - 1) & 1u);
  for (int i = 0; i < 2; ++i)
    if (loaded & (1u << i)) bwd_wait_drain(&sm.q_full[i], (par >> i) & 1u);
}

// MMA issue order per item of N steps (one step = one query block of one
// query head): S(0), dP(0), then per step n: dV(n) once P(n) is written,
// S(n+1) (its columns held P(n), which dV(n), issued before it, reads),
// dK(n) once dS(n) is written, dP(n+1) (its columns held dS(n)).  The
// element-wise work of step n+1 therefore overlaps dK(n) and dP(n+1).
template <int DH>
__device__ __forceinline__ void bwd_dkdv_issuer(BwdKvSmem<DH>& sm, const BwdParams& p,
                                                volatile int* abort) {
  using Cfg = BwdCfg<DH>;
  constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t idesc_acc = idesc_bf16_f32(128, DH, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kBox, 1024);
  const uint64_t dk_ = kKmajor | (smem_u32(sm.k) >> 4);
  const uint64_t dv_ = kKmajor | (smem_u32(sm.v) >> 4);
  const uint64_t dq_k = kKmajor | (smem_u32(sm.q[0]) >> 4);
  const uint64_t ddo_k = kKmajor | (smem_u32(sm.dO[0]) >> 4);
  const uint64_t dq_mn = kMnMajor | (smem_u32(sm.q[0]) >> 4);
  const uint64_t ddo_mn = kMnMajor | (smem_u32(sm.dO[0]) >> 4);
  constexpr uint64_t kStage = Cfg::kTile >> 4;   // q[1] - q[0] (and dO) in descriptor units
  // D (128 x 128) = A (128 x DH) B^T, both K-major (DH contiguous)
  auto mma_nt = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const uint32_t off = ((kk / 4) * Cfg::kBox + (kk % 4) * 32) >> 4;
      mma_bf16_ss_warp(d, a + off, b + off, idesc_ss, kk > 0 ? 1u : 0u);
    }
  };
  // D (128 x DH) (+)= A (tensor memory, 128 x 128 bf16 pairs at bwd_packed_col) B,
  // B MN-major (DH contiguous)
  auto mma_acc = [&](uint32_t d, uint32_t a, uint64_t b, bool first) {
#pragma unroll
    for (int kk = 0; kk < 128 / 16; ++kk)
      mma_bf16_ts_warp(d, a + bwd_packed_col(kk), b + kk * (2048 >> 4), idesc_acc,
                       (!first || kk > 0) ? 1u : 0u);
  };
  auto wait_all = [&](uint64_t* bar, uint32_t ph) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort));
  };
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd_kv_item_of(p, w);
    const int N = p.group * (I.hi - I.lo + 1);
    if (!(ok = wait_all(&sm.kv_full, (uint32_t)items & 1u))) break;
    ++items;
    if (!(ok = wait_all(&sm.q_full[u & 1u], (u >> 1) & 1u))) break;
    tc_fence_after_sync();
    mma_nt(Cfg::kColS, dk_, dq_k + (u & 1u) * kStage);
    mma_commit_warp(&sm.s_full);
    mma_nt(Cfg::kColDP, dv_, ddo_k + (u & 1u) * kStage);
    mma_commit_warp(&sm.dp_full);
    if (N == 1) mma_commit_warp(&sm.kv_empty);
    for (int n = 0; n < N; ++n, ++u) {
      const uint64_t st = u & 1u, st1 = (u + 1) & 1u;
      if (!(ok = wait_all(&sm.p_full, u & 1u))) break;
      tc_fence_after_sync();
      mma_acc(Cfg::kColA0, Cfg::kColS, ddo_mn + st * kStage, n == 0);   // dV += P^T dO
      if (n + 1 < N) {
        if (!(ok = wait_all(&sm.q_full[st1], ((u + 1) >> 1) & 1u))) break;
        tc_fence_after_sync();
        mma_nt(Cfg::kColS, dk_, dq_k + st1 * kStage);                  // S^T(n+1) = K Q^T
        mma_commit_warp(&sm.s_full);
      }
      if (!(ok = wait_all(&sm.ds_full, u & 1u))) break;
      tc_fence_after_sync();
      mma_acc(Cfg::kColA1, Cfg::kColDP, dq_mn + st * kStage, n == 0);   // dK += dS^T Q
      mma_commit_warp(&sm.q_empty[st]);
      if (n + 1 < N) {
        mma_nt(Cfg::kColDP, dv_, ddo_k + st1 * kStage);                 // dP^T(n+1) = V dO^T
        mma_commit_warp(&sm.dp_full);
        if (n + 2 == N) mma_commit_warp(&sm.kv_empty);
      }
    }
    if (ok) mma_commit_warp(&sm.acc_final);
  }
  mma_commit_warp(&sm.mma_done);
  bwd_wait_drain(&sm.mma_done, 0);
}

// Store 32 fp32 accumulator columns (times `mul`) as bf16 to dst (16-byte aligned).
__device__ __forceinline__ void bwd_store32(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(__uint_as_float(r[8 * q + 2 * e]) * mul,
                         __uint_as_float(r[8 * q + 2 * e + 1]) * mul);
    d[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Element-wise work of the dK/dV pass (warps 0-7; thread t of warpgroup wg
// owns key row k0 + t, tensor-memory lane t, and query columns
// kCols wg .. kCols (wg + 1) - 1).  Per step: P^T = exp2(S^T * scale*log2e - lse2[query])
// (0 where masked), written as bf16 pairs (see bwd_packed_col) and kept in
// fp32 registers; then dS^T = P^T o (dP^T - D[query]), as bf16 pairs over dP^T.
// Per item: the first half of the warpgroups write dV, the second scale * dK.
template <int DH>
__device__ __forceinline__ void bwd_dkdv_softmax(BwdKvSmem<DH>& sm, const BwdParams& p,
                                                 uint32_t tbase, volatile int* abort, int warp,
                                                 int lane) {
  using Cfg = BwdCfg<DH>;
  const int wg = warp / 4;
  const int t = (warp % 4) * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)((warp % 4) * 32) << 16);
  const uint32_t colS = lane_addr + Cfg::kColS + Cfg::kCols * wg;   // this warpgroup's scores
  const uint32_t colDP = lane_addr + Cfg::kColDP + Cfg::kCols * wg;
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdKvItem I = bwd_kv_item_of(p, w);
    const int j = 128 * I.kb + t;   // this thread's key
    for (int hh = 0; ok && hh < p.group; ++hh) {
      for (int qb = I.lo; qb <= I.hi; ++qb, ++u) {
        const int st = (int)(u & 1u);
        // the stage's lse2 / D (bulk copies counted on q_full)
        if (!(ok = mbar_wait(&sm.q_full[st], (u >> 1) & 1u, abort))) break;
        if (!(ok = mbar_wait(&sm.s_full, u & 1u, abort))) break;
        tc_fence_after_sync();
        const float4* L4 = reinterpret_cast<const float4*>(sm.lse2[st] + Cfg::kCols * wg);
        const float4* D4 = reinterpret_cast<const float4*>(sm.dlt[st] + Cfg::kCols * wg);
        // visible query columns of key j: c in [clo, chi] of this warpgroup's
        // columns (query i = 128 qb + kCols wg + c)
        const bool msk = bwd_needs_mask(p, qb, I.kb);
        const int i0 = 128 * qb + Cfg::kCols * wg;
        int clo = 0, chi = Cfg::kCols - 1;
        if (p.causal) clo = j - i0;                                     // i >= j
        if (p.window > 0) chi = min(chi, j - i0 + p.window - 1);        // i - j < W
        chi = min(chi, p.S - 1 - i0);                                   // i < S
        const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
        if (chi < clo) clo = 1 << 30;

        uint32_t x[Cfg::kChunks][32];
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) tmem_ld_32x32b_x32(colS + 32 * c, x[c]);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) tmem_ld_wait(x[c]);
        float pf[Cfg::kCols];   // P^T of this row's columns (fp32)
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
          uint32_t w16[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l = L4[8 * c + e4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e4 + h, col = 32 * c + 2 * e;
              const float2 xs = __ffma2_rn(
                  make_float2(__uint_as_float(x[c][2 * e]), __uint_as_float(x[c][2 * e + 1])), sl2,
                  h ? make_float2(-l.z, -l.w) : make_float2(-l.x, -l.y));
              float a = ex2_approx(xs.x), b = ex2_approx(xs.y);
              if (msk) {
                a = zero_unless_le(a, (uint32_t)(col - clo), span);
                b = zero_unless_le(b, (uint32_t)(col + 1 - clo), span);
              }
              pf[col] = a;
              pf[col + 1] = b;
              w16[e] = pack_bf16x2(a, b);
            }
          }
          tmem_st_32x32b_x16(colS + 16 * c, w16);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sm.p_full);

        if (!(ok = mbar_wait(&sm.dp_full, u & 1u, abort))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
          uint32_t y[32];
          tmem_ld_32x32b_x32(colDP + 32 * c, y);
          tmem_ld_wait(y);
          uint32_t w16[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 d = D4[8 * c + e4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e4 + h, col = 32 * c + 2 * e;
              const float2 dd = __fadd2_rn(
                  make_float2(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1])),
                  h ? make_float2(-d.z, -d.w) : make_float2(-d.x, -d.y));
              const float2 ds = __fmul2_rn(make_float2(pf[col], pf[col + 1]), dd);
              w16[e] = pack_bf16x2(ds.x, ds.y);
            }
          }
          // (the pairs land on columns this thread loaded in chunk 0)
          tmem_st_32x32b_x16(colDP + 16 * c, w16);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sm.ds_full);
      }
    }
    if (!ok) break;

    // ---- epilogue: dV and scale * dK of key j
    if (!(ok = mbar_wait(&sm.acc_final, (uint32_t)items & 1u, abort))) break;
    ++items;
    tc_fence_after_sync();
    const bool store = j < p.S;
    const size_t row = ((size_t)I.bkv * p.S + j) * DH;
    constexpr int kHalf = Cfg::kWG / 2;              // warpgroups per accumulator
    const bool is_dv = wg < kHalf;
    __nv_bfloat16* dst = (is_dv ? p.dv : p.dk) + row;
    const uint32_t colA = lane_addr + (is_dv ? Cfg::kColA0 : Cfg::kColA1);
    const float mul = is_dv ? 1.0f : p.scale;
#pragma unroll 1
    for (int c = wg % kHalf; c < DH / 32; c += kHalf) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(colA + 32 * c, r);
      tmem_ld_wait(r);
      if (store) bwd_store32(dst + 32 * c, r, mul);
    }
    // the next item's first dV / dK overwrite the accumulators only after
    // this thread's next arrive on p_full / ds_full, which follows these loads
  }
}

template <int DH>
__global__ void __launch_bounds__(BwdCfg<DH>::kThreads, 1)
    attn_bwd_dkdv(const __grid_constant__ CUtensorMap map_q,
                  const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v,
                  const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using Cfg = BwdCfg<DH>;
  using Smem = BwdKvSmem<DH>;
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
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.dp_full, 1);
    mbar_init(&sm.p_full, Cfg::kEW);
    mbar_init(&sm.ds_full, Cfg::kEW);
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
  // launched as a programmatic dependent of the prep kernel: its D and lse2
  // (and the inputs) are read only after it has completed; then the dQ pass,
  // which needs no output of this one, may be scheduled on SMs this grid frees
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const uint32_t tbase = sm.tmem_base;
  // compile-time tensor-memory columns: the allocation must start at column 0
  if (tbase != 0 && threadIdx.x == 0) sm.abort_flag = 1;
  if (tbase == 0) {
    if (warp == Cfg::kWarpProducer) {
      if (lane == 0) bwd_dkdv_producer<DH>(sm, p, &map_q, &map_k, &map_v, &map_do, abort);
    } else if (warp == Cfg::kWarpIssuer) {
      bwd_dkdv_issuer<DH>(sm, p, abort);
    } else {
      bwd_dkdv_softmax<DH>(sm, p, tbase, abort, warp, lane);
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
}

// ============================================================ dQ pass

template <int DH>
struct __align__(1024) BwdQSmem {
  using Cfg = BwdCfg<DH>;
  static constexpr int kStagesK = 3, kStagesV = 2;
  uint8_t q[Cfg::kTile];           // this item's query block (stays)
  uint8_t dO[Cfg::kTile];          // and its output gradient
  uint8_t k[kStagesK][Cfg::kTile];   // key blocks: read by S(n) and dQ(n)
  uint8_t v[kStagesV][Cfg::kTile];   // value blocks: read by dP(n) only
  uint64_t q_full, q_empty;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full, s_free, acc_final, mma_done;
  uint64_t dp_full[2], ds_full[2];   // per dP / dS buffer
  uint32_t tmem_base;
  int abort_flag;
};

// Item w of the dQ pass: query block qb (heaviest, i.e. last, first under a
// causal mask) of query head bh = b * Hq + h.
struct BwdQItem {
  int qb, bh, bkv, lo, hi;
};

__device__ __forceinline__ BwdQItem bwd_q_item_of(const BwdParams& p, int w) {
  BwdQItem r;
  const int per = p.B * p.Hq;
  const int blk = w / per;
  r.qb = p.nblk - 1 - blk;
  r.bh = w - blk * per;
  const int b = r.bh / p.Hq;
  r.bkv = b * p.Hkv + (r.bh - b * p.Hq) / p.group;   // g(h) = floor(h / (H/G))
  bwd_kblocks_of(p, r.qb, r.lo, r.hi);
  return r;
}

template <int DH>
__device__ __forceinline__ void bwd_dq_producer(BwdQSmem<DH>& sm, const BwdParams& p,
                                                const CUtensorMap* map_q, const CUtensorMap* map_k,
                                                const CUtensorMap* map_v,
                                                const CUtensorMap* map_do, volatile int* abort) {
  using Cfg = BwdCfg<DH>;
  using Smem = BwdQSmem<DH>;
  constexpr int kBoxes = DH / 64;
  const uint64_t keep = policy_evict_last();   // key blocks are re-read by other query blocks
  uint32_t u = 0, k_loaded = 0, k_par = 0, v_loaded = 0, v_par = 0;
  uint32_t ks = 0, kph = 0;   // K stage and its phase for block u (u % 3, (u / 3) & 1)
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd_q_item_of(p, w);
    if (items > 0 && !(ok = mbar_wait(&sm.q_empty, (uint32_t)(items - 1) & 1u, abort))) break;
    // (checked builds: a query block of the sequence, of a query head of the batch)
    const bool q_in_range = attn_check(I.qb >= 0 && 128 * I.qb < p.S && I.bh >= 0 &&
                                           I.bh < p.B * p.Hq,
                                       p.error_word);
    mbar_arrive_expect_tx(&sm.q_full, q_in_range ? 2u * Cfg::kTile : 0u);
    for (int hf = 0; q_in_range && hf < kBoxes; ++hf) {
      tma_load_3d(sm.q + hf * Cfg::kBox, map_q, &sm.q_full, 64 * hf, 128 * I.qb, I.bh);
      tma_load_3d(sm.dO + hf * Cfg::kBox, map_do, &sm.q_full, 64 * hf, 128 * I.qb, I.bh);
    }
    ++items;
    for (int kb = I.lo; kb <= I.hi; ++kb, ++u) {
      // (checked builds: a key block of the sequence, of a K/V head of the batch)
      const bool in_range = attn_check(kb >= 0 && 128 * kb < p.S && I.bkv >= 0 &&
                                           I.bkv < p.B * p.Hkv,
                                       p.error_word);
      const uint32_t bytes = in_range ? (uint32_t)Cfg::kTile : 0u;
      if (!(ok = mbar_wait(&sm.k_empty[ks], kph ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.k_full[ks], bytes);
      for (int hf = 0; in_range && hf < kBoxes; ++hf)
        tma_load_3d_hint(sm.k[ks] + hf * Cfg::kBox, map_k, &sm.k_full[ks], 64 * hf, 128 * kb,
                         I.bkv, keep);
      k_loaded |= 1u << ks;
      k_par = (k_par & ~(1u << ks)) | (kph << ks);
      if (++ks == Smem::kStagesK) { ks = 0; kph ^= 1u; }
      const uint32_t vs = u & 1u, vph = (u >> 1) & 1u;
      if (!(ok = mbar_wait(&sm.v_empty[vs], vph ^ 1u, abort))) break;
      mbar_arrive_expect_tx(&sm.v_full[vs], bytes);
      for (int hf = 0; in_range && hf < kBoxes; ++hf)
        tma_load_3d_hint(sm.v[vs] + hf * Cfg::kBox, map_v, &sm.v_full[vs], 64 * hf, 128 * kb,
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
// of two dP buffers, then dQ(n) once dS(n) is written over dP(n).  With two
// buffers the next block's S and dP run on the tensor core while the
// element-wise warps turn dP(n) into dS(n), and dQ(n) is the only MMA that
// waits for them; dP(n+2) reuses dP(n)'s columns after dQ(n), issued before
// it, has read dS(n) there.  A value block is released when its dP is done,
// a key block only after dQ: three key stages let block n+2's keys load
// while blocks n and n+1 are in use.
template <int DH>
__device__ __forceinline__ void bwd_dq_issuer(BwdQSmem<DH>& sm, const BwdParams& p,
                                              volatile int* abort) {
  using Cfg = BwdCfg<DH>;
  using Smem = BwdQSmem<DH>;
  constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t idesc_acc = idesc_bf16_f32(128, DH, false, true);
  constexpr uint64_t kKmajor = smem_desc_sw128(0, 16, 1024);
  constexpr uint64_t kMnMajor = smem_desc_sw128(0, Cfg::kBox, 1024);
  const uint64_t dq_ = kKmajor | (smem_u32(sm.q) >> 4);
  const uint64_t ddo_ = kKmajor | (smem_u32(sm.dO) >> 4);
  const uint64_t dk_k = kKmajor | (smem_u32(sm.k[0]) >> 4);
  const uint64_t dv_k = kKmajor | (smem_u32(sm.v[0]) >> 4);
  const uint64_t dk_mn = kMnMajor | (smem_u32(sm.k[0]) >> 4);
  constexpr uint64_t kStage = Cfg::kTile >> 4;
  auto mma_nt = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const uint32_t off = ((kk / 4) * Cfg::kBox + (kk % 4) * 32) >> 4;
      mma_bf16_ss_warp(d, a + off, b + off, idesc_ss, kk > 0 ? 1u : 0u);
    }
  };
  auto wait_all = [&](uint64_t* bar, uint32_t ph) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, ph, abort));
  };
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd_q_item_of(p, w);
    const int N = I.hi - I.lo + 1;
    if (!(ok = wait_all(&sm.q_full, (uint32_t)items & 1u))) break;
    ++items;
    // block u (counted across items) uses K stage u % 3, V stage u & 1 and
    // dP buffer u & 1
    auto col_dp = [](uint32_t b) { return b ? Cfg::kColDP1 : Cfg::kColDP; };
    auto kst = [](uint32_t x) { return x % (uint32_t)Smem::kStagesK; };
    auto kph = [](uint32_t x) { return (x / (uint32_t)Smem::kStagesK) & 1u; };
    if (!(ok = wait_all(&sm.k_full[kst(u)], kph(u)))) break;
    tc_fence_after_sync();
    mma_nt(Cfg::kColS, dq_, dk_k + kst(u) * kStage);
    mma_commit_warp(&sm.s_full);
    if (!(ok = wait_all(&sm.v_full[u & 1u], (u >> 1) & 1u))) break;
    tc_fence_after_sync();
    mma_nt(col_dp(u & 1u), ddo_, dv_k + (u & 1u) * kStage);
    mma_commit_warp(&sm.dp_full[u & 1u]);
    mma_commit_warp(&sm.v_empty[u & 1u]);
    if (N == 1) mma_commit_warp(&sm.q_empty);
    for (int n = 0; n < N; ++n, ++u) {
      const uint32_t st = u & 1u, st1 = (u + 1) & 1u;
      if (n + 1 < N) {
        if (!(ok = wait_all(&sm.s_free, u & 1u))) break;
        if (!(ok = wait_all(&sm.k_full[kst(u + 1)], kph(u + 1)))) break;
        tc_fence_after_sync();
        mma_nt(Cfg::kColS, dq_, dk_k + kst(u + 1) * kStage);             // S(n+1) = Q K^T
        mma_commit_warp(&sm.s_full);
        if (!(ok = wait_all(&sm.v_full[st1], ((u + 1) >> 1) & 1u))) break;
        tc_fence_after_sync();
        mma_nt(col_dp(st1), ddo_, dv_k + st1 * kStage);                  // dP(n+1) = dO V^T
        mma_commit_warp(&sm.dp_full[st1]);
        mma_commit_warp(&sm.v_empty[st1]);
        if (n + 2 == N) mma_commit_warp(&sm.q_empty);
      }
      if (!(ok = wait_all(&sm.ds_full[st], (u >> 1) & 1u))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < 128 / 16; ++kk)                              // dQ += dS K
        mma_bf16_ts_warp(Cfg::kColA0, col_dp(st) + bwd_packed_col(kk),
                         dk_mn + kst(u) * kStage + kk * (2048 >> 4),
                         idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
      mma_commit_warp(&sm.k_empty[kst(u)]);
    }
    if (ok) mma_commit_warp(&sm.acc_final);
  }
  mma_commit_warp(&sm.mma_done);
  bwd_wait_drain(&sm.mma_done, 0);
}

// Element-wise work of the dQ pass (warps 0-7; thread t of warpgroup wg owns
// query row 128 qb + t and key columns kCols wg .. kCols (wg + 1) - 1):
// P = exp2(S * scale*log2e - lse2_i) (0 where masked), kept in fp32
// registers; dS = P o (dP - D_i) as bf16 pairs over dP (see bwd_packed_col).
// Per item: scale * dQ out, the 32-column chunks dealt to the warpgroups.
template <int DH>
__device__ __forceinline__ void bwd_dq_softmax(BwdQSmem<DH>& sm, const BwdParams& p,
                                               uint32_t tbase, volatile int* abort, int warp,
                                               int lane) {
  using Cfg = BwdCfg<DH>;
  const int wg = warp / 4;
  const int t = (warp % 4) * 32 + lane;
  const uint32_t lane_addr = tbase + ((uint32_t)((warp % 4) * 32) << 16);
  const uint32_t colS = lane_addr + Cfg::kColS + Cfg::kCols * wg;
  const uint32_t colDP0 = lane_addr + Cfg::kColDP + Cfg::kCols * wg;    // dP buffer 0
  const uint32_t colDP1 = lane_addr + Cfg::kColDP1 + Cfg::kCols * wg;   // dP buffer 1
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
  uint32_t u = 0;
  int items = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int w = bwd_item(it, blockIdx.x, gridDim.x);
    if (w >= p.num_items) break;
    const BwdQItem I = bwd_q_item_of(p, w);
    const int i = 128 * I.qb + t;   // this thread's query
    const float L = p.lse2[(size_t)I.bh * p.S_pad + i];
    const float Di = p.delta[(size_t)I.bh * p.S_pad + i];
    const float2 negL = make_float2(-L, -L), negD = make_float2(-Di, -Di);
    for (int kb = I.lo; kb <= I.hi; ++kb, ++u) {
      if (!(ok = mbar_wait(&sm.s_full, u & 1u, abort))) break;
      tc_fence_after_sync();
      // visible keys of query i: [klo, khi], as columns [clo, chi] of this warpgroup's
      const bool msk = bwd_needs_mask(p, I.qb, kb);
      const int j0 = 128 * kb + Cfg::kCols * wg;
      int khi = p.S - 1;
      if (p.causal) khi = min(khi, i);
      const int klo = p.window > 0 ? i - p.window + 1 : 0;
      int clo = klo - j0;
      const int chi = khi - j0;
      const uint32_t span = chi >= clo ? (uint32_t)(chi - clo) : 0u;
      if (chi < clo) clo = 1 << 30;

      uint32_t x[Cfg::kChunks][32];
#pragma unroll
      for (int c = 0; c < Cfg::kChunks; ++c) tmem_ld_32x32b_x32(colS + 32 * c, x[c]);
#pragma unroll
      for (int c = 0; c < Cfg::kChunks; ++c) tmem_ld_wait(x[c]);
      // S is in registers: the next S may overwrite it
      tc_fence_before_sync();
      mbar_arrive(&sm.s_free);
      float pf[Cfg::kCols];
#pragma unroll
      for (int e = 0; e < Cfg::kCols / 2; ++e) {
        const int col = 2 * e, c = col / 32, k = col % 32;
        const float2 xs = __ffma2_rn(make_float2(__uint_as_float(x[c][k]), __uint_as_float(x[c][k + 1])),
                                     sl2, negL);
        float a = ex2_approx(xs.x), b = ex2_approx(xs.y);
        if (msk) {
          a = zero_unless_le(a, (uint32_t)(col - clo), span);
          b = zero_unless_le(b, (uint32_t)(col + 1 - clo), span);
        }
        pf[col] = a;
        pf[col + 1] = b;
      }

      const uint32_t b = u & 1u;   // this block's dP buffer
      const uint32_t colDP = b ? colDP1 : colDP0;
      if (!(ok = mbar_wait(&sm.dp_full[b], (u >> 1) & 1u, abort))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c = 0; c < Cfg::kChunks; ++c) {
        uint32_t y[32];
        tmem_ld_32x32b_x32(colDP + 32 * c, y);
        tmem_ld_wait(y);
        uint32_t w16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = 32 * c + 2 * e;
          const float2 dd = __fadd2_rn(
              make_float2(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1])), negD);
          const float2 ds = __fmul2_rn(make_float2(pf[col], pf[col + 1]), dd);
          w16[e] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st_32x32b_x16(colDP + 16 * c, w16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sm.ds_full[b]);
    }
    if (!ok) break;

    // ---- epilogue: scale * dQ of query i, this warpgroup's chunks of the columns
    if (!(ok = mbar_wait(&sm.acc_final, (uint32_t)items & 1u, abort))) break;
    ++items;
    tc_fence_after_sync();
    const bool store = i < p.S;
    const size_t row = ((size_t)I.bh * p.S + i) * DH;
#pragma unroll 1
    for (int c = wg; c < DH / 32; c += Cfg::kWG) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(lane_addr + Cfg::kColA0 + 32 * c, r);
      tmem_ld_wait(r);
      if (store) bwd_store32(p.dq + row + 32 * c, r, p.scale);
    }
  }
}

template <int DH>
__global__ void __launch_bounds__(BwdCfg<DH>::kThreads, 1)
    attn_bwd_dq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v,
                const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
  using Cfg = BwdCfg<DH>;
  using Smem = BwdQSmem<DH>;
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
  const uint32_t tbase = sm.tmem_base;
  if (tbase != 0 && threadIdx.x == 0) sm.abort_flag = 1;
  if (tbase == 0) {
    if (warp == Cfg::kWarpProducer) {
      if (lane == 0) bwd_dq_producer<DH>(sm, p, &map_q, &map_k, &map_v, &map_do, abort);
    } else if (warp == Cfg::kWarpIssuer) {
      bwd_dq_issuer<DH>(sm, p, abort);
    } else {
      bwd_dq_softmax<DH>(sm, p, tbase, abort, warp, lane);
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
  // Launched as a programmatic dependent of the dK/dV pass, this grid may run
  // beside that pass's last CTAs (it reads nothing the pass writes: only the
  // inputs and the prep kernel's D and lse2, complete before any dK/dV CTA
  // let this grid be scheduled).  It does not finish before the dK/dV pass
  // has, so that the next kernel in the stream sees dK and dV as well.
  if (threadIdx.x == 0) griddep_wait();
}

template <int DH>
constexpr size_t bwd_dkdv_smem_bytes() { return sizeof(BwdKvSmem<DH>) + 1024; }
template <int DH>
constexpr size_t bwd_dq_smem_bytes() { return sizeof(BwdQSmem<DH>) + 1024; }

}  // namespace chs
