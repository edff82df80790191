// decode_sm103a.cuh -- one KV-cache decode step, split along the cache.
//
// The query of sequence b sits at position L_b - 1 (L_b = seqlens[b]); its
// own key/value were appended to the cache first, so it attends to cached
// keys [lo_b, L_b) with lo_b = 0, or L_b - W under a sliding window of W keys
// ("Механизм внимания", llm-arch-research.openidealab.com/textbook/attention,
// sections "KV-кэш", "Prefill и decode" and "Скользящее окно").  The step reads
// the whole cache for little arithmetic, so it is bound by HBM bandwidth.
//
// One kernel, grid (Hkv * groups, nsplit, B).  A CTA takes `chunk` keys of one
// (b, K/V head) and HPB query heads of that head's group.  The library runs
// it with HPB = 1 for one query head per K/V head (MHA); groups of two or
// more heads take the tensor-core decode (decode_tc_sm103a.cuh), which reads
// each cached byte once per group and does the group's per-key softmax work
// on 128-row tiles.  One producer thread
// streams 32-key blocks of K and V into a four-stage shared-memory ring with
// cp.async.bulk; four consumer warps take 8 keys of each block.  In a warp,
// LPK = DH/8 lanes share a key, one 16-byte chunk (8 elements) each; every
// lane holds all HPB query heads' matching chunks and output accumulators as
// packed float2 (fma.rn.f32x2).  A key's HPB dot products are finished with a
// transposing xor-shuffle reduction, and each key slot keeps its own running
// max, running sum and output (the online softmax).  The CTA merges its slots
// and writes an unnormalised partial with its max and sum.
//
// The last CTA to finish a (b, K/V head, group) -- counted with one atomic per
// CTA -- merges the partials of all splits in split order (so the result does
// not depend on which CTA was last):
//   o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
#pragma once

#include "sm103a_ptx.cuh"

namespace chs {

struct DecodeParams {
  const __nv_bfloat16* q;   // [B, Hq, 1, DH]
  const __nv_bfloat16* kc;  // [B, Hkv, Tmax, DH]
  const __nv_bfloat16* vc;  // [B, Hkv, Tmax, DH]
  const int* seqlens;       // [B], device
  __nv_bfloat16* o;         // [B, Hq, 1, DH]
  float* o_part;            // [B, Hq, nsplit, DH]
  float* m_part;            // [B, Hq, nsplit]   (log2 domain)
  float* l_part;            // [B, Hq, nsplit]
  int* counters;            // [B, Hkv * groups], zero between calls
  int B, Hq, Hkv, Tmax, window;
  int nsplit, chunk;
  float scale_log2;
  int* error_word;
  int fault;                // test hook: 2 = the first key block is never loaded
  int ring;                 // 1: the Tmax cache rows are a ring, position t at row t % Tmax
};

constexpr int kDecodeBlockKeys = 32;    // keys per pipeline stage at Dh = 128
// Keys per pipeline stage: 8 KiB of K and 8 KiB of V per stage at either head
// size, so that as many bytes are in flight (at Dh = 64, 32-key stages kept
// too few bytes in flight to cover the HBM latency).
template <int DH>
__host__ __device__ constexpr int decode_block_keys() { return kDecodeBlockKeys * 128 / DH; }
constexpr int kDecodeStages = 4;
constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (kDecodeConsumerWarps + 1);
constexpr int kDecodeCtasPerSm = 3;

template <int DH, int HPB>
struct __align__(128) DecodeSmem {
  __nv_bfloat16 k[kDecodeStages][decode_block_keys<DH>() * DH];
  __nv_bfloat16 v[kDecodeStages][decode_block_keys<DH>() * DH];
  float red_o[kDecodeConsumerWarps][HPB][DH];
  float red_m[kDecodeConsumerWarps][HPB];
  float red_l[kDecodeConsumerWarps][HPB];
  uint64_t full[kDecodeStages], empty[kDecodeStages];
  int abort_flag;
  int is_last;
};

// The visible key positions of a sequence of L tokens are [lo, L); splits
// are `chunk` positions wide, counted from `base`.  A linear cache counts
// them from position 0 (fixed split boundaries); a ring, whose positions
// grow without bound, from lo.
struct DecodeSpan {
  int lo, base;
};

__device__ __forceinline__ DecodeSpan decode_span(const DecodeParams& p, int L) {
  DecodeSpan d;
  if (p.ring) {
    const int w = p.window > 0 ? p.window : p.Tmax;   // <= Tmax, checked on the host
    d.lo = max(0, L - w);
    d.base = d.lo;
  } else {
    d.lo = p.window > 0 ? max(0, L - p.window) : 0;
    d.base = 0;
  }
  return d;
}

// keys [k_begin, k_end) of split `split`
__device__ __forceinline__ void decode_split_range(const DecodeSpan& d, int L, int split, int chunk,
                                                   int& k_begin, int& k_end) {
  // (64-bit: a ring's positions may come close to 2^31)
  k_begin = (int)max((long long)d.base + (long long)split * chunk, (long long)d.lo);
  k_end = (int)min((long long)d.base + (long long)(split + 1) * chunk, (long long)L);
}

// bf16 pair (low half = lower-addressed element) -> float2
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

__device__ __forceinline__ void unpack_chunk(const uint4& w, float2 (&f)[4]) {
  f[0] = bf16x2_to_float2(w.x);
  f[1] = bf16x2_to_float2(w.y);
  f[2] = bf16x2_to_float2(w.z);
  f[3] = bf16x2_to_float2(w.w);
}

// Sum each of s[0..HPB) over the LPK lanes of a key group (aligned groups of
// LPK consecutive lanes), transposing as it goes: in each of the first
// log2(HPB) rounds a lane passes on half of its values and keeps half, so a
// lane ends holding the full sum of ONE head (2 + 1 shuffles for four heads,
// then one per remaining round).  Returns that sum; key_group_owner() names
// a lane of the group that holds head h.
template <int HPB, int LPK>
__device__ __forceinline__ float key_group_reduce_owned(const float (&s)[HPB], int lane) {
  static_assert(HPB == 1 || HPB == 2 || HPB == 4, "heads per CTA");
  static_assert(LPK >= HPB, "a key group must hold every head");
  float k;
  int first_plain;   // first offset of the plain (non-transposing) rounds
  if constexpr (HPB == 4) {
    constexpr int o1 = LPK / 2, o2 = LPK / 4;
    const bool up1 = (lane & o1) != 0, up2 = (lane & o2) != 0;
    float k0 = up1 ? s[2] : s[0], k1 = up1 ? s[3] : s[1];
    const float x0 = up1 ? s[0] : s[2], x1 = up1 ? s[1] : s[3];
    k0 += __shfl_xor_sync(0xffffffffu, x0, o1);
    k1 += __shfl_xor_sync(0xffffffffu, x1, o1);
    k = up2 ? k1 : k0;
    const float x = up2 ? k0 : k1;
    k += __shfl_xor_sync(0xffffffffu, x, o2);
    first_plain = LPK / 8;
  } else if constexpr (HPB == 2) {
    constexpr int o1 = LPK / 2;
    const bool up1 = (lane & o1) != 0;
    k = up1 ? s[1] : s[0];
    const float x = up1 ? s[0] : s[1];
    k += __shfl_xor_sync(0xffffffffu, x, o1);
    first_plain = LPK / 4;
  } else {
    k = s[0];
    first_plain = LPK / 2;
  }
#pragma unroll
  for (int off = LPK / 2; off >= 1; off /= 2)
    if (off <= first_plain) k += __shfl_xor_sync(0xffffffffu, k, off);
  return k;
}

// Head whose sum key_group_reduce_owned leaves in `lane`.
template <int HPB, int LPK>
__device__ __forceinline__ int key_group_owned_head(int lane) {
  if constexpr (HPB == 4)
    return 2 * ((lane & (LPK / 2)) != 0) + ((lane & (LPK / 4)) != 0);
  else if constexpr (HPB == 2)
    return (lane & (LPK / 2)) != 0;
  else
    return 0;
}

// A lane of `lane`'s key group that holds head h after key_group_reduce_owned.
template <int HPB, int LPK>
__device__ __forceinline__ int key_group_owner(int h, int lane) {
  const int base = lane & ~(LPK - 1);
  if constexpr (HPB == 4)
    return base + (h >> 1) * (LPK / 2) + (h & 1) * (LPK / 4);
  else if constexpr (HPB == 2)
    return base + h * (LPK / 2);
  else
    return base;
}

template <int DH, int HPB>
__global__ void __launch_bounds__(kDecodeThreads, kDecodeCtasPerSm)
    attn_decode_sm103a(const DecodeParams p) {
  constexpr int LPK = DH / 8;           // lanes per key (one 16-byte chunk each)
  constexpr int KPS = 32 / LPK;         // keys per warp step
  constexpr int BK = decode_block_keys<DH>();   // keys per block
  constexpr int KPW = BK / kDecodeConsumerWarps;   // keys per warp per block
  constexpr int ROW = DH * 2;           // bytes per cached row
  using Smem = DecodeSmem<DH, HPB>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                      ~uintptr_t(127));
  volatile int* abort = &sm.abort_flag;
  // the lengths and the cache may come from the previous kernel in the
  // stream: wait for it before the first global read (a no-op unless this
  // launch is a programmatic dependent)
  griddep_wait();

  // grid (head groups, splits, B): the CTAs of one split -- the query-head
  // groups that read the same K/V rows when Hq / Hkv exceeds 4 (MQA) -- are
  // launched side by side, so the rows come from L2 after the first read
  const int split = blockIdx.y;
  const int groups = (p.Hq / p.Hkv) / HPB;
  const int g = blockIdx.x / groups;
  const int hsub = blockIdx.x % groups;
  const int b = blockIdx.z;
  const int hq0 = g * (p.Hq / p.Hkv) + hsub * HPB;   // first query head of this CTA
  const int L = p.seqlens[b];
  if (L < 1 || (!p.ring && L > p.Tmax)) {
    // a sequence length outside [1, Tmax]: zero output, latch the error
    if (split == 0) {
      for (int i = threadIdx.x; i < HPB * DH; i += blockDim.x)
        p.o[(size_t)(b * p.Hq + hq0) * DH + i] = __float2bfloat16(0.f);
      if (threadIdx.x == 0) atomicExch(p.error_word, 1);   // ATTN_ERR_INVALID_ARG
    }
    return;
  }
  int k_begin, k_end;
  const DecodeSpan span = decode_span(p, L);
  decode_split_range(span, L, split, p.chunk, k_begin, k_end);
  if (k_begin >= k_end) return;      // this split holds no visible key
  const int nkeys = k_end - k_begin;
  const int nblk = (nkeys + BK - 1) / BK;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    for (int i = 0; i < kDecodeStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kDecodeConsumerWarps);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == kDecodeConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const size_t head0 = ((size_t)b * p.Hkv + g) * p.Tmax;   // row 0 of this head
      const uint8_t* kg = reinterpret_cast<const uint8_t*>(p.kc) + head0 * ROW;
      const uint8_t* vg = reinterpret_cast<const uint8_t*>(p.vc) + head0 * ROW;
      const uint64_t stream_once = policy_evict_first();
      // cache row of the block's first key (a linear cache never wraps)
      int row = p.ring ? k_begin % p.Tmax : k_begin;
      uint32_t st = 0, ph = 0, loaded = 0, par = 0;
      for (int blk = 0; blk < nblk; ++blk) {
        const int n = min(BK, nkeys - blk * BK);
        if (!mbar_wait(&sm.empty[st], ph ^ 1, abort)) break;
        if (p.fault != 2 || blk != 0) {   // (the test hook withholds one block)
          // a block that runs past the end of a ring continues at row 0
          const int n1 = min(n, p.Tmax - row);
          // (checked builds: both copies inside the head's Tmax rows)
          const bool in_range = attn_check(row >= 0 && n >= 1 && n <= BK && n1 >= 1 &&
                                               (p.ring || n1 == n) && n - n1 <= row,
                                           p.error_word);
          mbar_arrive_expect_tx(&sm.full[st], in_range ? 2u * n * ROW : 0u);
          if (in_range) {
            bulk_load(sm.k[st], kg + (size_t)row * ROW, n1 * ROW, &sm.full[st], stream_once);
            bulk_load(sm.v[st], vg + (size_t)row * ROW, n1 * ROW, &sm.full[st], stream_once);
            if (n1 < n) {   // (offsets in bytes: the stage arrays hold bf16 elements)
              bulk_load(reinterpret_cast<uint8_t*>(sm.k[st]) + n1 * ROW, kg, (n - n1) * ROW,
                        &sm.full[st], stream_once);
              bulk_load(reinterpret_cast<uint8_t*>(sm.v[st]) + n1 * ROW, vg, (n - n1) * ROW,
                        &sm.full[st], stream_once);
            }
          }
          loaded |= 1u << st;
          par = (par & ~(1u << st)) | (ph << st);
        }
        row += n;
        if (row >= p.Tmax) row -= p.Tmax;
        if (++st == kDecodeStages) { st = 0; ph ^= 1; }
      }
      // every copy this thread started has landed before the CTA may exit
      for (int i = 0; i < kDecodeStages; ++i) {
        if (!(loaded & (1u << i))) continue;
        const uint32_t a = smem_u32(&sm.full[i]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, (par >> i) & 1u))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int kslot = lane / LPK, part = lane % LPK;
    float2 q2[HPB][4], acc[HPB][4];
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      const uint4 w =
          reinterpret_cast<const uint4*>(p.q + (size_t)(b * p.Hq + hq0 + h) * DH)[part];
      unpack_chunk(w, q2[h]);
      const float2 sc = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q2[h][i] = __fmul2_rn(q2[h][i], sc);
        acc[h][i] = make_float2(0.f, 0.f);
      }
    }
    // Online-softmax state of the one head whose score this lane finishes in
    // the reduction (every lane of a key slot holding that head agrees).  The
    // running max is raised lazily: only when a score exceeds it by more than
    // 8 (weights then stay <= 2^8), which after the first key is rare, so the
    // rescale of the accumulators sits in a warp-uniform branch.
    float m_own = -INFINITY, l_own = 0.f;
    const int lane_off = (warp * KPW + kslot) * ROW + part * 16;   // this lane's chunk

    // One block: this warp's KPW keys, KPS at a time (one per key slot), in
    // three phases so that the NS independent keys of each phase overlap
    // their latencies (loads, shuffle reductions, ex2) instead of running
    // one dependent chain per key: all scores, then one lazy max update for
    // the lot, then the weights and the V accumulation.
    constexpr int NS = KPW / KPS;
    auto do_block = [&](const uint8_t* kp, const uint8_t* vp, int n) {
      float s_own[NS];
      bool val[NS];
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        val[j] = warp * KPW + j * KPS + kslot < n;
        uint4 kw = make_uint4(0, 0, 0, 0);
        if (val[j]) kw = *reinterpret_cast<const uint4*>(kp + j * KPS * ROW);
        float2 k2[4];
        unpack_chunk(kw, k2);
        float sh[HPB];
#pragma unroll
        for (int h = 0; h < HPB; ++h) {
          float2 d = __fmul2_rn(q2[h][0], k2[0]);
#pragma unroll
          for (int i = 1; i < 4; ++i) d = __ffma2_rn(q2[h][i], k2[i], d);
          sh[h] = d.x + d.y;
        }
        s_own[j] = key_group_reduce_owned<HPB, LPK>(sh, lane);
      }
      float smax = -INFINITY;
#pragma unroll
      for (int j = 0; j < NS; ++j)
        if (val[j]) smax = fmaxf(smax, s_own[j]);
      const bool grow = smax > m_own + 8.0f;
      if (__any_sync(0xffffffffu, grow)) {
        const float corr = grow ? ex2_approx(m_own - smax) : 1.0f;   // 0 for the first keys
        if (grow) m_own = smax;
        l_own *= corr;
#pragma unroll
        for (int h = 0; h < HPB; ++h) {
          const float c = __shfl_sync(0xffffffffu, corr, key_group_owner<HPB, LPK>(h, lane));
          const float2 c2 = make_float2(c, c);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[h][i] = __fmul2_rn(acc[h][i], c2);
        }
      }
      float p_own[NS];
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        p_own[j] = val[j] ? ex2_approx(s_own[j] - m_own) : 0.f;
        l_own += p_own[j];
      }
#pragma unroll
      for (int j = 0; j < NS; ++j) {
        uint4 vw = make_uint4(0, 0, 0, 0);
        if (val[j]) vw = *reinterpret_cast<const uint4*>(vp + j * KPS * ROW);
        float2 v2[4];
        unpack_chunk(vw, v2);
#pragma unroll
        for (int h = 0; h < HPB; ++h) {
          const float pw = __shfl_sync(0xffffffffu, p_own[j], key_group_owner<HPB, LPK>(h, lane));
          const float2 p2 = make_float2(pw, pw);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[h][i] = __ffma2_rn(p2, v2[i], acc[h][i]);
        }
      }
    };

    uint32_t st = 0, ph = 0;
    for (int blk = 0; blk < nblk; ++blk) {
      if (!mbar_wait(&sm.full[st], ph, abort)) break;
      const int n = min(BK, nkeys - blk * BK);
      const uint8_t* kp = reinterpret_cast<const uint8_t*>(sm.k[st]) + lane_off;
      const uint8_t* vp = reinterpret_cast<const uint8_t*>(sm.v[st]) + lane_off;
      if (n == BK)
        do_block(kp, vp, BK);   // the common, full block (validity folds away)
      else
        do_block(kp, vp, n);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
      if (++st == kDecodeStages) { st = 0; ph ^= 1; }
    }

    // every lane of a key slot gets all heads' running max and sum
    float m[HPB], l[HPB];
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      m[h] = __shfl_sync(0xffffffffu, m_own, key_group_owner<HPB, LPK>(h, lane));
      l[h] = __shfl_sync(0xffffffffu, l_own, key_group_owner<HPB, LPK>(h, lane));
    }
    // merge the key slots of this warp (lanes with equal `part`)
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      float mw = m[h];
#pragma unroll
      for (int off = LPK; off < 32; off *= 2) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
      const float f = (m[h] == -INFINITY) ? 0.f : ex2_approx(m[h] - mw);
      const float2 f2 = make_float2(f, f);
      float lw = l[h] * f;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = __fmul2_rn(acc[h][i], f2);
#pragma unroll
      for (int off = LPK; off < 32; off *= 2) {
        lw += __shfl_xor_sync(0xffffffffu, lw, off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[h][i].x += __shfl_xor_sync(0xffffffffu, acc[h][i].x, off);
          acc[h][i].y += __shfl_xor_sync(0xffffffffu, acc[h][i].y, off);
        }
      }
      if (lane == 0) {
        sm.red_m[warp][h] = mw;
        sm.red_l[warp][h] = lw;
      }
      if (kslot == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sm.red_o[warp][h][part * 8 + 2 * i] = acc[h][i].x;
          sm.red_o[warp][h][part * 8 + 2 * i + 1] = acc[h][i].y;
        }
      }
    }
    named_bar_sync(1, 32 * kDecodeConsumerWarps);

    const int s_first = (span.lo - span.base) / p.chunk, s_last = (L - 1 - span.base) / p.chunk;
    const bool single = s_first == s_last;   // the whole key range is this CTA's
    // merge the warps: this CTA's result for each (head, d)
    for (int idx = threadIdx.x; idx < HPB * DH; idx += 32 * kDecodeConsumerWarps) {
      const int h = idx / DH, d = idx % DH;
      float M = sm.red_m[0][h];
#pragma unroll
      for (int w = 1; w < kDecodeConsumerWarps; ++w) M = fmaxf(M, sm.red_m[w][h]);
      float o = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeConsumerWarps; ++w) {
        const float mw = sm.red_m[w][h];
        const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
        o = fmaf(f, sm.red_o[w][h][d], o);
        lsum = fmaf(f, sm.red_l[w][h], lsum);
      }
      const size_t bh = (size_t)b * p.Hq + hq0 + h;
      if (single) {
        p.o[bh * DH + d] = __float2bfloat16(o / lsum);
      } else {
        const size_t ps = bh * p.nsplit + split;
        p.o_part[ps * DH + d] = o;
        if (d == 0) {
          p.m_part[ps] = M;
          p.l_part[ps] = lsum;
        }
      }
    }

    if (!single) {
      // the last CTA of this (b, K/V head, group) to get here merges all splits
      __threadfence();
      named_bar_sync(1, 32 * kDecodeConsumerWarps);
      int* counter = p.counters + (size_t)b * gridDim.x + blockIdx.x;
      if (threadIdx.x == 0) {
        const int prev = atomicAdd(counter, 1);
        sm.is_last = prev == s_last - s_first;
      }
      named_bar_sync(1, 32 * kDecodeConsumerWarps);
      if (sm.is_last) {
        __threadfence();
        for (int idx = threadIdx.x; idx < HPB * DH; idx += 32 * kDecodeConsumerWarps) {
          const int h = idx / DH, d = idx % DH;
          const size_t bh = (size_t)b * p.Hq + hq0 + h;
          const float* mp = p.m_part + bh * p.nsplit;
          const float* lp = p.l_part + bh * p.nsplit;
          const float* op = p.o_part + bh * p.nsplit * DH;
          float M = -INFINITY;
          for (int s = s_first; s <= s_last; ++s) M = fmaxf(M, __ldcg(mp + s));
          float o = 0.f, lsum = 0.f;
          for (int s = s_first; s <= s_last; ++s) {
            const float f = ex2_approx(__ldcg(mp + s) - M);
            o = fmaf(f, __ldcg(op + (size_t)s * DH + d), o);
            lsum = fmaf(f, __ldcg(lp + s), lsum);
          }
          p.o[bh * DH + d] = __float2bfloat16(o / lsum);
        }
        if (threadIdx.x == 0) *counter = 0;   // ready for the next call
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
}

template <int DH, int HPB>
constexpr size_t decode_smem_bytes() {
  return sizeof(DecodeSmem<DH, HPB>) + 128;
}

}  // namespace chs
