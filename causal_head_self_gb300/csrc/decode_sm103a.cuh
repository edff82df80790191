// decode_sm103a.cuh -- one KV-cache decode step, split along the cache.
//
// The query of sequence b sits at position L_b - 1 (L_b = seqlens[b]); its
// own key/value were appended to the cache first, so it attends to cached
// keys [lo_b, L_b) with lo_b = 0, or L_b - W under a sliding window of W keys
// ("Механизм внимания", llm-arch-research.openidealab.com/textbook/attention,
// sections "KV-кэш", "Prefill и decode" and "Скользящее окно").  The step reads
// the whole cache for little arithmetic, so it is bound by HBM bandwidth.
//
// Split kernel: grid (nsplit, Hkv * groups, B).  A CTA takes `chunk` keys of
// one (b, K/V head) and every query head of its GQA group that it holds
// (heads_per_cta of them), so each cached K/V byte is read once per group.
// One producer thread streams 64-key blocks of K and V into a shared-memory
// ring with cp.async.bulk; four consumer warps take 16 keys each per block.
// Within a warp, LPK = DH/16 lanes share one key (16 elements of DH each),
// dot products are finished with xor shuffles, and each key slot keeps its
// own running max / running sum / output (the online softmax).  The CTA then
// merges its 16 slot states and writes an unnormalised partial output with
// its max and sum.
//
// Combine kernel: grid B * Hq.  Merges the partials of a query head:
// o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s with M = max_s m_s.
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
  int B, Hq, Hkv, Tmax, window;
  int nsplit, chunk;
  float scale_log2;
  int* error_word;
};

constexpr int kDecodeBlockKeys = 64;    // keys per pipeline stage
constexpr int kDecodeStages = 3;
constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (kDecodeConsumerWarps + 1);

template <int DH, int HPB>
struct __align__(128) DecodeSmem {
  __nv_bfloat16 k[kDecodeStages][kDecodeBlockKeys * DH];
  __nv_bfloat16 v[kDecodeStages][kDecodeBlockKeys * DH];
  float red_o[kDecodeConsumerWarps][HPB][DH];
  float red_m[kDecodeConsumerWarps][HPB];
  float red_l[kDecodeConsumerWarps][HPB];
  uint64_t full[kDecodeStages], empty[kDecodeStages];
  int abort_flag;
};

// keys [k_begin, k_end) of split `split`, for a sequence of L keys
__device__ __forceinline__ void decode_split_range(int L, int window, int split, int chunk,
                                                   int& k_begin, int& k_end) {
  const int lo = window > 0 ? max(0, L - window) : 0;
  k_begin = max(split * chunk, lo);
  k_end = min((split + 1) * chunk, L);
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float (&f)[16]) {
  f[0] = bf16lo(a.x); f[1] = bf16hi(a.x); f[2] = bf16lo(a.y); f[3] = bf16hi(a.y);
  f[4] = bf16lo(a.z); f[5] = bf16hi(a.z); f[6] = bf16lo(a.w); f[7] = bf16hi(a.w);
  f[8] = bf16lo(b.x); f[9] = bf16hi(b.x); f[10] = bf16lo(b.y); f[11] = bf16hi(b.y);
  f[12] = bf16lo(b.z); f[13] = bf16hi(b.z); f[14] = bf16lo(b.w); f[15] = bf16hi(b.w);
}

template <int DH, int HPB>
__global__ void __launch_bounds__(kDecodeThreads)
    attn_decode_split_sm103a(const DecodeParams p) {
  constexpr int LPK = DH / 16;          // lanes per key
  constexpr int KPS = 32 / LPK;         // keys per warp step
  constexpr int KPW = kDecodeBlockKeys / kDecodeConsumerWarps;   // keys per warp per block
  constexpr int ROW = DH * 2;           // bytes per cached row
  using Smem = DecodeSmem<DH, HPB>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                      ~uintptr_t(127));
  volatile int* abort = &sm.abort_flag;

  const int split = blockIdx.x;
  const int groups = (p.Hq / p.Hkv) / HPB;
  const int g = blockIdx.y / groups;
  const int hsub = blockIdx.y % groups;
  const int b = blockIdx.z;
  const int L = p.seqlens[b];
  if (L < 1 || L > p.Tmax) return;   // rejected by the combine kernel
  int k_begin, k_end;
  decode_split_range(L, p.window, split, p.chunk, k_begin, k_end);
  if (k_begin >= k_end) return;      // this split holds no visible key
  const int nkeys = k_end - k_begin;
  const int nblk = (nkeys + kDecodeBlockKeys - 1) / kDecodeBlockKeys;
  const int hq0 = g * (p.Hq / p.Hkv) + hsub * HPB;   // first query head of this CTA

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
      const size_t row0 = ((size_t)b * p.Hkv + g) * p.Tmax + k_begin;
      const uint8_t* kg = reinterpret_cast<const uint8_t*>(p.kc) + row0 * ROW;
      const uint8_t* vg = reinterpret_cast<const uint8_t*>(p.vc) + row0 * ROW;
      const uint64_t stream_once = policy_evict_first();
      uint32_t st = 0, ph = 0, loaded = 0, par = 0;
      for (int blk = 0; blk < nblk; ++blk) {
        const int n = min(kDecodeBlockKeys, nkeys - blk * kDecodeBlockKeys);
        if (!mbar_wait(&sm.empty[st], ph ^ 1, abort)) break;
        mbar_arrive_expect_tx(&sm.full[st], 2u * n * ROW);
        const size_t off = (size_t)blk * kDecodeBlockKeys * ROW;
        bulk_load(sm.k[st], kg + off, n * ROW, &sm.full[st], stream_once);
        bulk_load(sm.v[st], vg + off, n * ROW, &sm.full[st], stream_once);
        loaded |= 1u << st;
        par = (par & ~(1u << st)) | (ph << st);
        if (++st == kDecodeStages) { st = 0; ph ^= 1; }
      }
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
    const int flip = (lane >> 2) & 1;   // spreads a quarter-warp over all banks
    const int c1 = 2 * part + flip, c2 = 2 * part + 1 - flip;   // 16-byte chunks of a row

    float qr[HPB][16];
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (size_t)(b * p.Hq + hq0 + h) * DH);
      float f[16];
      unpack16(qrow[c1], qrow[c2], f);
#pragma unroll
      for (int e = 0; e < 16; ++e) qr[h][e] = f[e] * p.scale_log2;
    }
    float acc[HPB][16], m[HPB], l[HPB];
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[h][e] = 0.f;
    }

    uint32_t st = 0, ph = 0;
    for (int blk = 0; blk < nblk; ++blk) {
      if (!mbar_wait(&sm.full[st], ph, abort)) break;
      const int n = min(kDecodeBlockKeys, nkeys - blk * kDecodeBlockKeys);
      const uint8_t* kb = reinterpret_cast<const uint8_t*>(sm.k[st]);
      const uint8_t* vb = reinterpret_cast<const uint8_t*>(sm.v[st]);
#pragma unroll
      for (int step = 0; step < KPW / KPS; ++step) {
        const int key = warp * KPW + step * KPS + kslot;
        const bool valid = key < n;
        uint4 ka = make_uint4(0, 0, 0, 0), kb2 = ka, va = ka, vb2 = ka;
        if (valid) {
          ka = *reinterpret_cast<const uint4*>(kb + key * ROW + c1 * 16);
          kb2 = *reinterpret_cast<const uint4*>(kb + key * ROW + c2 * 16);
          va = *reinterpret_cast<const uint4*>(vb + key * ROW + c1 * 16);
          vb2 = *reinterpret_cast<const uint4*>(vb + key * ROW + c2 * 16);
        }
        float kf[16];
        unpack16(ka, kb2, kf);
        float s[HPB];
#pragma unroll
        for (int h = 0; h < HPB; ++h) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) d = fmaf(qr[h][e], kf[e], d);
          s[h] = d;
        }
#pragma unroll
        for (int off = LPK / 2; off >= 1; off /= 2)
#pragma unroll
          for (int h = 0; h < HPB; ++h) s[h] += __shfl_xor_sync(0xffffffffu, s[h], off);
        if (valid) {
          float vf[16];
          unpack16(va, vb2, vf);
#pragma unroll
          for (int h = 0; h < HPB; ++h) {
            if (s[h] > m[h]) {   // the running max grows: rescale this slot's state
              const float corr = ex2_approx(m[h] - s[h]);
              l[h] *= corr;
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[h][e] *= corr;
              m[h] = s[h];
            }
            const float pw = ex2_approx(s[h] - m[h]);
            l[h] += pw;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[h][e] = fmaf(pw, vf[e], acc[h][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[st]);
      if (++st == kDecodeStages) { st = 0; ph ^= 1; }
    }

    // bring every slot to the chunk order of key slot 0 (lane == part), whose
    // lanes write the merged result below
    const int flip0 = (part >> 2) & 1;
    if (flip != flip0) {
#pragma unroll
      for (int h = 0; h < HPB; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = acc[h][e];
          acc[h][e] = acc[h][8 + e];
          acc[h][8 + e] = t;
        }
    }
    // merge the key slots of this warp (lanes with equal `part`)
#pragma unroll
    for (int h = 0; h < HPB; ++h) {
      float mw = m[h];
#pragma unroll
      for (int off = LPK; off < 32; off *= 2) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
      const float f = (m[h] == -INFINITY) ? 0.f : ex2_approx(m[h] - mw);
      float lw = l[h] * f;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[h][e] *= f;
#pragma unroll
      for (int off = LPK; off < 32; off *= 2) {
        lw += __shfl_xor_sync(0xffffffffu, lw, off);
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], off);
      }
      if (lane == 0) {
        sm.red_m[warp][h] = mw;
        sm.red_l[warp][h] = lw;
      }
      if (kslot == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sm.red_o[warp][h][8 * c1 + e] = acc[h][e];
          sm.red_o[warp][h][8 * c2 + e] = acc[h][8 + e];
        }
      }
    }
    named_bar_sync(1, 32 * kDecodeConsumerWarps);
    // merge the warps and write this split's partial
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
      const size_t ph_idx = ((size_t)b * p.Hq + hq0 + h) * p.nsplit + split;
      p.o_part[ph_idx * DH + d] = o;
      if (d == 0) {
        p.m_part[ph_idx] = M;
        p.l_part[ph_idx] = lsum;
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0 && sm.abort_flag) atomicExch(p.error_word, 4);   // ATTN_ERR_TIMEOUT
}

template <int DH>
__global__ void __launch_bounds__(DH) attn_decode_combine_sm103a(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int d = threadIdx.x;
  const int L = p.seqlens[b];
  __nv_bfloat16* out = p.o + (size_t)bh * DH;
  if (L < 1 || L > p.Tmax) {   // a sequence length outside [1, Tmax]: zeros + error
    out[d] = __float2bfloat16(0.f);
    if (d == 0) atomicExch(p.error_word, 1);   // ATTN_ERR_INVALID_ARG
    return;
  }
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int s0 = lo / p.chunk, s1 = (L - 1) / p.chunk;
  const float* mp = p.m_part + (size_t)bh * p.nsplit;
  const float* lp = p.l_part + (size_t)bh * p.nsplit;
  const float* op = p.o_part + (size_t)bh * p.nsplit * DH;
  float M = -INFINITY;
  for (int s = s0; s <= s1; ++s) M = fmaxf(M, mp[s]);
  float o = 0.f, lsum = 0.f;
  for (int s = s0; s <= s1; ++s) {
    const float f = ex2_approx(mp[s] - M);
    o = fmaf(f, op[(size_t)s * DH + d], o);
    lsum = fmaf(f, lp[s], lsum);
  }
  out[d] = __float2bfloat16(o / lsum);
}

template <int DH, int HPB>
constexpr size_t decode_smem_bytes() {
  return sizeof(DecodeSmem<DH, HPB>) + 128;
}

}  // namespace chs
