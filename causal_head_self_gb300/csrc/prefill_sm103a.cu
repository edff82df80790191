// prefill_sm103a.cu -- host launchers of the tcgen05 prefill kernels.
#include "launch.h"
#include "prefill_k64_sm103a.cuh"
#include "prefill_sm103a.cuh"

namespace chs {

template <int DH>
static cudaError_t launch_prefill_dh(const CUtensorMap& mq, const CUtensorMap& mk,
                                     const CUtensorMap& mv, const CUtensorMap& mo,
                                     const PrefillParams& prm,
                                     int num_sms, int device, cudaStream_t stream) {
  constexpr size_t smem = prefill_smem_bytes<DH>();
  static_assert(smem <= 232448, "shared memory budget of one sm_103a CTA");
  // The warpgroups' register rebalance assumes the kernel was compiled to the
  // full kRegsLaunch registers per thread; with fewer, the increase could
  // wait forever, so the launch is refused.  Checked once per device, with
  // the shared-memory attribute: a device is marked configured only when
  // both succeed.
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, device, [] {
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, attn_prefill_sm103a<DH>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs < PrefillCfg<DH>::kRegsLaunch) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(attn_prefill_sm103a<DH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (the shared memory allows no second), each
  // walking its share of the work items
  const int grid = prm.num_items < num_sms ? prm.num_items : num_sms;
  // a programmatic dependent launch: set-up overlaps the previous kernel's tail
  return launch_pdl(attn_prefill_sm103a<DH>, dim3(grid), dim3(PrefillCfg<DH>::kThreads), smem,
                    stream, mq, mk, mv, mo, prm);
}

// Multiplier and shift for FastDiv (exact for dividends below 2^31).
static FastDiv make_fast_div(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const unsigned __int128 one = 1;
  const uint64_t m = (uint64_t)(((one << (31 + l)) + d - 1) / d);
  return FastDiv{(uint32_t)m, 31 + l, d};
}

// One 128-row sub-tile per work item, 64-key tiles: head size 256, and head
// size 128 on short sequences (two CTAs per SM).
template <int DH>
static cudaError_t launch_prefill_k64(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int Hq, int Hkv, int Sq, int Tkv,
                                      int start_pos, int causal, int window, float scale_log2,
                                      const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = PrefillK64Cfg<DH>;
  const int Skv = start_pos + Sq;
  CUtensorMap mq, mk, mv, mo;
  if (!encode_bf16_map(&mq, q, Cfg::DH, Sq, (long long)B * Hq, 128) ||
      !encode_bf16_map(&mk, k, Cfg::DH, Skv, (long long)B * Hkv, Cfg::kKeys, Tkv) ||
      !encode_bf16_map(&mv, v, Cfg::DH, Skv, (long long)B * Hkv, Cfg::kKeys, Tkv))
    return cudaErrorInvalidValue;
  // the output map (32 rows x 64 columns per box) where the kernel stores
  // through it; otherwise an unused copy of the Q map
  mo = mq;
  if (Cfg::kTmaStore && !encode_bf16_map(&mo, o, Cfg::DH, Sq, (long long)B * Hq, 32))
    return cudaErrorInvalidValue;
  PrefillK64Params prm;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.q_off = start_pos;
  prm.causal = causal;
  prm.window = window;
  prm.scale_log2 = scale_log2;
  prm.num_qblocks = (Sq + 127) / 128;
  prm.per_qb = B * Hq;
  prm.group = Hq / Hkv;
  const long long items = (long long)prm.num_qblocks * B * Hq;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  prm.num_items = (int)items;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.o_wide = (reinterpret_cast<uintptr_t>(o) & 31) == 0;
  prm.lse = lse;
  prm.error_word = dev.error_word;
  prm.fault = dev.fault;
  constexpr size_t smem = prefill_k64_smem_bytes<DH>();
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, dev.device, [] {
    return cudaFuncSetAttribute(attn_prefill_k64_sm103a<DH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  // persistent: as many CTAs as the SMs hold at once
  const int cap = Cfg::kCtasPerSm * dev.num_sms;
  const int grid = prm.num_items < cap ? prm.num_items : cap;
  return launch_pdl(attn_prefill_k64_sm103a<DH>, dim3(grid), dim3(Cfg::kThreads), smem, stream,
                    mq, mk, mv, mo, prm);
}

// Head size 128 takes the two-CTA 64-key kernel up to this many keys per
// head (measured on GB300: 7 % faster at 1024 keys, even at 2048, 12-15 %
// slower from 4096 on, where the ping-pong kernel's 128-key MMAs win).
constexpr int kPrefillK64MaxKeys128 = 1536;

cudaError_t launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Sq, int Tkv, int start_pos, int Dh,
                           int causal, int window, float scale_log2, const DeviceInfo& dev,
                           cudaStream_t stream) {
  if (Dh == 256)
    return launch_prefill_k64<256>(q, k, v, o, lse, B, Hq, Hkv, Sq, Tkv, start_pos, causal,
                                   window, scale_log2, dev, stream);
  if (Dh == 128 && start_pos + Sq <= kPrefillK64MaxKeys128)
    return launch_prefill_k64<128>(q, k, v, o, lse, B, Hq, Hkv, Sq, Tkv, start_pos, causal,
                                   window, scale_log2, dev, stream);
  // K and V hold Tkv rows per head in memory; the chunk sees the first
  // start_pos + Sq of them, and the maps cover only those (the last key
  // tile's rows past them are zero-filled, never read from the cache)
  const int Skv = start_pos + Sq;
  // the output is written 32 rows (one softmax warp) x 64 columns per box
  CUtensorMap mq, mk, mv, mo;
  if (!encode_bf16_map(&mq, q, Dh, Sq, (long long)B * Hq, 128) ||
      !encode_bf16_map(&mk, k, Dh, Skv, (long long)B * Hkv, 128, Tkv) ||
      !encode_bf16_map(&mv, v, Dh, Skv, (long long)B * Hkv, 128, Tkv) ||
      !encode_bf16_map(&mo, o, Dh, Sq, (long long)B * Hq, 32))
    return cudaErrorInvalidValue;
  PrefillParams prm;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Sq = Sq;
  prm.Skv = Skv;
  prm.q_off = start_pos;
  prm.causal = causal;
  prm.window = window;
  prm.scale_log2 = scale_log2;
  prm.num_qblocks = (Sq + 255) / 256;
  const long long items = (long long)prm.num_qblocks * B * Hq;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  prm.num_items = (int)items;
  prm.lse = lse;
  prm.error_word = dev.error_word;
  prm.fault = dev.fault;
  prm.div_bh = make_fast_div((uint32_t)(B * Hq));
  prm.div_hq = make_fast_div((uint32_t)Hq);
  prm.div_group = make_fast_div((uint32_t)(Hq / Hkv));
  return Dh == 128 ? launch_prefill_dh<128>(mq, mk, mv, mo, prm, dev.num_sms, dev.device, stream)
                   : launch_prefill_dh<64>(mq, mk, mv, mo, prm, dev.num_sms, dev.device, stream);
}

}  // namespace chs
