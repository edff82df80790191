// decode_sm103a.cu -- split planning and host launchers of the decode kernels.
#include "decode_sm103a.cuh"
#include "decode_tc_sm103a.cuh"
#include "launch.h"

namespace chs {

DecodePlan plan_decode(int B, int Hq, int Hkv, int Tmax, int Dh, int num_sms) {
  DecodePlan plan;
  const long long bk = Dh == 64    ? decode_block_keys<64>()
                       : Dh == 256 ? decode_block_keys<256>()
                                   : decode_block_keys<128>();
  const int group = Hq / Hkv;
  // groups of two or more query heads take the tensor-core path, so this
  // kernel runs one query head per K/V head: one head per CTA
  plan.heads_per_cta = 1;
  const long long ctas_per_split = (long long)B * Hkv * (group / plan.heads_per_cta);
  // aim for about eight waves of resident CTAs over the whole cache, in
  // whole blocks, between 2048 and 4096 keys per split (a CTA's start-up and
  // merge cost more than the imbalance of fewer, longer splits: with the
  // floor at 2048 keys a B=4 32k-key step and a B=16 8k-key step ran 25 %
  // faster than with 256), <= 64 splits
  const long long want = 8LL * kDecodeCtasPerSm * num_sms;
  long long per_split_keys = (long long)Tmax * ctas_per_split / (want > 0 ? want : 1);
  long long chunk = (per_split_keys + bk - 1) / bk * bk;
  if (chunk < 2048) chunk = 2048;
  if (chunk > 4096) chunk = 4096;
  long long nsplit = (Tmax + chunk - 1) / chunk;
  if (nsplit > 64) {
    chunk = ((Tmax + 63) / 64 + bk - 1) / bk * bk;
    nsplit = (Tmax + chunk - 1) / chunk;
  }
  plan.chunk = (int)chunk;
  plan.nsplit = (int)nsplit;
  return plan;
}

// partial buffers: o_part | m_part | l_part, each 256-byte aligned
struct DecodePartialsLayout {
  size_t o_off, m_off, l_off, total;
};

static DecodePartialsLayout partials_layout(int B, int Hq, int Dh, const DecodePlan& plan) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)B * Hq * plan.nsplit;
  DecodePartialsLayout w;
  w.o_off = 0;
  w.m_off = up(rows * Dh * sizeof(float));
  w.l_off = w.m_off + up(rows * sizeof(float));
  w.total = w.l_off + up(rows * sizeof(float));
  return w;
}

size_t decode_partials_bytes(int B, int Hq, int Dh, const DecodePlan& plan) {
  return partials_layout(B, Hq, Dh, plan).total;
}

size_t decode_counter_count(int B, int Hq, int Hkv, const DecodePlan& plan) {
  return (size_t)B * Hkv * ((Hq / Hkv) / plan.heads_per_cta);
}

template <int DH, int HPB>
static cudaError_t launch_dh(const DecodeParams& prm, int device, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_bytes<DH, HPB>();
  auto kernel = attn_decode_sm103a<DH, HPB>;
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, device, [kernel] {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (r != cudaSuccess) return r;
    // as much shared memory as the SM has, so that several CTAs fit
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
  });
  if (e != cudaSuccess) return e;
  const int groups = (prm.Hq / prm.Hkv) / HPB;
  dim3 grid(prm.Hkv * groups, prm.nsplit, prm.B);
  // a programmatic dependent launch: its launch overlaps the previous
  // kernel's tail (each CTA waits for that kernel before reading memory)
  return launch_pdl(kernel, grid, dim3(kDecodeThreads), smem, stream, prm);
}

// one query head per CTA (plan_decode); the kernel's HPB > 1 forms, which
// share a CTA's cached rows among several heads of a group, are not launched
// since groups of two or more heads run on the tensor cores
template <int DH>
static cudaError_t launch_hpb(const DecodeParams& prm, int hpb, int device, cudaStream_t stream) {
  if (hpb != 1) return cudaErrorInvalidConfiguration;
  return launch_dh<DH, 1>(prm, device, stream);
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int* seqlens,
                          void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window,
                          int ring, float scale_log2, const DecodePlan& plan, int* counters,
                          void* partials, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.kc = static_cast<const __nv_bfloat16*>(kc);
  prm.vc = static_cast<const __nv_bfloat16*>(vc);
  prm.seqlens = seqlens;
  prm.o = static_cast<__nv_bfloat16*>(o);
  const DecodePartialsLayout w = partials_layout(B, Hq, Dh, plan);
  uint8_t* ws = static_cast<uint8_t*>(partials);
  prm.o_part = reinterpret_cast<float*>(ws + w.o_off);
  prm.m_part = reinterpret_cast<float*>(ws + w.m_off);
  prm.l_part = reinterpret_cast<float*>(ws + w.l_off);
  prm.counters = counters;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Tmax = Tmax;
  prm.window = window;
  prm.ring = ring;
  prm.nsplit = plan.nsplit;
  prm.chunk = plan.chunk;
  prm.scale_log2 = scale_log2;
  prm.error_word = dev.error_word;
  prm.fault = dev.fault;
  if (Dh == 256) return launch_hpb<256>(prm, plan.heads_per_cta, dev.device, stream);
  return Dh == 128 ? launch_hpb<128>(prm, plan.heads_per_cta, dev.device, stream)
                   : launch_hpb<64>(prm, plan.heads_per_cta, dev.device, stream);
}

// ---------------------------------------------------------------- tensor-core path

DecodePlan plan_decode_tc(int B, int Hq, int Hkv, int Tmax, int num_sms) {
  DecodePlan plan;
  const int group = Hq / Hkv;
  plan.heads_per_cta = group < 128 ? group : 128;
  const long long units = (long long)B * Hkv * ((group + 127) / 128);
  // about one wave of one CTA per SM (measured: a CTA's start-up costs more
  // than the imbalance of longer splits), whole 128-key tiles, 256..32768
  // keys per split, at most 64 splits
  const long long want = 1LL * num_sms;
  long long chunk = ((long long)Tmax * units / (want > 0 ? want : 1) + 127) / 128 * 128;
  if (chunk < 256) chunk = 256;
  if (chunk > 32768) chunk = 32768;
  long long nsplit = (Tmax + chunk - 1) / chunk;
  if (nsplit > 64) {
    chunk = ((Tmax + 63) / 64 + 127) / 128 * 128;
    nsplit = (Tmax + chunk - 1) / chunk;
  }
  plan.chunk = (int)chunk;
  plan.nsplit = (int)nsplit;
  return plan;
}

template <int DH>
static cudaError_t launch_tc_dh(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const DecodeTcParams& prm, int device, cudaStream_t stream) {
  constexpr size_t smem = decode_tc_smem_bytes<DH>();
  static_assert(smem <= 232448, "shared memory budget of one sm_103a CTA");
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, device, [] {
    return cudaFuncSetAttribute(attn_decode_tc_sm103a<DH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(prm.nsplit, prm.B * prm.Hkv * prm.row_blocks);
  e = launch_pdl(attn_decode_tc_sm103a<DH>, grid, dim3(DecodeTcCfg<DH>::kThreads), smem, stream,
                 mq, mk, mv, prm);
  if (e != cudaSuccess) return e;
  // the combine kernel is a programmatic dependent launch: it is scheduled as
  // the decode CTAs finish and waits on the grid dependency, so its launch
  // latency overlaps the decode kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(prm.B * prm.Hq);
  cfg.blockDim = dim3(DH);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_tc_combine<DH>, prm);
}

cudaError_t launch_decode_tc(const void* q, const void* kc, const void* vc, const int* seqlens,
                             void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window,
                             int ring, float scale_log2, const DecodePlan& plan, void* partials,
                             const DeviceInfo& dev, cudaStream_t stream) {
  const int G = Hq / Hkv;
  CUtensorMap mq, mk, mv;
  const int keys = Dh == 256 ? DecodeTcCfg<256>::kKeys : DecodeTcCfg<128>::kKeys;   // tile rows
  if (!encode_bf16_map(&mq, q, Dh, G, (long long)B * Hkv, 128) ||
      !encode_bf16_map(&mk, kc, Dh, Tmax, (long long)B * Hkv, keys) ||
      !encode_bf16_map(&mv, vc, Dh, Tmax, (long long)B * Hkv, keys))
    return cudaErrorInvalidValue;
  DecodeTcParams prm;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = G;
  prm.Tmax = Tmax;
  prm.window = window;
  prm.ring = ring;
  prm.nsplit = plan.nsplit;
  prm.chunk = plan.chunk;
  prm.row_blocks = (G + 127) / 128;
  prm.scale_log2 = scale_log2;
  prm.seqlens = seqlens;
  const DecodePartialsLayout w = partials_layout(B, Hq, Dh, plan);
  uint8_t* ws = static_cast<uint8_t*>(partials);
  prm.o_part = reinterpret_cast<float*>(ws + w.o_off);
  prm.m_part = reinterpret_cast<float*>(ws + w.m_off);
  prm.l_part = reinterpret_cast<float*>(ws + w.l_off);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.error_word = dev.error_word;
  prm.fault = dev.fault;
  return Dh == 256   ? launch_tc_dh<256>(mq, mk, mv, prm, dev.device, stream)
         : Dh == 128 ? launch_tc_dh<128>(mq, mk, mv, prm, dev.device, stream)
                     : launch_tc_dh<64>(mq, mk, mv, prm, dev.device, stream);
}

}  // namespace chs
