// prefill_sm103a.cu -- host launcher of the tcgen05 prefill kernel.
#include "launch.h"
#include "prefill_sm103a.cuh"

namespace chs {

template <int DH>
static cudaError_t launch_prefill_dh(const CUtensorMap& mq, const CUtensorMap& mk,
                                     const CUtensorMap& mv, const CUtensorMap& mo,
                                     const PrefillParams& prm, cudaStream_t stream) {
  constexpr size_t smem = prefill_smem_bytes<DH>();
  static_assert(smem <= 232448, "shared memory budget of one sm_103a CTA");
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_sm103a<DH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)prm.num_qblocks * prm.B * prm.Hq;
  attn_prefill_sm103a<DH><<<(unsigned)grid, PrefillCfg<DH>::kThreads, smem, stream>>>(mq, mk, mv,
                                                                                     mo, prm);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                           int Hkv, int S, int Dh, int causal, int window, float scale_log2,
                           const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  if (!encode_bf16_map(&mq, q, Dh, S, (long long)B * Hq, 128) ||
      !encode_bf16_map(&mk, k, Dh, S, (long long)B * Hkv, 128) ||
      !encode_bf16_map(&mv, v, Dh, S, (long long)B * Hkv, 128) ||
      !encode_bf16_map(&mo, o, Dh, S, (long long)B * Hq, 32))
    return cudaErrorInvalidValue;
  PrefillParams prm;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.S = S;
  prm.causal = causal;
  prm.window = window;
  prm.scale_log2 = scale_log2;
  prm.num_qblocks = (S + 255) / 256;
  prm.error_word = dev.error_word;
  return Dh == 128 ? launch_prefill_dh<128>(mq, mk, mv, mo, prm, stream)
                   : launch_prefill_dh<64>(mq, mk, mv, mo, prm, stream);
}

}  // namespace chs
