// decode_sm103a.cu -- split planning and host launchers of the decode kernels.
#include "decode_sm103a.cuh"
#include "launch.h"

namespace chs {

DecodePlan plan_decode(int B, int Hq, int Hkv, int Tmax, int Dh, int num_sms) {
  (void)Dh;
  DecodePlan plan;
  const int group = Hq / Hkv;
  plan.heads_per_cta = group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1);
  const long long ctas_per_split = (long long)B * Hkv * (group / plan.heads_per_cta);
  // aim for about 16 CTAs of work per SM over the whole cache, in whole
  // 64-key blocks, between 256 and 4096 keys per split and at most 64 splits
  const long long want = 16LL * num_sms;
  long long per_split_keys = (long long)Tmax * ctas_per_split / (want > 0 ? want : 1);
  long long chunk = (per_split_keys + kDecodeBlockKeys - 1) / kDecodeBlockKeys * kDecodeBlockKeys;
  if (chunk < 256) chunk = 256;
  if (chunk > 4096) chunk = 4096;
  long long nsplit = (Tmax + chunk - 1) / chunk;
  if (nsplit > 64) {
    chunk = ((Tmax + 63) / 64 + kDecodeBlockKeys - 1) / kDecodeBlockKeys * kDecodeBlockKeys;
    nsplit = (Tmax + chunk - 1) / chunk;
  }
  plan.chunk = (int)chunk;
  plan.nsplit = (int)nsplit;
  return plan;
}

size_t decode_workspace_bytes(int B, int Hq, int Dh, const DecodePlan& plan) {
  const size_t rows = (size_t)B * Hq * plan.nsplit;
  const size_t o_bytes = (rows * Dh * sizeof(float) + 255) / 256 * 256;
  const size_t ml_bytes = (rows * sizeof(float) + 255) / 256 * 256;
  return o_bytes + 2 * ml_bytes;
}

template <int DH, int HPB>
static cudaError_t launch_split(const DecodeParams& prm, int groups, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_bytes<DH, HPB>();
  cudaError_t e = cudaFuncSetAttribute(attn_decode_split_sm103a<DH, HPB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(prm.nsplit, prm.Hkv * groups, prm.B);
  attn_decode_split_sm103a<DH, HPB><<<grid, kDecodeThreads, smem, stream>>>(prm);
  return cudaGetLastError();
}

template <int DH>
static cudaError_t launch_dh(const DecodeParams& prm, int hpb, cudaStream_t stream) {
  const int groups = (prm.Hq / prm.Hkv) / hpb;
  cudaError_t e;
  if (hpb == 4)
    e = launch_split<DH, 4>(prm, groups, stream);
  else if (hpb == 2)
    e = launch_split<DH, 2>(prm, groups, stream);
  else
    e = launch_split<DH, 1>(prm, groups, stream);
  if (e != cudaSuccess) return e;
  attn_decode_combine_sm103a<DH><<<prm.B * prm.Hq, DH, 0, stream>>>(prm);
  return cudaGetLastError();
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int* seqlens,
                          void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window,
                          float scale_log2, const DecodePlan& plan, void* workspace,
                          const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.kc = static_cast<const __nv_bfloat16*>(kc);
  prm.vc = static_cast<const __nv_bfloat16*>(vc);
  prm.seqlens = seqlens;
  prm.o = static_cast<__nv_bfloat16*>(o);
  const size_t rows = (size_t)B * Hq * plan.nsplit;
  const size_t o_bytes = (rows * Dh * sizeof(float) + 255) / 256 * 256;
  const size_t ml_bytes = (rows * sizeof(float) + 255) / 256 * 256;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  prm.o_part = reinterpret_cast<float*>(ws);
  prm.m_part = reinterpret_cast<float*>(ws + o_bytes);
  prm.l_part = reinterpret_cast<float*>(ws + o_bytes + ml_bytes);
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Tmax = Tmax;
  prm.window = window;
  prm.nsplit = plan.nsplit;
  prm.chunk = plan.chunk;
  prm.scale_log2 = scale_log2;
  prm.error_word = dev.error_word;
  return Dh == 128 ? launch_dh<128>(prm, plan.heads_per_cta, stream)
                   : launch_dh<64>(prm, plan.heads_per_cta, stream);
}

}  // namespace chs
