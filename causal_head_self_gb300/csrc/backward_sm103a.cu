// backward_sm103a.cu -- host launchers of the backward pass: D and lse2 per
// row, then the dK/dV pass and the dQ pass on the same stream (at head size
// 256: a dV pass, a dK pass and the dQ pass).
#include "backward256_sm103a.cuh"
#include "backward_sm103a.cuh"
#include "launch.h"

namespace chs {

template <int DH>
static cudaError_t launch_bwd_dh(const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const CUtensorMap& mdo, const BwdParams& prm,
                                 const void* o, const void* dout, const float* lse, float* lse2,
                                 float* delta, const DeviceInfo& dev, cudaStream_t stream) {
  constexpr size_t smem_kv = bwd_dkdv_smem_bytes<DH>(), smem_q = bwd_dq_smem_bytes<DH>();
  static_assert(smem_kv <= 232448 && smem_q <= 232448, "shared memory budget of one sm_103a CTA");
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, dev.device, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_bwd_dkdv<DH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attn_bwd_dq<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_q);
  });
  if (e != cudaSuccess) return e;
  const long long rows = (long long)prm.B * prm.Hq * prm.S_pad;
  constexpr int rpb = bwd_prep_rows_per_block<DH>();
  // three programmatic dependent launches: each kernel's launch and set-up
  // overlap the previous one's tail (the prep and the dK/dV pass wait for
  // their predecessor before reading; the dQ pass, which needs only the
  // prep's output, runs beside the dK/dV pass's last CTAs)
  e = launch_pdl(attn_bwd_prep<DH>, dim3((unsigned)((rows + rpb - 1) / rpb)), dim3(256), 0, stream,
                 static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
                 lse, lse2, delta, rows, prm.S, prm.S_pad);
  if (e != cudaSuccess) return e;
  // persistent passes: one CTA per SM (their shared memory allows no second)
  BwdParams pk = prm;
  pk.num_items = prm.nblk * prm.B * prm.Hkv;
  const int grid_kv = pk.num_items < dev.num_sms ? pk.num_items : dev.num_sms;
  e = launch_pdl(attn_bwd_dkdv<DH>, dim3(grid_kv), dim3(BwdCfg<DH>::kThreads), smem_kv, stream,
                 mq, mk, mv, mdo, pk);
  if (e != cudaSuccess) return e;
  BwdParams pq = prm;
  pq.num_items = prm.nblk * prm.B * prm.Hq;
  const int grid_q = pq.num_items < dev.num_sms ? pq.num_items : dev.num_sms;
  return launch_pdl(attn_bwd_dq<DH>, dim3(grid_q), dim3(BwdCfg<DH>::kThreads), smem_q, stream, mq,
                    mk, mv, mdo, pq);
}

// Head size 256: prep, then the dV, dK and dQ passes, each a programmatic
// dependent of the one before (the dK and dQ passes read only the inputs and
// the prep's output, so they start beside the previous pass's last CTAs and
// wait for it only before they end).
static cudaError_t launch_bwd256(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, const BwdParams& prm,
                                 float* lse2, float* delta, const DeviceInfo& dev,
                                 cudaStream_t stream) {
  using Cfg = Bwd256Cfg;
  constexpr size_t smem_dv = bwd256_kv_smem_bytes<false>(), smem_dk = bwd256_kv_smem_bytes<true>(),
                   smem_dq = bwd256_dq_smem_bytes();
  static_assert(smem_dv <= 232448 && smem_dk <= 232448 && smem_dq <= 232448,
                "shared memory budget of one sm_103a CTA");
  // the passes stream 64-row blocks past 128-row ones: each tensor needs a
  // map of each box height
  const long long oq = (long long)prm.B * prm.Hq, okv = (long long)prm.B * prm.Hkv;
  CUtensorMap mq64, mdo64, mk128, mv128, mq128, mdo128, mk64, mv64;
  if (!encode_bf16_map(&mq64, q, Cfg::DH, prm.S, oq, 64) ||
      !encode_bf16_map(&mdo64, dout, Cfg::DH, prm.S, oq, 64) ||
      !encode_bf16_map(&mk128, k, Cfg::DH, prm.S, okv, 128) ||
      !encode_bf16_map(&mv128, v, Cfg::DH, prm.S, okv, 128) ||
      !encode_bf16_map(&mq128, q, Cfg::DH, prm.S, oq, 128) ||
      !encode_bf16_map(&mdo128, dout, Cfg::DH, prm.S, oq, 128) ||
      !encode_bf16_map(&mk64, k, Cfg::DH, prm.S, okv, 64) ||
      !encode_bf16_map(&mv64, v, Cfg::DH, prm.S, okv, 64))
    return cudaErrorInvalidValue;
  static std::atomic<int> configured[kMaxDevices];
  cudaError_t e = configure_once(configured, dev.device, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_bwd256_kv<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_dv);
    if (r != cudaSuccess) return r;
    r = cudaFuncSetAttribute(attn_bwd256_kv<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_dk);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attn_bwd256_dq, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_dq);
  });
  if (e != cudaSuccess) return e;
  const long long rows = (long long)prm.B * prm.Hq * prm.S_pad;
  constexpr int rpb = bwd_prep_rows_per_block<256>();
  e = launch_pdl(attn_bwd_prep<256>, dim3((unsigned)((rows + rpb - 1) / rpb)), dim3(256), 0, stream,
                 static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
                 lse, lse2, delta, rows, prm.S, prm.S_pad);
  if (e != cudaSuccess) return e;
  // persistent passes: one CTA per SM
  BwdParams pk = prm;
  pk.num_items = prm.nblk * prm.B * prm.Hkv;
  const int grid_kv = pk.num_items < dev.num_sms ? pk.num_items : dev.num_sms;
  e = launch_pdl(attn_bwd256_kv<false>, dim3(grid_kv), dim3(Cfg::kThreads), smem_dv, stream, mq64,
                 mk128, mv128, mdo64, pk);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_bwd256_kv<true>, dim3(grid_kv), dim3(Cfg::kThreads), smem_dk, stream, mq64,
                 mk128, mv128, mdo64, pk);
  if (e != cudaSuccess) return e;
  BwdParams pq = prm;
  pq.num_items = prm.nblk * prm.B * prm.Hq;
  const int grid_q = pq.num_items < dev.num_sms ? pq.num_items : dev.num_sms;
  return launch_pdl(attn_bwd256_dq, dim3(grid_q), dim3(Cfg::kThreads), smem_dq, stream, mq128,
                    mk64, mv64, mdo128, pq);
}

size_t bwd_workspace_bytes(int B, int Hq, int S) {
  const size_t S_pad = ((size_t)S + 127) / 128 * 128;
  return 2 * (size_t)B * Hq * S_pad * sizeof(float);
}

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       float* workspace, int B, int Hq, int Hkv, int S, int Dh, int causal,
                       int window, float scale, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mdo;
  if (Dh != 256 && (!encode_bf16_map(&mq, q, Dh, S, (long long)B * Hq, 128) ||
      !encode_bf16_map(&mdo, dout, Dh, S, (long long)B * Hq, 128) ||
      !encode_bf16_map(&mk, k, Dh, S, (long long)B * Hkv, 128) ||
      !encode_bf16_map(&mv, v, Dh, S, (long long)B * Hkv, 128)))
    return cudaErrorInvalidValue;
  BwdParams prm{};
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.S = S;
  prm.causal = causal;
  prm.window = window;
  prm.scale = scale;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
  prm.nblk = (S + 127) / 128;
  prm.S_pad = prm.nblk * 128;
  prm.group = Hq / Hkv;
  if ((long long)prm.nblk * B * Hq > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (((long long)B * Hq * prm.S_pad + 15) / 16 > 0x7fffffffLL) return cudaErrorInvalidValue;
  float* lse2 = workspace;
  float* delta = workspace + (size_t)B * Hq * prm.S_pad;
  prm.lse2 = lse2;
  prm.delta = delta;
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.error_word = dev.error_word;
  prm.fault = dev.fault;
  if (Dh == 256) return launch_bwd256(q, k, v, o, dout, lse, prm, lse2, delta, dev, stream);
  return Dh == 128 ? launch_bwd_dh<128>(mq, mk, mv, mdo, prm, o, dout, lse, lse2, delta, dev, stream)
                   : launch_bwd_dh<64>(mq, mk, mv, mdo, prm, o, dout, lse, lse2, delta, dev, stream);
}

}  // namespace chs
