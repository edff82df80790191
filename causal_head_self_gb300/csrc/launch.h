// launch.h -- internal interface between the C-ABI layer and the kernel
// translation units.  Not part of the public ABI (see include/attn.h).
#pragma once

#include <atomic>
#include <utility>

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace chs {

// Kernel attributes (shared-memory size, carveout) are set once per device:
// `flags` is a per-kernel array of kMaxDevices entries.
constexpr int kMaxDevices = 64;
template <typename F>
inline cudaError_t configure_once(std::atomic<int>* flags, int device, F&& set) {
  const bool tracked = device >= 0 && device < kMaxDevices;
  if (tracked && flags[device].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = set();
  if (e == cudaSuccess && tracked) flags[device].store(1, std::memory_order_release);
  return e;
}

// Launch `kernel` on `stream` as a programmatic dependent of the kernel
// before it: its CTAs may be scheduled while that kernel finishes, and each
// waits (griddep_wait) for it to complete before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DeviceInfo {
  int device;
  int num_sms;
  int* error_word;   // device address of this device's latched error word
  int fault;         // test hook passed to the kernels (attn_debug_inject_fault)
};

// Encode a 3-D tensor map over a [outer, stride_rows, Dh] bf16 tensor of
// which the first `rows` rows per outer index are visible: dims {Dh, rows,
// outer}, 128-byte swizzle, box {64, box_rows, 1}.  Rows at or past `rows`
// are never read; a box reaching past them is zero-filled
// (stride_rows = 0 means stride_rows = rows).
bool encode_bf16_map(CUtensorMap* map, const void* base, int Dh, int rows, long long outer,
                     int box_rows, int stride_rows = 0);

// Queries: Sq rows per (b, h), at positions start_pos .. start_pos + Sq - 1.
// K, V: Tkv rows per (b, K/V head) in memory, of which the first
// start_pos + Sq are visible (a plain prefill: Tkv = Sq, start_pos = 0).
// lse (optional, [B, Hq, Sq] fp32) receives each row's log-sum-exp.
cudaError_t launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int Hq, int Hkv, int Sq, int Tkv, int start_pos, int Dh,
                           int causal, int window, float scale_log2, const DeviceInfo& dev,
                           cudaStream_t stream);

struct DecodePlan {
  int chunk;          // keys per split
  int nsplit;         // splits per (b, query head)
  int heads_per_cta;  // query heads of a GQA group handled by one CTA
};

DecodePlan plan_decode(int B, int Hq, int Hkv, int Tmax, int Dh, int num_sms);

// Bytes of split partials (o, max, sum) a decode call with this plan needs.
size_t decode_partials_bytes(int B, int Hq, int Dh, const DecodePlan& plan);

// Completion counters (one int per CTA group) a decode call needs.  They
// must be zero before the call, and every call leaves them zero again, so a
// buffer that only ever holds counters stays valid across calls and shapes.
size_t decode_counter_count(int B, int Hq, int Hkv, const DecodePlan& plan);

// ring = 1: the Tmax cache rows of a head hold position t at row t % Tmax
// (the last Tmax positions of an unbounded sequence).
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int* seqlens,
                          void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window,
                          int ring, float scale_log2, const DecodePlan& plan, int* counters,
                          void* partials, const DeviceInfo& dev, cudaStream_t stream);

// Tensor-core decode for query-head groups (Hq / Hkv >= kDecodeTcMinGroup):
// splits of whole 128-key tiles, one CTA per (split, b, K/V head, 128 heads),
// then a combine kernel.  Linear caches, and rings (ring = 1: position t at
// row t % Tmax, window <= Tmax, window <= 0 meaning Tmax).  Measured against
// the CUDA-core kernel on the same inputs (back-to-back launches): groups of
// 4 run at 6.8 TB/s instead of 6.3 (Dh 128), 5.6 instead of 3.8 (Dh 64) and
// 6.0 instead of 5.7 (Dh 256), groups of 2 at 6.7 instead of 6.6; with one
// query head per K/V head the CUDA-core kernel is as fast (Dh 128) or faster
// (Dh 64: 6.3 against 5.1 TB/s), so it keeps that case.
constexpr int kDecodeTcMinGroup = 2;
DecodePlan plan_decode_tc(int B, int Hq, int Hkv, int Tmax, int num_sms);
cudaError_t launch_decode_tc(const void* q, const void* kc, const void* vc, const int* seqlens,
                             void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window,
                             int ring, float scale_log2, const DecodePlan& plan, void* partials,
                             const DeviceInfo& dev, cudaStream_t stream);

// Backward pass (Dh 64 or 128): dq [B, Hq, S, Dh], dk and dv [B, Hkv, S, Dh]
// from q, k, v, the forward output o, its log-sum-exps lse [B, Hq, S] and
// dout; workspace holds bwd_workspace_bytes(B, Hq, S) bytes (16-byte aligned).
size_t bwd_workspace_bytes(int B, int Hq, int S);
cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       float* workspace, int B, int Hq, int Hkv, int S, int Dh, int causal,
                       int window, float scale, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace chs
