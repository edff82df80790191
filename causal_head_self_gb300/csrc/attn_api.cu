// attn_api.cu -- the C ABI declared in include/attn.h: argument checks,
// per-device state (SM count, latched error word, decode workspace), tensor
// maps, and the kernel launches.  No torch types cross this boundary.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

// Latched device-side status of the kernels (one per device: every device
// that loads this library holds its own copy of the symbol).
__device__ int g_attn_error_word;

struct DeviceState {
  bool ready = false;
  chs::DeviceInfo info{};
  // decode workspace: split partials, and completion counters kept in a
  // buffer of their own (always zero between calls)
  void* partials = nullptr;
  size_t partials_bytes = 0;
  int* counters = nullptr;
  size_t counters_n = 0;
  // backward workspace: per-row log-sum-exp (log2 units) and D = dO . o
  void* bwd_ws = nullptr;
  size_t bwd_ws_bytes = 0;
};

// Grow a device buffer (never inside a stream capture); zero it if asked.
int grow_buffer(void** buf, size_t* have, size_t need, bool zero, cudaStream_t stream) {
  if (*have >= need) return ATTN_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return ATTN_ERR_NO_MEMORY;   // cudaMalloc cannot run inside a capture
  if (*buf) cudaFree(*buf);      // cudaFree waits for work still using it
  *buf = nullptr;
  *have = 0;
  if (cudaMalloc(buf, need) != cudaSuccess) {
    *buf = nullptr;
    cudaGetLastError();
    return ATTN_ERR_NO_MEMORY;
  }
  if (zero && cudaMemset(*buf, 0, need) != cudaSuccess) {
    cudaFree(*buf);
    *buf = nullptr;
    return ATTN_ERR_CUDA;
  }
  *have = need;
  return ATTN_OK;
}

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode_fn() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Per-device set-up on first use, with that device current.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    void* word = nullptr;
    if (cudaGetSymbolAddress(&word, g_attn_error_word) != cudaSuccess) return ATTN_ERR_CUDA;
    if (!load_encode_fn()) return ATTN_ERR_CUDA;
    st.info.device = dev;
    st.info.num_sms = sms;
    st.info.error_word = static_cast<int*>(word);
    st.info.fault = 0;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// scale == 0 -> 1/sqrt(Dh); returns false for a negative or non-finite scale
bool resolve_scale(float scale, int Dh, float* scale_log2) {
  if (!std::isfinite(scale) || scale < 0.f) return false;
  const double s = scale == 0.f ? 1.0 / std::sqrt((double)Dh) : (double)scale;
  *scale_log2 = (float)(s * 1.4426950408889634);   // log2(e)
  return true;
}

}  // namespace

namespace chs {

// A tensor map is a pure function of these arguments, so a call that repeats
// an earlier one (the usual case: the same buffers every step) takes the map
// from a small per-thread cache instead of encoding it again.
namespace {
struct MapKey {
  const void* base;
  long long outer;
  int Dh, rows, box_rows, stride_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && outer == o.outer && Dh == o.Dh && rows == o.rows &&
           box_rows == o.box_rows && stride_rows == o.stride_rows;
  }
};
struct MapCache {
  static constexpr int kEntries = 64;
  MapKey key[kEntries];
  alignas(64) CUtensorMap map[kEntries];
  int used = 0, next = 0;
};
thread_local MapCache t_maps;
}  // namespace

bool encode_bf16_map(CUtensorMap* map, const void* base, int Dh, int rows, long long outer,
                     int box_rows, int stride_rows) {
  if (stride_rows == 0) stride_rows = rows;
  if (rows < 1 || stride_rows < rows) return false;
  const MapKey key{base, outer, Dh, rows, box_rows, stride_rows};
  MapCache& c = t_maps;
  for (int i = 0; i < c.used; ++i) {
    if (c.key[i] == key) {
      *map = c.map[i];
      return true;
    }
  }
  cuuint64_t dims[3] = {(cuuint64_t)Dh, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)Dh * 2, (cuuint64_t)Dh * 2 * (cuuint64_t)stride_rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t elem[3] = {1, 1, 1};
  if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int slot = c.next;
  c.key[slot] = key;
  c.map[slot] = *map;
  c.next = (slot + 1) % MapCache::kEntries;
  if (c.used < MapCache::kEntries) ++c.used;
  return true;
}

}  // namespace chs

extern "C" {

int attn_version(void) { return (1 << 16) | 0; }

const char* attn_error_string(int code) {
  switch (code) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_NO_MEMORY: return "ATTN_ERR_NO_MEMORY";
    case ATTN_ERR_SCRATCH_LIMIT: return "ATTN_ERR_SCRATCH_LIMIT";
    case ATTN_ERR_CHECK: return "ATTN_ERR_CHECK";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

// The test hook's current fault (attn_debug_inject_fault); 0 in normal use.
static std::atomic<int> g_fault{0};

static chs::DeviceInfo launch_info(const DeviceState* st) {
  chs::DeviceInfo d = st->info;
  d.fault = g_fault.load(std::memory_order_relaxed);
  return d;
}

int attn_debug_inject_fault(int kind) {
  if (kind < 0 || kind > 4) return ATTN_ERR_INVALID_ARG;
  g_fault.store(kind, std::memory_order_relaxed);
  return ATTN_OK;
}

// Shared by attn_fwd and attn_fwd_chunk: queries at positions
// start_pos .. start_pos + Sq - 1 against the first start_pos + Sq of Tkv
// key/value rows per head.
static int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Tkv, int start_pos, int Dh, int causal,
                      int window, float scale, cudaStream_t stream) {
  if (B < 0 || Sq < 0 || Tkv < 0 || start_pos < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if ((long long)start_pos + Sq > Tkv) return ATTN_ERR_INVALID_ARG;
  if (Dh != 64 && Dh != 128 && Dh != 256) return ATTN_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (window < 0) window = 0;
  if (window > 0 && !causal) return ATTN_ERR_INVALID_ARG;
  float scale_log2 = 0.f;
  if (!resolve_scale(scale, Dh, &scale_log2)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  const size_t qo_bytes = (size_t)B * Hq * Sq * Dh * 2, kv_bytes = (size_t)B * Hkv * Tkv * Dh * 2;
  if ((long long)B * Hq * ((Sq + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, qo_bytes, q, qo_bytes) || overlaps(o, qo_bytes, k, kv_bytes) ||
      overlaps(o, qo_bytes, v, kv_bytes))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const size_t lse_bytes = (size_t)B * Hq * Sq * 4;
    if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0 || overlaps(lse, lse_bytes, o, qo_bytes) ||
        overlaps(lse, lse_bytes, q, qo_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
        overlaps(lse, lse_bytes, v, kv_bytes))
      return ATTN_ERR_INVALID_ARG;
  }
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = chs::launch_prefill(q, k, v, o, lse, B, Hq, Hkv, Sq, Tkv, start_pos, Dh, causal,
                                      window, scale_log2, launch_info(st), stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int S,
             int Dh, int causal, int window, float scale, cudaStream_t stream) {
  return fwd_common(q, k, v, o, nullptr, B, Hq, Hkv, S, S, 0, Dh, causal, window, scale, stream);
}

int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int S, int Dh, int causal, int window, float scale,
                 cudaStream_t stream) {
  if (lse == nullptr && B > 0 && S > 0) return ATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, S, S, 0, Dh, causal, window, scale, stream);
}

int attn_fwd_chunk(const void* q, const void* kcache, const void* vcache, void* o, int B, int Hq,
                   int Hkv, int Sq, int Tmax, int start_pos, int Dh, int causal, int window,
                   float scale, cudaStream_t stream) {
  if (Tmax < 1) return ATTN_ERR_INVALID_ARG;
  return fwd_common(q, kcache, vcache, o, nullptr, B, Hq, Hkv, Sq, Tmax, start_pos, Dh, causal,
                    window, scale, stream);
}

// Argument and aliasing checks of every decode entry point (attn_decode,
// attn_decode_ring, attn_decode_noalloc), so that all three return the same
// errors for the same arguments.  On ATTN_OK, *window and *scale_log2 hold
// the resolved window (0: none) and softmax scale times log2(e); *empty is
// set when B == 0 (nothing to launch).
static int decode_check_args(const void* q, const void* kcache, const void* vcache,
                             const int* seqlens, const void* o, int B, int Hq, int Hkv, int Tmax,
                             int Dh, int* window, int ring, float scale, float* scale_log2,
                             bool* empty) {
  *empty = false;
  if (B < 0 || Tmax < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (Dh != 64 && Dh != 128 && Dh != 256) return ATTN_ERR_UNSUPPORTED;
  if (*window < 0) *window = 0;
  if (ring && *window > Tmax) return ATTN_ERR_INVALID_ARG;   // the ring holds Tmax positions
  if (!resolve_scale(scale, Dh, scale_log2)) return ATTN_ERR_INVALID_ARG;
  if (B == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (!q || !kcache || !vcache || !seqlens || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u))
    return ATTN_ERR_INVALID_ARG;
  const size_t qo_bytes = (size_t)B * Hq * Dh * 2;
  const size_t kv_bytes = (size_t)B * Hkv * Tmax * Dh * 2;
  if (overlaps(o, qo_bytes, q, qo_bytes) || overlaps(o, qo_bytes, kcache, kv_bytes) ||
      overlaps(o, qo_bytes, vcache, kv_bytes) || overlaps(o, qo_bytes, seqlens, (size_t)B * 4))
    return ATTN_ERR_INVALID_ARG;
  if ((long long)B * Hkv * (Hq / Hkv) > 65535LL * 65535LL) return ATTN_ERR_INVALID_ARG;
  if (B > 65535) return ATTN_ERR_INVALID_ARG;   // grid.z
  return ATTN_OK;
}

// Shared by attn_decode (ring = 0) and attn_decode_ring (ring = 1).
static int decode_common(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                         void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window, int ring,
                         float scale, cudaStream_t stream) {
  float scale_log2 = 0.f;
  bool empty = false;
  int rc = decode_check_args(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh, &window, ring,
                             scale, &scale_log2, &empty);
  if (rc != ATTN_OK || empty) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  if (Hq / Hkv >= chs::kDecodeTcMinGroup) {
    // two or more query heads per cached byte: the tensor-core path (a contraction)
    const chs::DecodePlan plan = chs::plan_decode_tc(B, Hq, Hkv, Tmax, st->info.num_sms);
    if ((long long)B * Hkv * ((Hq / Hkv + 127) / 128) > 65535) return ATTN_ERR_INVALID_ARG;
    void* partials = nullptr;
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      rc = grow_buffer(&st->partials, &st->partials_bytes,
                       chs::decode_partials_bytes(B, Hq, Dh, plan), false, stream);
      if (rc != ATTN_OK) return rc;
      partials = st->partials;
    }
    cudaError_t e = chs::launch_decode_tc(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh,
                                          window, ring, scale_log2, plan, partials,
                                          launch_info(st), stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const chs::DecodePlan plan = chs::plan_decode(B, Hq, Hkv, Tmax, Dh, st->info.num_sms);
  if ((long long)Hkv * ((Hq / Hkv) / plan.heads_per_cta) > 65535) return ATTN_ERR_INVALID_ARG;
  const size_t need_partials = chs::decode_partials_bytes(B, Hq, Dh, plan);
  const size_t need_counters = chs::decode_counter_count(B, Hq, Hkv, plan);
  void* partials = nullptr;
  int* counters = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    rc = grow_buffer(&st->partials, &st->partials_bytes, need_partials, false, stream);
    if (rc != ATTN_OK) return rc;
    size_t counter_bytes = st->counters_n * sizeof(int);
    void* cbuf = st->counters;
    rc = grow_buffer(&cbuf, &counter_bytes, need_counters * sizeof(int), true, stream);
    st->counters = static_cast<int*>(cbuf);
    st->counters_n = counter_bytes / sizeof(int);
    if (rc != ATTN_OK) return rc;
    partials = st->partials;
    counters = st->counters;
  }
  cudaError_t e = chs::launch_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh, window,
                                     ring, scale_log2, plan, counters, partials, launch_info(st),
                                     stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int Dh,
             int causal, int window, float scale, cudaStream_t stream) {
  if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (Dh != 64 && Dh != 128 && Dh != 256) return ATTN_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (window < 0) window = 0;
  if (window > 0 && !causal) return ATTN_ERR_INVALID_ARG;
  float scale_log2 = 0.f;
  if (!resolve_scale(scale, Dh, &scale_log2)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return ATTN_OK;
  const void* in[] = {q, k, v, o, dout};
  void* out[] = {dq, dk, dv};
  for (const void* x : in)
    if (!x || !aligned16(x)) return ATTN_ERR_INVALID_ARG;
  for (const void* x : out)
    if (!x || !aligned16(x)) return ATTN_ERR_INVALID_ARG;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * Hq * ((S + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * Hq * S * Dh * 2, kb = (size_t)B * Hkv * S * Dh * 2;
  const size_t in_bytes[] = {qb, kb, kb, qb, qb};
  const size_t out_bytes[] = {qb, kb, kb};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 5; ++b)
      if (overlaps(out[a], out_bytes[a], in[b], in_bytes[b])) return ATTN_ERR_INVALID_ARG;
    if (overlaps(out[a], out_bytes[a], lse, (size_t)B * Hq * S * 4)) return ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(out[a], out_bytes[a], out[b], out_bytes[b])) return ATTN_ERR_INVALID_ARG;
  }
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    rc = grow_buffer(&st->bwd_ws, &st->bwd_ws_bytes, chs::bwd_workspace_bytes(B, Hq, S), false,
                     stream);
    if (rc != ATTN_OK) return rc;
    ws = st->bwd_ws;
  }
  const float sc = scale == 0.f ? (float)(1.0 / std::sqrt((double)Dh)) : scale;
  cudaError_t e = chs::launch_bwd(q, k, v, o, dout, lse, dq, dk, dv, static_cast<float*>(ws), B,
                                  Hq, Hkv, S, Dh, causal, window, sc, launch_info(st), stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_decode(const void* q, const void* kcache, const void* vcache, const int* seqlens, void* o,
                int B, int Hq, int Hkv, int Tmax, int Dh, int window, float scale,
                cudaStream_t stream) {
  return decode_common(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh, window, 0, scale,
                       stream);
}

int attn_decode_ring(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                     void* o, int B, int Hq, int Hkv, int C, int Dh, int window, float scale,
                     cudaStream_t stream) {
  return decode_common(q, kcache, vcache, seqlens, o, B, Hq, Hkv, C, Dh, window, 1, scale, stream);
}

int attn_status(cudaStream_t stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyAsync(&word, st->info.error_word, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaMemsetAsync(st->info.error_word, 0, sizeof(int), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return word;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_decode_noalloc: the decode step for callers that must not allocate
// device memory.  Its split partials and completion counters live in one
// file-scope device array instead of the library's cudaMalloc'd workspace.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB per device

// Held by every device that loads this library, until the process exits.
// In host code this name is only a stand-in: the device address comes from
// cudaGetSymbolAddress, taken once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

unsigned char* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                                   const int* seqlens, void* o, int B, int Hq, int Hkv, int Tmax,
                                   int Dh, int window, float scale, cudaStream_t stream) {
  float scale_log2 = 0.f;
  bool empty = false;
  int rc = decode_check_args(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh, &window, 0,
                             scale, &scale_log2, &empty);
  if (rc != ATTN_OK || empty) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  // the fixed array's address, looked up once per device with that device current
  auto scratch_ptr = [&](unsigned char** out) -> int {
    std::lock_guard<std::mutex> lock(g_mutex);
    const int dev = st->info.device;
    if (!g_noalloc_ptr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return ATTN_ERR_CUDA;
      g_noalloc_ptr[dev] = static_cast<unsigned char*>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return ATTN_OK;
  };
  unsigned char* scratch = nullptr;
  if (Hq / Hkv >= chs::kDecodeTcMinGroup) {
    // query-head groups: the tensor-core path, as in attn_decode; its
    // split partials are the scratch's only content (it keeps no counters)
    const chs::DecodePlan plan = chs::plan_decode_tc(B, Hq, Hkv, Tmax, st->info.num_sms);
    if ((long long)B * Hkv * ((Hq / Hkv + 127) / 128) > 65535) return ATTN_ERR_INVALID_ARG;
    if (chs::decode_partials_bytes(B, Hq, Dh, plan) > kNoAllocScratchBytes)
      return ATTN_ERR_SCRATCH_LIMIT;
    if ((rc = scratch_ptr(&scratch)) != ATTN_OK) return rc;
    cudaError_t e = chs::launch_decode_tc(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh,
                                          window, 0, scale_log2, plan, scratch,
                                          launch_info(st), stream);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  const chs::DecodePlan plan = chs::plan_decode(B, Hq, Hkv, Tmax, Dh, st->info.num_sms);
  if ((long long)Hkv * ((Hq / Hkv) / plan.heads_per_cta) > 65535) return ATTN_ERR_INVALID_ARG;
  // scratch layout: counters (256-byte aligned) | split partials
  const size_t n_counters = chs::decode_counter_count(B, Hq, Hkv, plan);
  const size_t counter_bytes = (n_counters * sizeof(int) + 255) / 256 * 256;
  const size_t partial_bytes = chs::decode_partials_bytes(B, Hq, Dh, plan);
  if (counter_bytes + partial_bytes > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
  if ((rc = scratch_ptr(&scratch)) != ATTN_OK) return rc;
  int* counters = reinterpret_cast<int*>(scratch);
  // the array keeps the previous call's contents: the counters must start at zero
  if (cudaMemsetAsync(counters, 0, n_counters * sizeof(int), stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  cudaError_t e = chs::launch_decode(q, kcache, vcache, seqlens, o, B, Hq, Hkv, Tmax, Dh, window,
                                     0, scale_log2, plan, counters, scratch + counter_bytes,
                                     launch_info(st), stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
