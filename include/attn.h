/*
 * attn.h -- C ABI of the GB300 (sm_103a) scaled dot-product causal
 * multi-head self-attention library (libattn_sm103a.so).
 *
 * The operation is the one defined in "Механизм внимания"
 * (llm-arch-research.openidealab.com/textbook/attention), section
 * "Scaled dot-product attention":
 *
 *     O = softmax(Q K^T * scale + M) V        per (batch b, query head h)
 *
 * with M in {0, -inf} the mask of sections "Маскирование" (causal: key j is
 * visible to query i only if j <= i) and "Скользящее окно" (sliding window),
 * and query head h reading K/V head g(h) = floor(h / (Hq / Hkv)) as in
 * section "Виды по числу голов K/V: MHA, GQA, MQA" (Hkv == Hq is MHA,
 * Hkv == 1 is MQA).
 *
 * Conventions shared by every entry point:
 *   - Tensors are bf16, contiguous, row-major, in the layout [B, H, S, Dh]
 *     ("多头注意力机制" (blog.euler0525.cn), section "Multi-head Attention":
 *     heads moved ahead of the sequence axis).  All tensor pointers are
 *     DEVICE pointers, 16-byte aligned.  The caller owns every tensor.
 *   - Dh must be 64, 128 or 256 (the Gemma head size) for every entry
 *     point (ATTN_ERR_UNSUPPORTED otherwise).
 *   - Hq % Hkv == 0 is required (ATTN_ERR_INVALID_ARG otherwise).
 *   - scale == 0 selects 1/sqrt(Dh), the textbook's choice (divide by the
 *     square root of the HEAD size, not the model width); a positive scale is
 *     used as given; a negative or non-finite scale is ATTN_ERR_INVALID_ARG.
 *   - window <= 0 means no window.  window = W > 0 keeps key j visible to the
 *     query at position i only if i - W < j <= i: W keys including the
 *     query's own (the i - j < W form the textbook quotes from HuggingFace;
 *     the page's own rule 0 <= i - j <= W equals window W + 1 here).
 *   - Argument errors are returned before anything is launched.  Kernels run
 *     asynchronously on `stream`; a launch failure returns ATTN_ERR_CUDA.
 *     Errors found on the device (a bounded wait that gave up, an invalid
 *     sequence length) are latched in a per-device error word that
 *     attn_status() reads.  After a non-OK status the output is undefined.
 *   - The same inputs give bit-identical outputs (no atomics in any
 *     reduction; the decode split plan depends only on the arguments and
 *     the device's SM count).
 *   - Workspaces (the decode split partials and completion counters, the
 *     backward pass's per-row statistics) belong to the library, one set
 *     per device, grown under a lock and never shrunk.  They are shared by
 *     every stream of the device: calls that use them (attn_decode,
 *     attn_decode_ring, attn_bwd) may be issued from several host threads,
 *     but must not run concurrently on different streams of one device.
 *     attn_decode_noalloc uses a fixed array of its own instead, under the
 *     same rule (see there).  Growing a workspace is refused inside a
 *     stream capture (ATTN_ERR_NO_MEMORY): make one call outside the
 *     capture first.
 */
#ifndef CAUSAL_HEAD_SELF_ATTN_H_
#define CAUSAL_HEAD_SELF_ATTN_H_

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* bad shape, pointer, alignment, aliasing, scale or window */
  ATTN_ERR_UNSUPPORTED = 2,  /* a head size the entry point does not take */
  ATTN_ERR_CUDA = 3,         /* a CUDA runtime or launch error */
  ATTN_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (reported by attn_status) */
  ATTN_ERR_NO_MEMORY = 5,    /* a library workspace could not be allocated */
  ATTN_ERR_SCRATCH_LIMIT = 6, /* attn_decode_noalloc: the call needs more than its fixed scratch */
  ATTN_ERR_CHECK = 7          /* checked builds only (ATTN_CHECK): a kernel's own range check of a
                                 copy it was about to issue failed; the copy was skipped */
} attn_status_t;

/*
 * attn_fwd -- prefill / full-sequence attention.
 *   q  [B, Hq,  S, Dh]   queries          (device, bf16, read)
 *   k  [B, Hkv, S, Dh]   keys             (device, bf16, read)
 *   v  [B, Hkv, S, Dh]   values           (device, bf16, read)
 *   o  [B, Hq,  S, Dh]   output           (device, bf16, written; must not
 *                                           overlap q, k or v)
 *   causal   1: causal mask; 0: every key visible (window must then be <= 0)
 *   window, scale: see the conventions above.
 * B == 0 or S == 0 is a no-op returning ATTN_OK.
 * Work: 4*Dh FLOPs per visible (query, key) pair per query head; wholly
 * masked tiles (128 query rows by 128 keys, or by 64 keys at Dh 256 and at
 * Dh 128 up to 1536 keys per head) are never computed.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
             int S, int Dh, int causal, int window, float scale, cudaStream_t stream);

/*
 * attn_fwd_lse -- attn_fwd that also writes each query row's log-sum-exp,
 *   lse  [B, Hq, S]  (device, fp32, written; 4-byte aligned, must not
 *                     overlap the other tensors)
 *   lse[b, h, i] = log sum_j exp(s_ij) over the visible keys j, natural log,
 *   with s_ij = scale * q_i . k_j the scaled score (the softmax
 *   normaliser of "Механизм внимания", section "Scaled dot-product
 *   attention", in log form).  attn_bwd recomputes the weights from it.
 * o is bit-identical to attn_fwd's.  lse == NULL is ATTN_ERR_INVALID_ARG
 * (unless B == 0 or S == 0, a no-op).
 */
int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int S, int Dh, int causal, int window, float scale,
                 cudaStream_t stream);

/*
 * attn_bwd -- backward pass of attn_fwd: the gradients of a loss L with
 * respect to q, k and v, given dout = dL/do.  The chain rule through the
 * definition, with the softmax derivative dp_i/dz_j = p_i (delta_ij - p_j)
 * of "Механизм внимания", section "Почему делить на корень из d_h"; the
 * weights are recomputed block by block from lse (section "Эффективные
 * реализации": FlashAttention recomputes them in the backward pass):
 *     dV = P^T dO,  dS = P o (dO V^T - D),  D_i = dO_i . o_i,
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, causal, window, scale  exactly as passed to attn_fwd_lse
 *   o     [B, Hq,  S, Dh]  attn_fwd_lse's output       (device, bf16, read)
 *   dout  [B, Hq,  S, Dh]  dL/do                       (device, bf16, read)
 *   lse   [B, Hq,  S]      attn_fwd_lse's lse          (device, fp32, read)
 *   dq    [B, Hq,  S, Dh]  dL/dq                       (device, bf16, written)
 *   dk    [B, Hkv, S, Dh]  dL/dk, summed over the query heads of each group
 *   dv    [B, Hkv, S, Dh]  dL/dv, likewise             (device, bf16, written)
 * dq, dk and dv must not overlap each other or any input.  Dh must be 64,
 * 128 or 256 (ATTN_ERR_UNSUPPORTED otherwise).  The result is deterministic
 * (no atomics): at Dh 64 and 128 one pass computes dK and dV per key block, a
 * second dQ per query block; at Dh 256, where a 256-column accumulator fills
 * half of tensor memory, dV, dK and dQ each take a pass of their own.
 * Per-row intermediates live in a library-owned device workspace
 * (8 bytes per query row, allocated on first use and grown on demand,
 * ATTN_ERR_NO_MEMORY if that fails); backward calls that overlap on the GPU
 * race on it.  B == 0 or S == 0 is a no-op.
 * Work: 10*Dh FLOPs per visible (query, key) pair per query head (S
 * recomputed, dP, dV, dQ, dK: 2*Dh each), 2.5 x attn_fwd's; the kernels
 * execute 14*Dh (S and dP are computed in both passes; at Dh 256, 16*Dh:
 * S in all three passes, dP in two).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int S, int Dh,
             int causal, int window, float scale, cudaStream_t stream);

/*
 * attn_fwd_chunk -- prefill of one chunk against a KV cache ("Механизм
 * внимания", section "Prefill и decode": a long prompt may be fed in chunks;
 * the chunk's keys and values are written into the cache first, then its
 * queries attend to everything cached before them and to the chunk).
 *   q       [B, Hq, Sq, Dh]     the chunk's queries        (device, bf16, read)
 *   kcache  [B, Hkv, Tmax, Dh]  cached keys                (device, bf16, read)
 *   vcache  [B, Hkv, Tmax, Dh]  cached values              (device, bf16, read)
 *   o       [B, Hq, Sq, Dh]     output                     (device, bf16, written;
 *                                                           must not overlap the others)
 *   start_pos  position of the chunk's first token; the chunk's own keys
 *              are cache rows start_pos .. start_pos + Sq - 1, and only rows
 *              [0, start_pos + Sq) are read (0 <= start_pos, start_pos + Sq <= Tmax).
 * Query row r sits at position start_pos + r and, with causal = 1, sees keys
 * 0 .. start_pos + r (the window, if any, as in attn_fwd); with causal = 0
 * every key 0 .. start_pos + Sq - 1.  start_pos = 0 and Tmax = Sq is exactly
 * attn_fwd (the same kernel and bits).  Errors and the empty case (B == 0 or
 * Sq == 0) as in attn_fwd.
 */
int attn_fwd_chunk(const void* q, const void* kcache, const void* vcache, void* o, int B, int Hq,
                   int Hkv, int Sq, int Tmax, int start_pos, int Dh, int causal, int window,
                   float scale, cudaStream_t stream);

/*
 * attn_decode -- one KV-cache decode step ("Механизм внимания", section
 * "Prefill и decode": the new token's key and value are appended to the
 * cache first, then its query meets every cached key, its own included).
 *   q        [B, Hq, 1, Dh]     the new tokens' queries   (device, bf16, read)
 *   kcache   [B, Hkv, Tmax, Dh] cached keys               (device, bf16, read)
 *   vcache   [B, Hkv, Tmax, Dh] cached values             (device, bf16, read)
 *   seqlens  [B]                keys held per sequence, 1 <= seqlens[b] <= Tmax
 *                               (device, int32, read).  Only rows
 *                               [0, seqlens[b]) of a cache are read.
 *   o        [B, Hq, 1, Dh]     output (device, bf16, written)
 * The query of sequence b sits at position seqlens[b] - 1 and sees keys
 * [max(0, seqlens[b] - window), seqlens[b]) (all of them when window <= 0).
 * A seqlens entry outside [1, Tmax] zeroes that sequence's output and latches
 * ATTN_ERR_INVALID_ARG for attn_status().
 * With Hq / Hkv >= 2 (GQA and MQA) the step runs on the tensor cores (the
 * group's query heads packed as the rows of one contraction with each key
 * tile) followed by a small combine kernel (a programmatic dependent launch
 * on the same stream); with one query head per K/V head (MHA) on the CUDA
 * cores, whose last CTA per head merges the splits.
 * The split-KV partials live in a library-owned device workspace, allocated
 * on first use per device and grown on demand (cudaMalloc): make the first
 * call with the largest shape outside any CUDA graph capture.  Calls on one
 * device share that workspace, so decode calls that overlap on the GPU
 * (different streams, no ordering) race.
 * B == 0 is a no-op returning ATTN_OK.
 */
int attn_decode(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                void* o, int B, int Hq, int Hkv, int Tmax, int Dh, int window, float scale,
                cudaStream_t stream);

/*
 * attn_decode_ring -- the decode step over a rolling-buffer cache
 * ("Механизм внимания", section "Скользящее окно": with a window the cache
 * need only hold the last W positions, and a ring buffer does that).
 *   kcache, vcache [B, Hkv, C, Dh]: position t of sequence b is at row t % C
 *                  (the last min(seqlens[b], C) positions are held).
 *   seqlens [B]    tokens of sequence b so far, own token included (>= 1,
 *                  any size below 2^31 - C); the query sits at position
 *                  seqlens[b] - 1.
 *   window         W <= C: keys [seqlens[b] - W, seqlens[b]) are visible;
 *                  window <= 0 means W = C (every held position).
 *                  window > C is ATTN_ERR_INVALID_ARG.
 * Other arguments, the workspace and the errors as in attn_decode.  While a
 * sequence has not wrapped (seqlens[b] <= C) and window <= 0 the result is
 * bit-identical to attn_decode on the same buffers.
 */
int attn_decode_ring(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                     void* o, int B, int Hq, int Hkv, int C, int Dh, int window, float scale,
                     cudaStream_t stream);

/*
 * attn_decode_noalloc -- the same decode step as attn_decode (same arguments,
 * same result up to rounding, same errors), for callers that must not
 * allocate device memory.  The pages describe no such call; it exists for
 * this library's users.  A serving runtime that reserves nearly all device
 * memory up front for its own KV-cache pool, or a process that runs under a
 * fixed device-memory budget, cannot let a library allocate behind its back:
 * an allocation there can fail, and cudaMalloc / cudaFree also stall on the
 * device.  attn_decode allocates its workspace on first use; this entry point
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Its scratch (split partials and completion counters) is one fixed
 *     16 MiB device array inside this library.  Every GPU that loads the
 *     library holds it until the process exits.
 *   - It runs the kernels attn_decode runs for the same arguments (the
 *     tensor-core path for Hq / Hkv >= 2 at every head size, the CUDA-core
 *     path otherwise), with the same split plan, so the results are the
 *     same bits.
 *   - On the CUDA-core path a call needs 4*B*Hq bytes of counters (one per
 *     query head, rounded up to 256 bytes) plus
 *     B*Hq*nsplit*(Dh+2)*4 bytes of partials (each part rounded up to 256),
 *     where nsplit is the split count attn_decode would use; on the
 *     tensor-core path only the partials.  A call that needs more than
 *     16 MiB returns ATTN_ERR_SCRATCH_LIMIT before anything runs.  (The
 *     B=16, Hq=32, Hkv=8, Tmax=32768, Dh=128 decode step needs about 4.3 MB.)
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents; each call clears the counters it uses (cudaMemsetAsync on
 *     `stream`).  Calls that overlap on the GPU (on different streams with no
 *     ordering between them) race on the array and give wrong results.
 */
int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                        const int* seqlens, void* o, int B, int Hq, int Hkv, int Tmax, int Dh,
                        int window, float scale, cudaStream_t stream);

/*
 * attn_status -- synchronise `stream`, then return (and clear) the current
 * device's latched error word: ATTN_OK, ATTN_ERR_TIMEOUT, ATTN_ERR_INVALID_ARG,
 * or ATTN_ERR_CUDA if the synchronisation itself failed (or a prefill kernel
 * found its dynamic shared memory not 1024-byte aligned and wrote nothing).
 */
int attn_status(cudaStream_t stream);

/*
 * attn_debug_inject_fault -- test hook for the failure path; the pages
 * describe no such call.  Every later attn_fwd / attn_decode /
 * attn_decode_noalloc / attn_bwd launch in this process runs with the given fault until
 * it is reset with kind 0:
 *   0  none (the default)
 *   1  attn_fwd: the producer never loads the first K tile of each CTA's
 *      first work item, so the MMA issuers' bounded waits run out
 *   2  attn_decode (CUDA-core path, Hq == Hkv): the producer never loads the
 *      first key block of each CTA
 *   3  attn_decode (tensor-core path, Hq / Hkv >= 2): the producer never loads
 *      the first K tile of each CTA
 *   4  attn_bwd: the dK/dV pass's producer never loads the K/V block of each
 *      CTA's first work item
 * A faulted launch ends by itself after its waits give up (about 2 s): no
 * GPU fault, trap or hang.  attn_status() then returns ATTN_ERR_TIMEOUT and
 * clears it; the outputs of that launch are undefined, and the next launch
 * without a fault is correct (the decode completion counters are left at
 * zero).  Returns ATTN_OK, or ATTN_ERR_INVALID_ARG for an unknown kind.
 * Not for production use: the setting is process-wide and unsynchronised
 * with launches already queued.
 */
int attn_debug_inject_fault(int kind);

/* attn_error_string -- a static, human-readable name for a status code. */
const char* attn_error_string(int code);

/* attn_version -- library ABI version, (major << 16) | minor. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CAUSAL_HEAD_SELF_ATTN_H_ */
