/*
 * attn_prefill.h — C ABI of the GB300 (sm_103a) causal GQA prefill attention:
 * the forward pass (square and chunked, bf16 and fp8), decode, the backward
 * pass and two diagnostics.
 *
 * Operation (one call computes, for every batch b, query head h and row i):
 *
 *     kv(h)       = h / g,  g = n_q / n_kv            (contiguous head groups)
 *     s_ij        = scale * dot(Q[b,i,h,:], K[b,j,kv(h),:])
 *     J(i)        = {0..i} if causal, else {0..L-1}    (diagonal kept)
 *     O[b,i,h,:]  = sum_{j in J(i)} softmax_j(s_i.) * V[b,j,kv(h),:]
 *     LSE[b,h,i]  = ln sum_{j in J(i)} exp(s_ij)
 *
 * as defined by "Why Attention Scaling Breaks" (shivam2003), section
 * "The O(n^2) problem" (S = Q K^T, A = softmax(S / sqrt(d)), O = A V), with
 * the causal restriction of "Long-Context Attention Explained" (sevydevy),
 * quadratic-cost section (each token looks only backwards, itself included),
 * and the grouped K/V heads of the "prefill-attention" flop record
 * (phantomic12), "Workarounds" (MQA/GQA). It is evaluated the FlashAttention
 * way, tile by tile with an online softmax ("Long-Context Attention
 * Explained", sections "Tiling" and "Online softmax"), so the L x L score
 * matrix never reaches device memory.
 *
 * Layouts (all row-major, contiguous, device memory):
 *     q   bf16 [B, L, n_q,  d_h]
 *     k   bf16 [B, L, n_kv, d_h]
 *     v   bf16 [B, L, n_kv, d_h]
 *     o   bf16 [B, L, n_q,  d_h]   written
 *     lse fp32 [B, n_q, L]         written (natural log, of the scaled scores)
 *
 * Ownership: the caller allocates and owns q, k, v, o, lse and the stream.
 * The library never frees caller memory and allocates nothing per call. On
 * the first call on a device it allocates one 256-byte status word for that
 * device (kept until process exit) and sets the kernels' shared-memory limit.
 *
 * Execution: asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream). The call returns after the launch is enqueued; o and lse are valid
 * once the stream has reached that point. q, k, v are not modified. Results
 * are deterministic: the same inputs give bit-identical o and lse.
 *
 * CUDA graphs: the first call of each family (forward, decode, backward) on a
 * device does a one-time set-up and must not be made while a stream capture
 * is under way; made there, it returns ATTN_ERR_UNSUPPORTED and sets up
 * nothing. After it, every compute entry point can be captured with the
 * stream it is given (attn_decode_fwd as two kernel nodes joined by a
 * programmatic dependency); replaying the graph recomputes from whatever the
 * captured input buffers hold then. attn_device_check synchronizes and cannot
 * be captured. attn_prefill_fwd_host enqueues its copies and its launch on
 * the caller's stream like the other entry points, but it is not covered by
 * this library's capture tests, so nothing is promised for it under capture.
 */
#ifndef ATTN_PREFILL_H
#define ATTN_PREFILL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, n_q % n_kv != 0,
                                Lk < Lq, non-finite scale, causal not 0/1,
                                misaligned pointer */
  ATTN_ERR_UNSUPPORTED = 2,  /* d_h not 64 or 128 (128 for fp8), sizes beyond 32-bit
                                tile indexing, device that is not sm_103, a first
                                call on a device made during stream capture */
  ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call or the launch failed */
  ATTN_ERR_TIMEOUT = 4,      /* a kernel wait ran past its limit (reported by
                                attn_device_check); outputs of that launch are
                                undefined */
  ATTN_ERR_CHECK = 5         /* a device-side consistency check failed (only the
                                library built with ATTN_DEBUG runs them; reported
                                by attn_device_check); outputs undefined */
} attn_status_t;

/*
 * Causal (or full) GQA attention forward over bf16 [B, L, H, d_h] tensors.
 *
 *   q, k, v   device pointers, 16-byte aligned, layouts above
 *   o         device pointer, 16-byte aligned, bf16 [B, L, n_q, d_h]
 *   lse       device pointer, 4-byte aligned, fp32 [B, n_q, L]; never NULL
 *   B, L      batch size and sequence length, >= 1
 *   n_q, n_kv query heads and K/V heads, >= 1, n_q a multiple of n_kv
 *   d_h       head dimension: 64 or 128
 *   causal    1: key j <= query i is kept (diagonal included); 0: all keys
 *   scale     finite multiplier of the dot products (1/sqrt(d_h) in the usual
 *             case; 0 and negative values are allowed)
 *   stream    cudaStream_t to enqueue on, passed as void*
 *
 * Returns ATTN_OK after enqueueing. Argument errors return synchronously
 * before any CUDA call or launch. A device-side wait that runs past its
 * limit is reported by attn_device_check().
 */
attn_status_t attn_prefill_fwd(const void* q, const void* k, const void* v,
                               void* o, float* lse,
                               int64_t B, int64_t L, int32_t n_q, int32_t n_kv,
                               int32_t d_h, int32_t causal, float scale,
                               void* stream);

/*
 * Chunked prefill: the query is the last Lq positions of a sequence whose
 * Lk >= Lq keys and values (earlier chunks' and its own) are all present, as
 * when a long prompt is prefilled piece by piece ("prefill-attention" flop
 * record (phantomic12), "Workarounds": chunked prefill splits a long prompt
 * into pieces). Query row i sits at absolute position i + Lk - Lq; with
 * causal = 1 it attends to keys j <= i + Lk - Lq (the chunk is aligned to the
 * end of the key range), with causal = 0 to all Lk keys.
 *
 *   q    bf16 [B, Lq, n_q,  d_h]       k, v  bf16 [B, Lk, n_kv, d_h]
 *   o    bf16 [B, Lq, n_q,  d_h]       lse   fp32 [B, n_q, Lq]
 *   1 <= Lq <= Lk; every other argument, alignment rule, ownership and error
 *   behaviour as attn_prefill_fwd, which is this call with Lq = Lk.
 */
attn_status_t attn_prefill_fwd_chunk(const void* q, const void* k, const void* v,
                                     void* o, float* lse,
                                     int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                     int32_t n_kv, int32_t d_h, int32_t causal, float scale,
                                     void* stream);

/*
 * FP8 variant: Q, K and V in e4m3 (OCP FP8 E4M3, 1 byte per element, same
 * [B, L, H, d_h] layouts) with per-tensor descale factors, so the real inputs
 * are q*q_descale, k*k_descale, v*v_descale ("prefill-attention" flop record
 * (phantomic12), "Workarounds": FP8 attention doubles the tensor rate and the
 * ridge). Both products run on the fp8 tensor cores with fp32 accumulation;
 * the softmax weights P are rounded to e4m3 for the P.V product (their row
 * sum stays fp32). O is bf16 and LSE fp32 as above, of the scaled real
 * scores. Chunks work as in attn_prefill_fwd_chunk (1 <= Lq <= Lk).
 *
 *   d_h must be 128 (ATTN_ERR_UNSUPPORTED otherwise); descales must be
 *   finite (ATTN_ERR_INVALID_ARG otherwise). Everything else as
 *   attn_prefill_fwd.
 */
attn_status_t attn_prefill_fwd_fp8(const void* q, const void* k, const void* v,
                                   void* o, float* lse,
                                   int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                   int32_t n_kv, int32_t d_h, int32_t causal, float scale,
                                   float q_descale, float k_descale, float v_descale,
                                   void* stream);

/*
 * Decode attention: one new query token per sequence attends to its whole
 * key/value cache ("Long-Context Attention Explained" (sevydevy), prefill vs
 * decode: decode has one new query per step and reads every cached key and
 * value). It is attn_prefill_fwd_chunk with Lq = 1 (the token sits at
 * position Lk - 1, so it sees keys 0..Lk-1), computed by a kernel built for
 * a memory-bound step: the key range is split over many CTAs that stream K
 * and V once, and a second kernel merges the partial results.
 *
 *   q    bf16 [B, 1, n_q, 128]           k, v  bf16 [B, Lk, n_kv, 128]
 *   o    bf16 [B, 1, n_q, 128]           lse   fp32 [B, n_q, 1]
 *   workspace  device memory of at least attn_decode_workspace_bytes(...)
 *              bytes, 16-byte aligned, owned by the caller; its contents
 *              on entry are ignored and on exit unspecified.
 *   n_q / n_kv <= 16 and d_h = 128 (ATTN_ERR_UNSUPPORTED otherwise); a NULL
 *   or too-small workspace is ATTN_ERR_INVALID_ARG. Everything else as
 *   attn_prefill_fwd.
 *
 * Both kernels are launched as programmatic dependents (CUDA programmatic
 * dependent launch) of the kernel before them on `stream`: they may start
 * their set-up while that kernel finishes, but each waits for it to complete
 * before touching global memory, so stream order holds for every input and
 * for the workspace. The merge kernel lets the next kernel on the stream
 * start its own set-up early in the same way; a kernel launched without that
 * attribute waits for the call's completion as usual.
 */
int64_t attn_decode_workspace_bytes(int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv,
                                    int32_t d_h);   /* -1 on invalid or unsupported sizes */
attn_status_t attn_decode_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, int64_t workspace_bytes,
                              int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv, int32_t d_h,
                              float scale, void* stream);

/*
 * Backward pass: gradients of attn_prefill_fwd with respect to q, k and v for
 * an upstream gradient dout, computed by rebuilding the score tiles from q, k
 * and the forward's lse instead of storing the L x L table ("Long-Context
 * Attention Explained" (sevydevy), "What FlashAttention does not change":
 * the backward pass recomputes the blocks from the saved row statistics).
 * With P the forward's softmax weights (masked entries 0), D_i = dout_i . o_i:
 *
 *     dV_j = sum_i P_ij dout_i                 dP_ij = dout_i . V_j
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i = scale sum_j dS_ij K_j             dK_j = scale sum_i dS_ij Q_i
 *
 * where the sums for dK and dV run over every query head of the K/V head's
 * group. No atomics: results are deterministic.
 *
 *   q, k, v, o, lse   the forward's inputs and outputs (layouts above)
 *   dout              bf16 [B, L, n_q, d_h], 16-byte aligned
 *   dq                bf16 [B, L, n_q, d_h]   written
 *   dk, dv            bf16 [B, L, n_kv, d_h]  written
 *   workspace         device memory of at least attn_prefill_bwd_workspace_bytes
 *                     bytes, 16-byte aligned, owned by the caller; contents on
 *                     entry ignored, on exit unspecified
 *   d_h must be 64 or 128 (ATTN_ERR_UNSUPPORTED otherwise); square problems only
 *   (the forward's Lq = Lk = L). Everything else as attn_prefill_fwd.
 *
 * Launches: a row kernel, then the dK/dV kernel as its programmatic
 * dependent (set-up overlaps the row kernel's end; it waits for it before
 * reading), then the dQ kernel as dK/dV's programmatic dependent (it reads
 * only the inputs and the row statistics, so it starts on the SMs dK/dV's
 * last CTAs free; it does not end before dK/dV has). Every result is complete
 * when the call's last kernel is, for stream-ordered and programmatic
 * successors alike.
 */
int64_t attn_prefill_bwd_workspace_bytes(int64_t B, int64_t L, int32_t n_q, int32_t n_kv,
                                         int32_t d_h);   /* -1 on invalid or unsupported sizes */
attn_status_t attn_prefill_bwd(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout,
                               void* dq, void* dk, void* dv,
                               void* workspace, int64_t workspace_bytes,
                               int64_t B, int64_t L, int32_t n_q, int32_t n_kv, int32_t d_h,
                               int32_t causal, float scale, void* stream);

/*
 * Forward pass over host buffers (no counterpart on the pages: a deployment
 * convenience for callers whose tensors live in host memory). Enqueues on
 * `stream`: one cudaMemcpyAsync per input (q, k, v) into `staging`, the
 * forward pass of attn_prefill_fwd_chunk there, and one cudaMemcpyAsync per
 * result (o, lse) back to the host buffers. Returns after enqueueing; the
 * host outputs are valid once the stream has reached that point.
 *
 *   q, k, v, o, lse  host pointers, same layouts and sizes as the device entry
 *                    points (Lq = Lk is a square prefill). Page-locked host
 *                    memory lets the copies overlap other work; pageable
 *                    memory works but the copies may then synchronise.
 *   staging          device memory of at least attn_prefill_host_staging_bytes
 *                    bytes, 256-byte aligned, owned by the caller; holds the
 *                    device copies of q, k, v, o, lse; contents on entry
 *                    ignored, on exit unspecified. A call must not share a
 *                    staging buffer with another call still in flight.
 *   Every check of attn_prefill_fwd_chunk (arguments, sizes, the device and
 *   its first-call set-up) runs before the first copy is enqueued, so
 *   ATTN_ERR_INVALID_ARG (NULL pointers, a misaligned or too-small staging
 *   buffer, the forward's argument errors) and ATTN_ERR_UNSUPPORTED (its
 *   unsupported sizes or device, a first call during capture) leave nothing
 *   enqueued. ATTN_ERR_CUDA: a copy or the launch could not be enqueued
 *   (work enqueued before it stays on the stream).
 */
int64_t attn_prefill_host_staging_bytes(int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                        int32_t n_kv, int32_t d_h);  /* -1 on invalid sizes */
attn_status_t attn_prefill_fwd_host(const void* q, const void* k, const void* v,
                                    void* o, float* lse, void* staging, int64_t staging_bytes,
                                    int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                    int32_t n_kv, int32_t d_h, int32_t causal, float scale,
                                    void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* attn_status_string(attn_status_t status);

/*
 * Synchronises `stream`, then reports: ATTN_ERR_CUDA if the stream or an
 * earlier launch failed, ATTN_ERR_TIMEOUT if any launch on the current device
 * since the previous check hit a wait limit, else ATTN_OK. It reads two
 * status words, the one the allocating entry points share and the fixed one
 * of attn_prefill_fwd_noalloc, and clears whichever was set. It allocates
 * nothing.
 */
attn_status_t attn_device_check(void* stream);

/*
 * Diagnostic of the device-side wait limit (no counterpart on the pages; it
 * exists so that the timeout path can be exercised without a fault). Enqueues
 * one small kernel that runs the attention kernels' bounded wait on an
 * mbarrier nothing completes, with a limit of spin_cycles SM clock cycles
 * (1 .. 2^31; ATTN_ERR_INVALID_ARG otherwise): the wait gives up, raises the
 * kernel's abort flag (a second waiting warp leaves through it) and sets the
 * device status word, so the next attn_device_check returns ATTN_ERR_TIMEOUT
 * and clears it. The CUDA context stays usable. Returns ATTN_OK after
 * enqueueing.
 */
attn_status_t attn_selftest_wait_timeout(int64_t spin_cycles, void* stream);

/*
 * The same diagnostic for the allocation-free entry point: the wait's status
 * lands in attn_prefill_fwd_noalloc's fixed status word, which the next
 * attn_device_check reports and clears. Allocates nothing; its first call on
 * a device does attn_prefill_fwd_noalloc's set-up (refused during capture).
 */
attn_status_t attn_selftest_wait_timeout_noalloc(int64_t spin_cycles, void* stream);

/*
 * Consistency checks of the debug build (no counterpart on the pages; a
 * development aid). The library compiled with ATTN_DEBUG (libattn_prefill_debug.so,
 * built beside the release library) checks, in the forward kernels, before
 * each operation: that every TMA copy starts inside its tensor with its
 * innermost offset 16-byte aligned and lands inside the CTA's shared memory;
 * that the tensor-memory allocation starts at lane 0, column 0 (every warp's
 * loads and stores then use its own lane quarter and fixed columns below
 * 512); that every tensor-core operand tile lies inside shared memory; and
 * that every mbarrier parity wait is sound (no more than one phase beyond the
 * awaited one has been started). A failed check raises the kernel's abort
 * flag (every role leaves as after a wait timeout) and attn_device_check
 * returns ATTN_ERR_CHECK. This call returns the number of checks the debug
 * build has run since it was loaded (synchronising the device first), or -1
 * in the release build (which runs none) or on a CUDA error.
 */
int64_t attn_debug_check_count(void);

/*
 * Number of persistent CTAs the forward kernel launches for these sizes on
 * the current device (min(#SMs, #work units)), or -1 on an argument error.
 * Host-side only apart from the SM-count query; used for reporting.
 */
int64_t attn_prefill_grid_size(int64_t B, int64_t L, int32_t n_q, int32_t n_kv,
                               int32_t d_h, int32_t causal);

/*
 * Allocation-free variant of attn_prefill_fwd. (No counterpart on the pages:
 * this is a deployment convenience of this library.)
 *
 * Same arguments, layouts, results and errors as attn_prefill_fwd, for
 * callers that cannot let a library allocate device memory: code whose
 * device memory all comes from its own pool or arena (a cudaMalloc behind
 * its back would escape its accounting and limits), or a host framework
 * that owns the allocator and forbids libraries to call it. The one piece
 * of global scratch the kernel uses (its 4-byte status word) sits in a fixed
 * 256-byte array compiled into the library instead of a cudaMalloc'd buffer;
 * every GPU that loads the library holds that array until process exit. This
 * kernel's scratch does not grow with the problem size, so every size
 * attn_prefill_fwd accepts fits (a build whose scratch exceeded the 256 bytes
 * would fail to compile).
 *
 * The first call on a device does a one-time set-up on that device (it
 * looks up the array's device address and sets the kernels' shared-memory
 * limit, without allocating); made while `stream` is being captured, that
 * first call returns ATTN_ERR_UNSUPPORTED and sets up nothing, so make it
 * before any stream capture. The status word is zero when the library is
 * loaded; a wait that runs past its limit sets a bit in it, and
 * attn_device_check reports it (ATTN_ERR_TIMEOUT, outputs of that launch
 * undefined) and clears it, as for the allocating entry points. All calls
 * share the one array: calls that overlap on the GPU (different streams, no
 * ordering between them) race on it, and a timeout is then not tied to one
 * call.
 */
attn_status_t attn_prefill_fwd_noalloc(const void* q, const void* k, const void* v,
                                       void* o, float* lse,
                                       int64_t B, int64_t L, int32_t n_q, int32_t n_kv,
                                       int32_t d_h, int32_t causal, float scale,
                                       void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_PREFILL_H */
