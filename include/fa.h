/*
 * fa.h -- C ABI of the exact-attention library for one NVIDIA GB300 (sm_103a).
 *
 * What is computed.  Exact scaled-dot-product attention and its gradients:
 *
 *     O   = softmax(scale * Q K^T [+ causal mask]) V
 *     LSE = per-row log-sum-exp of the masked, scaled scores (natural log)
 *
 * evaluated tile by tile with an online softmax so that the score matrix never
 * reaches device memory, plus the backward pass producing dQ, dK and dV.
 * Sources: "FlashAttention-4: matrix throughput bottlenecks" (lecompute.fr),
 * section "Between the matrix products the kernel must produce weights" (the
 * definition: scores, row softmax, second product with V); "FlashAttention-4:
 * Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling"
 * (fdeinterviews.com summary), opening paragraph (tiling, online softmax, no
 * full matrix in memory), bullets "Lazy rescaling" and "Paired-CTA backward
 * pass", and the paragraph on causal masks, variable lengths and the
 * deterministic backward mode.
 *
 * Conventions shared by every call.
 *   - Element types: Q, K, V, O, dO, dQ, dK, dV are BF16; LSE is FP32.
 *   - Dense layout (cu_seqlens == NULL): Q, O, dO, dQ are [B, Sq, Hq, D];
 *     K, V, dK, dV are [B, Sk, Hkv, D]; LSE is [B, Hq, Sq].  All contiguous,
 *     D innermost.
 *   - Packed variable-length layout (cu_seqlens != NULL): sequence b owns
 *     tokens [cu_seqlens[b], cu_seqlens[b+1]) of Q, K, V, O shaped [total, H, D];
 *     LSE is [Hq, total].  cu_seqlens is an int32 DEVICE array of B + 1
 *     non-decreasing offsets with cu_seqlens[0] = 0; the same offsets apply
 *     to queries and keys.  Sq and Sk must both equal the total token count
 *     cu_seqlens[B] (the row count of the packed arrays; the host cannot read
 *     it from device memory without a synchronisation).  At most 1024
 *     sequences of at most 262,144 tokens each.  Offsets that break these
 *     rules are detected on the device: nothing is computed and
 *     fa_get_device_error() reports FA_ERR_INVALID_ARG.
 *   - Grouped-query attention: query head h reads key/value head
 *     h / (Hq / Hkv); Hq must be a multiple of Hkv.
 *   - Causal mask, bottom-right aligned: query i sees key j iff
 *     j <= i + (Sk - Sq).  A query row that sees no key gets O = 0 and
 *     LSE = -inf.
 *   - scale must be finite and > 0 (callers normally pass 1/sqrt(D)).
 *   - Head dimension D must be 64 or 128.
 *   - Every pointer is caller-owned device memory, 16-byte aligned.  The
 *     library allocates no device memory in these calls; the backward pass
 *     takes its scratch from the caller's workspace.
 *   - Calls are asynchronous on `stream`; argument errors are reported
 *     synchronously by the return value before anything is launched.  A
 *     device-side wait that exceeded its time bound is reported later by
 *     fa_get_device_error().  No C++ exception crosses this interface.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols of the shared library. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

typedef struct CUstream_st* fa_stream_t; /* the same handle as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, bad scale ... */
  FA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (D, device) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 4,      /* a device-side pipeline wait exceeded its bound */
  FA_ERR_WORKSPACE = 5     /* workspace missing, misaligned or too small */
} fa_status;

/*
 * Forward pass.  Writes O and LSE.
 *   q, k, v      device, BF16, layouts above
 *   o            device, BF16, same shape as q
 *   lse          device, FP32, [B, Hq, Sq] dense or [Hq, total] packed
 *   B, Hq, Hkv   batch (number of sequences when packed) and head counts
 *   Sq, Sk, D    sequence lengths (total tokens when packed) and head dim
 *   causal       0 or 1
 *   scale        multiplier of Q K^T
 *   cu_seqlens   device int32 [B + 1], or NULL for the dense layout
 * Returns FA_OK once the work is enqueued on `stream`.
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, int D, int causal, float scale, const int* cu_seqlens, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd() needs for this problem.
 *   Dense layout: cu_seqlens_host = NULL and total_q = 0.  The workspace holds
 *   the FP32 dQ accumulator [B, Sq, Hq, D], the per-row terms
 *   -Delta_i = -sum_d dO_id * O_id and -LSE * log2(e) (FP32 [B, Hq, Sq rounded
 *   up to a multiple of 64] each) and, when `deterministic` is set, two int32
 *   tickets per (b, h, 64-row query block).
 *   Packed layout: total_q = the packed row count (the Sq = Sk of the fa_bwd
 *   call); cu_seqlens_host is an optional HOST copy of the B + 1 offsets,
 *   checked against the layout rules when given.  The size is a bound that
 *   does not depend on the individual lengths: FP32 accumulator [total, Hq, D],
 *   row terms over each sequence's rows rounded up to 64 (Hq x (total rounded
 *   up to 64 + 64 B) each), the per-sequence offset tables, the order of the
 *   work units ((total / 128 + B) x Hkv entries of 8 bytes) and the tickets.
 * Returns 0 for arguments fa_bwd() would reject.
 */
FA_API size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, const int* cu_seqlens_host,
                                    int total_q, int deterministic);

/*
 * Backward pass of fa_fwd(), dense or packed layout.  Given the forward
 * inputs, its outputs O and LSE, and the upstream gradient dO, writes dQ, dK,
 * dV (BF16; dK/dV of a key/value head sum over its query-head group).
 *   deterministic  0: dQ partial sums are added with FP32 atomics (order may
 *                  vary run to run); 1: dQ is summed over the key blocks in
 *                  a fixed order, so repeated calls give bitwise-identical
 *                  dQ (by default a second main kernel computes each dQ
 *                  tile whole in tensor memory; fa_bwd_ex can select
 *                  ticket-ordered additions in the fused kernel instead).
 *   workspace      device, 256-byte aligned, at least
 *                  fa_bwd_workspace_size(...) bytes (for the packed layout
 *                  sized with total_q = Sq); contents on entry are ignored
 *                  and clobbered.
 * Head dimension 64 or 128, like fa_fwd().
 * Launches three kernels on `stream` (row terms, main pass, dQ conversion; in
 * deterministic mode the last is the dQ kernel), four for the packed layout (a first one checks the offsets and builds the
 * per-sequence tables).
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk,
                        int D, int causal, float scale, const int* cu_seqlens, int deterministic,
                        void* workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd() for callers that cannot allocate device memory: some programs run
 * under an allocator or serving runtime that owns every byte of the GPU and
 * forbids allocating after start-up, or call from a point where an
 * allocation would stall the device.  Arguments are those of fa_bwd() minus
 * the workspace: the scratch comes from one buffer of
 * FA_BWD_STATIC_SCRATCH_BYTES (64 MiB) compiled into the library, which every
 * GPU that loads the library holds until the process exits.  The paper has
 * no counterpart; this is an interface convenience.
 *   - Needs no more than fa_bwd_workspace_size(...) <= 64 MiB (for example
 *     B * Sq * Hq * D * 4 bytes of dQ accumulator); larger problems are
 *     rejected with FA_ERR_WORKSPACE before anything is launched.
 *   - Allocates nothing.  The first call on a device (more exactly, in each
 *     CUDA context: again after cudaDeviceReset or in a context the caller
 *     created) looks up the buffer's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream
 *     capture.
 *   - All calls share the one buffer and it keeps the last call's contents;
 *     the call clears what must start at zero itself.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on the
 *     buffer: serialise them.
 */
#define FA_BWD_STATIC_SCRATCH_BYTES (64ull << 20)
FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
                                int Sk, int D, int causal, float scale, const int* cu_seqlens, int deterministic,
                                fa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the first device-side
 * failure recorded by any kernel of this library on the current device since
 * the last call (FA_OK if none).  A pipeline wait that exceeds its bound
 * (about two seconds) makes every role of the affected thread block stop and
 * exit cleanly, records FA_ERR_TIMEOUT here and leaves the outputs undefined;
 * the CUDA context stays usable.
 */
FA_API fa_status fa_get_device_error(fa_stream_t stream);

/* Static, human-readable name of a status code. */
FA_API const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
