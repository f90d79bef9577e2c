/*
 * fa_diag.h -- tuning and self-check entry points of the exact-attention
 * library (same shared library as fa.h).  They exist so that tests and the
 * benchmark can exercise the method's individual claims on the GPU; a normal
 * caller only needs fa.h.
 */
#ifndef FA_GB300_FA_DIAG_H
#define FA_GB300_FA_DIAG_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Forward-pass knobs (fa_fwd uses the defaults).
 *   rescale_threshold  Lazy rescaling: the running output of a row is
 *                      rescaled only when the row maximum grows by more than
 *                      this many log2 units; 8.0 is the method's value
 *                      ("FlashAttention-4: Algorithm and Kernel Pipelining
 *                      Co-Design ...", bullet "Lazy rescaling").  0.0 gives
 *                      the classic eager online softmax.  Must be in [0, 16]:
 *                      larger values let unnormalised weights overflow.
 *   emu_per_16         How many of every 16 softmax exponentials are computed
 *                      by the FMA-unit polynomial instead of the hardware
 *                      exponential (same page, bullet "Software
 *                      exponentials", which uses 10-25%): 0, 2, 3 or 4.
 *                      Negative selects the library default.
 *   split_p            1: the weights P of each 128-key block are handed to
 *                      the tensor cores in two halves of 64 keys, each on its
 *                      own signal, so the product with V over the first half
 *                      starts while the second half is still being computed
 *                      ("FlashAttention-4: matrix throughput bottlenecks",
 *                      lecompute.fr, section "Keep tiles moving without
 *                      overwriting live data"); 0: one signal once all of P
 *                      is written.  Negative selects the library default.
 *   kv_stages          Depth of the K/V ring in shared memory: 2 .. 4 for
 *                      D = 128, 2 .. 10 for D = 64.  0 or negative selects
 *                      the library default.
 *   head_group         Dense layout under a causal mask: the work units
 *                      (pairs of 128-row query tiles) run longest first
 *                      ("FlashAttention-4: Algorithm and Kernel Pipelining
 *                      Co-Design ...", the paragraph on longest-first
 *                      scheduling) within groups of this many (batch, head)
 *                      pairs, group after group; B * Hq orders all heads
 *                      together.  0 or negative selects the library default.
 */
typedef struct {
  float rescale_threshold;
  int emu_per_16;
  int split_p;
  int kv_stages;
  int head_group;
} fa_fwd_tuning;

/* The defaults fa_fwd() uses.  emu_per_16, split_p, kv_stages and
 * head_group are -1 there: the library picks them per configuration (head
 * dimension, causal mask, sequence length) from a table of measured
 * choices. */
FA_API fa_fwd_tuning fa_fwd_default_tuning(void);

/* fa_fwd() with explicit knobs; `t` may be NULL for the defaults. */
FA_API fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                           int Hkv, int Sq, int Sk, int D, int causal, float scale, const int* cu_seqlens,
                           const fa_fwd_tuning* t, fa_stream_t stream);

/*
 * Backward-pass knobs (fa_bwd uses the defaults).
 *   paired  1: the main kernel runs on two-CTA clusters and issues every
 *           product as a paired (cta_group::2) tcgen05 MMA over two adjacent
 *           key blocks ("FlashAttention-4: Algorithm and Kernel Pipelining
 *           Co-Design ...", bullet "Paired-CTA backward pass"): each CTA
 *           reads only half of every B operand from shared memory and the
 *           pair adds each dQ element once instead of twice.  0: one CTA per
 *           key block, every product on one SM.  Negative selects the
 *           default, 0: on GB300 the unpaired kernel is faster, because the
 *           paired dQ product needs the two CTAs to exchange dS^T through
 *           distributed shared memory (thousands of cycles of latency that
 *           the fully used tensor memory leaves no room to hide) and runs
 *           at 64 rows per SM.
 * The other knobs apply to the unpaired kernel (head_group also orders the
 * paired kernel's units, pairs of key blocks); negative selects the
 * default, which depends on the call (layout, mask, deterministic mode).
 *   schedule        dense layout: 0: CTA c of the persistent grid takes
 *                   work units c, c + grid, ...; 1: each CTA claims its
 *                   next unit from a counter in the workspace (packed
 *                   layouts always claim).
 *   head_group      the unit order visits the key blocks of head_group
 *                   (batch, kv head) pairs -- packed layout: (sequence, kv
 *                   head) pairs, sorted by length, longest first -- block
 *                   by block (block 0 of each pair, then block 1, ...),
 *                   group after group; 1 is head-major, a value >= B * Hkv
 *                   key-block-major.  Under a causal mask block 0 is the
 *                   longest, so this is the longest-first order of
 *                   "FlashAttention-4 ..." (the paragraph on longest-first
 *                   scheduling), per group.
 *   reverse_blocks  1: a unit visits its query blocks last to first.
 *   scores_first    1: the next step's S^T product is issued before the
 *                   MMA warp waits for the dQ read-out of its TMEM buffer;
 *                   0: after.
 *   split_dq        1: the backward runs as two main kernels: one per key
 *                   block accumulating dK and dV (no dQ product), one per
 *                   128-row query tile accumulating dQ over the key blocks
 *                   in order inside tensor memory and writing it directly;
 *                   no FP32 dQ accumulator, no atomics, and the same bits on
 *                   every run.  0: one main kernel adds dQ partial sums into
 *                   the FP32 accumulator (in deterministic mode in ticket
 *                   order).  Default: 1 in deterministic mode (measured
 *                   faster for dense and packed layouts), 0 otherwise.  The
 *                   paired kernel ignores it.
 * FA_ERR_INVALID_ARG for a value out of range (paired, schedule,
 * reverse_blocks, scores_first or split_dq > 1, head_group 0).
 */
typedef struct {
  int paired;
  int schedule;
  int head_group;
  int reverse_blocks;
  int scores_first;
  int split_dq;
} fa_bwd_tuning;

/* The defaults fa_bwd() uses: paired 0, every other knob -1 (chosen per
 * call). */
FA_API fa_bwd_tuning fa_bwd_default_tuning(void);

/* fa_bwd() with explicit knobs; `t` may be NULL for the defaults.  Same
 * arguments, workspace and errors as fa_bwd(), plus FA_ERR_INVALID_ARG for a
 * knob out of range. */
/* The paired kernel covers the dense layout at D = 128; paired = 1 with a
 * packed layout or D = 64 returns FA_ERR_UNSUPPORTED. */
FA_API fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk,
                           int D, int causal, float scale, const int* cu_seqlens, int deterministic,
                           void* workspace, size_t workspace_bytes, const fa_bwd_tuning* t, fa_stream_t stream);

/*
 * Evaluates 2^x for n FP32 inputs both ways the softmax can: y_emu with the
 * FMA-unit polynomial (split x into floor and fraction, cubic on the
 * fraction, add the integer to the exponent bits), y_hw with the hardware
 * exponential instruction.  All pointers are device memory.
 */
FA_API fa_status fa_diag_exp2(const float* x, float* y_emu, float* y_hw, long long n, fa_stream_t stream);

/*
 * Launches one thread block that waits on a pipeline barrier nothing will
 * ever complete, with a time bound of `limit_ns`.  The wait gives up, the
 * block exits cleanly, and the next fa_get_device_error() returns
 * FA_ERR_TIMEOUT.  Used to test the bounded-wait path without hanging the GPU.
 */
FA_API fa_status fa_diag_wait_timeout(unsigned long long limit_ns, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_DIAG_H */
