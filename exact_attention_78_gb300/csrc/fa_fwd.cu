// Forward pass of exact attention on sm_103a: one persistent, warp-specialised
// kernel per call.
//
// Method (FlashAttention-4 pages):
//   * tiles of 128 query rows and 128 keys; online softmax; the score matrix
//     lives only in tensor memory ("FlashAttention-4: Algorithm and Kernel
//     Pipelining Co-Design for Asymmetric Hardware Scaling", fdeinterviews.com
//     summary, opening paragraph);
//   * roles: a load warp (TMA into an mbarrier ring), an MMA warp issuing
//     tcgen05 MMAs into TMEM, softmax warpgroups, and a separate correction
//     warpgroup that rescales the output and runs the epilogue (same page,
//     bullet "Pipeline for asynchronous tensor cores"; "FlashAttention-4:
//     matrix throughput bottlenecks", lecompute.fr, section "Keep tiles moving
//     without overwriting live data");
//   * two query tiles per work unit in ping-pong: while one tile's softmax
//     runs, the tensor cores work on the other tile (same bullet);
//   * part of the exponentials on the FMA units by a cubic polynomial with
//     exponent-bit insertion, the rest on the hardware unit (bullet "Software
//     exponentials");
//   * lazy rescaling: the running output is rescaled only when the row
//     maximum grows by more than the threshold (8 log2 units), with the final
//     division by the row sum taken at the same, possibly stale, maximum
//     (bullet "Lazy rescaling");
//   * longest-processing-time-first order of work units for causal masks and
//     packed variable lengths (paragraph after the bullets).
//
// Thread layout (512 threads, 16 warps, one CTA per SM):
//   warps 0-3   softmax of query tile 0    (192 registers each)
//   warps 4-7   softmax of query tile 1    (192)
//   warps 8-11  correction + epilogue      (80)
//   warp  12    TMA producer (one lane)    (48)
//   warp  13    TMEM owner + MMA issuer    (48; converged warp, one elected lane issues)
//   warps 14-15 idle                       (48)
// Register budget: 2*128*192 + 128*80 + 128*48 = 65,536 = 512 threads x 128.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)    S of tile 0 (FP32); P of tile 0 (BF16 pairs) in its first 64
//   [128,256)  S / P of tile 1
//   [256,256+D)     O of tile 0 (FP32)
//   [256+D,256+2D)  O of tile 1
//
// Shared memory: Q of both tiles, a ring of K/V tiles (each 128 x D BF16 in
// 64-column chunks with 128-byte swizzle, as TMA writes them and tcgen05
// reads them), the barriers, per-row statistics handed from the softmax to the
// correction warpgroup, and the packed-length schedule tables.
#include <cuda_runtime.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"
#include "q_sched.cuh"
#include "softmax_math.cuh"

namespace fa {
namespace fwd {

__device__ DeviceError g_err;

constexpr int kThreads = 512;
constexpr int kBM = 128;      // query rows per tile
constexpr int kBN = 128;      // keys per block
constexpr int kPairRows = qs::kPairRows;
using qs::PackedSched;

// Failure sites recorded with FA_ERR_TIMEOUT.
enum Site { kSiteSoftmaxS = 1, kSiteCorrP, kSiteCorrO, kSiteMmaQ, kSiteMmaKV, kSiteMmaO, kSiteProdQ, kSiteProdKV };

template <int D, bool VARLEN>
struct Layout {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kBM * D * 2;     // 128 rows x D BF16
  static constexpr int kChunkBytes = kBM * 128;      // 128 rows x 64 BF16
  // K/V ring depth: chosen per call (FwdParams::stages), at most this many
  static constexpr int kMaxStages = (D == 128) ? 4 : 10;
  static constexpr int kQ = 0;
  static constexpr int kBars = kQ + 2 * kTileBytes;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_lo[2], p_hi[2], o_ready[2], o_full[2]
  static constexpr int kNumBars = 2 + 2 * kMaxStages + 10;
  static constexpr int kMisc = kBars + kNumBars * 8;   // tmem slot, abort, warp flags[8]
  static constexpr int kStats = kMisc + 64;            // scale/l/m/lr: 4 x [2][128] floats
  static constexpr int kSched = kStats + 4 * 2 * kBM * 4;
  // packed schedule tables (qs::PackedSched)
  static constexpr int kSchedBytes = VARLEN ? qs::kSchedBytes : 0;
  // the K/V ring last, 1024-byte aligned (whole 128-byte swizzle atoms)
  static constexpr int kKV = (kSched + kSchedBytes + 1023) / 1024 * 1024;
  static constexpr int dynamic_bytes(int stages) { return kKV + stages * kTileBytes + kSmemAlignSlack; }
  static constexpr int kMaxDynamic = kKV + kMaxStages * kTileBytes + kSmemAlignSlack;
  static_assert(kMaxDynamic <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// One work unit: a pair of 128-row query tiles of one (sequence, head), and
// the key blocks each tile visits.
struct Unit : qs::QUnit {
  int nt[2];      // KV blocks each query tile sees (0: no valid row, or no visible key)
  int n;          // KV blocks to load: max(nt[0], nt[1])
};

// KV blocks the query tile starting at row `row0` needs: 0 when the tile has
// no valid row; under the causal mask up to the block holding the last key
// its last valid row sees (row r sees keys <= r + (seq_k - seq_q)).  Tile 0 of
// a causal pair skips the block that only tile 1 sees.
template <bool CAUSAL>
__device__ __forceinline__ int tile_kv_blocks(int row0, int seq_q, int seq_k) {
  if (row0 >= seq_q) return 0;
  int kv_end = seq_k;
  if (CAUSAL) {
    const int last = min(row0 + kBM, seq_q) - 1;
    kv_end = min(seq_k, last + 1 + (seq_k - seq_q));
  }
  return kv_end <= 0 ? 0 : (kv_end + kBN - 1) / kBN;
}

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Unit decode_unit(int u, const FwdParams& p, const PackedSched& ps) {
  Unit w;
  static_cast<qs::QUnit&>(w) = qs::decode_pair_unit<CAUSAL, VARLEN>(u, p, ps);
  w.nt[0] = tile_kv_blocks<CAUSAL>(w.pair * kPairRows, w.seq_q, w.seq_k);
  w.nt[1] = tile_kv_blocks<CAUSAL>(w.pair * kPairRows + kBM, w.seq_q, w.seq_k);
  w.n = max(w.nt[0], w.nt[1]);
  return w;
}

// Position in the K/V ring: stage index and the parity of its barriers'
// current phase, advanced without a division by the (run-time) ring depth.
struct RingPos {
  int stage;
  uint32_t phase;
};
FA_DEV RingPos ring_next(RingPos r, int stages) {
  return (r.stage + 1 == stages) ? RingPos{0, r.phase ^ 1u} : RingPos{r.stage + 1, r.phase};
}

// Shared-memory handles.  Barriers and the abort flag are addressed through
// 32-bit shared-window addresses to keep the issue warps' register use low.
template <int D, bool VARLEN>
struct Shared {
  using L = Layout<D, VARLEN>;
  uint8_t* base;    // aligned dynamic shared memory (generic pointer)
  uint32_t sbase;   // same, shared-window address
  FA_DEV uint32_t bar(int i) const { return sbase + L::kBars + 8 * i; }
  FA_DEV uint32_t q_full() const { return bar(0); }
  FA_DEV uint32_t q_empty() const { return bar(1); }
  FA_DEV uint32_t kv_full(int s) const { return bar(2 + s); }
  FA_DEV uint32_t kv_empty(int s) const { return bar(2 + L::kMaxStages + s); }
  FA_DEV uint32_t s_full(int t) const { return bar(2 + 2 * L::kMaxStages + t); }
  // P of tile t written: keys 0-63 (p_lo) and keys 64-127 (p_hi); one
  // arrival per softmax thread
  FA_DEV uint32_t p_lo(int t) const { return bar(4 + 2 * L::kMaxStages + t); }
  FA_DEV uint32_t p_hi(int t) const { return bar(6 + 2 * L::kMaxStages + t); }
  FA_DEV uint32_t o_ready(int t) const { return bar(8 + 2 * L::kMaxStages + t); }
  FA_DEV uint32_t o_full(int t) const { return bar(10 + 2 * L::kMaxStages + t); }
  FA_DEV uint32_t abort() const { return sbase + L::kMisc + 4; }
  FA_DEV uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + L::kMisc); }
  FA_DEV int* warp_flag() const { return reinterpret_cast<int*>(base + L::kMisc + 8); }   // [2][4]
  FA_DEV float* st_scale() const { return reinterpret_cast<float*>(base + L::kStats); }   // [2][128]
  FA_DEV float* st_l() const { return st_scale() + 2 * kBM; }                             // [2][128]
  FA_DEV float* st_m() const { return st_l() + 2 * kBM; }                                 // [2][128]
  FA_DEV float* st_lr() const { return st_m() + 2 * kBM; }                                // [2][128]
};

// ------------------------------------------------------------------ roles --

// Softmax warpgroup of query tile t: one thread per row of the tile.
template <int D, bool CAUSAL, bool VARLEN, int EMU>
__device__ void softmax_role(const int t, const Shared<D, VARLEN>& sh, const uint32_t tmem, const FwdParams& p,
                             const PackedSched& ps, const int total_units) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wq = warp & 3;
  const int r_in_tile = wq * 32 + lane;
  const uint32_t tm_s = tmem + (uint32_t(wq * 32) << 16) + uint32_t(t * kBN);
  const float sl2 = p.scale_log2;
  uint32_t sit = 0;
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const Unit w = decode_unit<CAUSAL, VARLEN>(u, p, ps);
    const int nt = t ? w.nt[1] : w.nt[0];   // (no dynamic index into the struct's array)
    if (nt == 0) continue;
    const int tile_row0 = w.pair * kPairRows + t * kBM;
    const int row = tile_row0 + r_in_tile;
    const int diag = w.seq_k - w.seq_q;
    float m_run = -INFINITY, l_run = 0.0f, lr_run = 0.0f;
    for (int j = 0; j < nt; ++j, ++sit) {
      if (!mbar_wait_bounded(sh.s_full(t), sit & 1, sh.abort(), &g_err, kSiteSoftmaxS, p.wait_limit_ns)) return;
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tm_s + c * 32, r[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_fence(r[c]);

      const int kv0 = j * kBN;
      const bool need_mask = (kv0 + kBN > w.seq_k) || (CAUSAL && kv0 + kBN - 1 > tile_row0 + diag);
      if (need_mask) {
        int lim = w.seq_k - kv0;                       // columns >= lim are masked
        if (CAUSAL) lim = min(lim, row + diag - kv0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) r[c / 32][c % 32] = __float_as_uint(-INFINITY);
      }
      // row maximum of the raw scores (scale > 0), with 3-input max
      float mx[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float m = __uint_as_float(r[g][0]);
#pragma unroll
        for (int c = 1; c < 31; c += 2) m = max3(m, __uint_as_float(r[g][c]), __uint_as_float(r[g][c + 1]));
        mx[g] = fmaxf(m, __uint_as_float(r[g][31]));
      }
      const float m_blk = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
      // lazy rescaling: move the running maximum only when it grows by more
      // than the threshold; otherwise keep the stale one (weights <= 2^thr)
      float factor = 1.0f;
      bool rescaled = false;
      if (j == 0) {
        m_run = m_blk;
      } else if (m_blk - m_run > p.thr) {   // false for m_blk = -inf
        factor = ex2_mufu(m_run - m_blk);    // 0 when m_run = -inf
        m_run = m_blk;
        rescaled = true;
      }
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      // Two row sums: of the FP32 weights (for the log-sum-exp) and of the
      // BF16-rounded weights the PV product actually multiplies V by (for the
      // final division, so the weights used sum to one; under a stale maximum
      // the largest weight is not 1 and not exact in BF16).  Pairs of columns
      // go through packed FP32x2 instructions.
      const uint64_t sl2x2 = pk2(sl2, sl2), negm2 = pk2(-m_use, -m_use);
      uint64_t se2[4] = {0ull, 0ull, 0ull, 0ull}, sr2[4] = {0ull, 0ull, 0ull, 0ull};
      // P in two halves of 64 keys, each as BF16 pairs over 32 TMEM columns
      // (the first 64 columns of S).  With split_p the first half is
      // signalled on its own, so the PV product over keys 0-63 may start
      // while the exponentials of keys 64-127 are still being computed
      // ("FlashAttention-4: matrix throughput bottlenecks", section "Keep
      // tiles moving without overwriting live data": an initial portion of
      // the coefficients is announced before the rest, which is protected by
      // its own synchronisation).
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 64 * half; c < 64 * half + 64; c += 2) {
          const uint64_t x2 = fma2(pk2(__uint_as_float(r[c / 32][c % 32]), __uint_as_float(r[c / 32][c % 32 + 1])),
                                   sl2x2, negm2);
          float x0, x1, e0, e1;
          up2(x2, x0, x1);
          exp2_pair<EMU>(x0, x1, c, e0, e1);
          const uint32_t pp = pack_bf16x2(e0, e1);
          pk[(c / 2) % 32] = pp;
          se2[(c / 2) & 3] = add2(se2[(c / 2) & 3], pk2(e0, e1));
          sr2[(c / 2) & 3] = add2(sr2[(c / 2) & 3], pk2(__uint_as_float(pp << 16), __uint_as_float(pp & 0xFFFF0000u)));
        }
        tmem_st32(tm_s + 32 * half, pk);
        if (half == 0) {
          // the rescale factor goes to the correction warpgroup with the
          // first half of P, so that it may act as soon as that is signalled
          sh.st_scale()[t * kBM + r_in_tile] = factor;
          const unsigned any = __any_sync(0xffffffffu, rescaled);
          if (lane == 0) sh.warp_flag()[t * 4 + wq] = any ? 1 : 0;
          if (p.split_p) {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(sh.p_lo(t));
          }
        }
      }
      float a0, a1, b0, b1;
      up2(add2(add2(se2[0], se2[1]), add2(se2[2], se2[3])), a0, a1);
      up2(add2(add2(sr2[0], sr2[1]), add2(sr2[2], sr2[3])), b0, b1);
      l_run = l_run * factor + (a0 + a1);
      lr_run = lr_run * factor + (b0 + b1);
      tmem_st_wait();
      if (j == nt - 1) {
        sh.st_l()[t * kBM + r_in_tile] = l_run;
        sh.st_lr()[t * kBM + r_in_tile] = lr_run;
        sh.st_m()[t * kBM + r_in_tile] = m_run;
      }
      tc_fence_before();
      if (!p.split_p) mbar_arrive(sh.p_lo(t));
      mbar_arrive(sh.p_hi(t));
    }
  }
}

// Correction warpgroup: rescales O rows in TMEM when the softmax moved a
// row's maximum, and runs the epilogue (O / l in BF16, LSE).
template <int D, bool CAUSAL, bool VARLEN>
__device__ void correction_role(const Shared<D, VARLEN>& sh, const uint32_t tmem, const FwdParams& p,
                                const PackedSched& ps, const int total_units) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wq = warp & 3;
  const int r_in_tile = wq * 32 + lane;
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const int total_tok = VARLEN ? ps.header[2] : p.B * p.Sq;
  __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(p.o);
  // phase counters per tile: a tile takes part only in the blocks it sees
  uint32_t sit[2] = {0u, 0u}, uit[2] = {0u, 0u};
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const Unit w = decode_unit<CAUSAL, VARLEN>(u, p, ps);
    float fin_l[2] = {0.0f, 0.0f}, fin_lr[2] = {0.0f, 0.0f}, fin_m[2] = {-INFINITY, -INFINITY};
    for (int j = 0; j < w.n; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= w.nt[t]) continue;
        const uint32_t ph = sit[t] & 1;
        ++sit[t];
        if (!mbar_wait_bounded(sh.p_lo(t), ph, sh.abort(), &g_err, kSiteCorrP, p.wait_limit_ns)) return;
        tc_fence_after();
        if (j > 0 && sh.warp_flag()[t * 4 + wq]) {
          const float f = sh.st_scale()[t * kBM + r_in_tile];
          const uint32_t tm_o = tmem + lane_off + uint32_t(256 + t * D);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tm_o + c * 32, r);
            tmem_ld_wait();
            tmem_ld_fence(r);
            const uint64_t f2 = pk2(f, f);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float y0, y1;
              up2(mul2(pk2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), f2), y0, y1);
              r[i] = __float_as_uint(y0);
              r[i + 1] = __float_as_uint(y1);
            }
            tmem_st32(tm_o + c * 32, r);
          }
          tmem_st_wait();
        }
        // The row statistics of the tile are written with the second half
        // of P of its last block: wait for it and take them into registers
        // before O is released (after that, the next unit's softmax may
        // overwrite them; and waiting before o_ready keeps this barrier
        // from running a phase ahead of the wait).
        if (j == w.nt[t] - 1) {
          if (!mbar_wait_bounded(sh.p_hi(t), ph, sh.abort(), &g_err, kSiteCorrP, p.wait_limit_ns)) return;
          fin_l[t] = sh.st_l()[t * kBM + r_in_tile];
          fin_lr[t] = sh.st_lr()[t * kBM + r_in_tile];
          fin_m[t] = sh.st_m()[t * kBM + r_in_tile];
        }
        tc_fence_before();
        mbar_arrive(sh.o_ready(t));
      }
    }
    // epilogue: O / l in BF16, LSE in natural log (a tile that sees no key
    // writes O = 0 and LSE = -inf for its valid rows)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int row = w.pair * kPairRows + t * kBM + r_in_tile;
      const bool valid = row < w.seq_q;
      const bool has = w.nt[t] > 0;
      const float l = fin_l[t], lr = fin_lr[t], m = fin_m[t];
      if (has) {
        if (!mbar_wait_bounded(sh.o_full(t), uit[t] & 1, sh.abort(), &g_err, kSiteCorrO, p.wait_limit_ns)) return;
        ++uit[t];
        tc_fence_after();
      }
      const float inv = (lr > 0.0f) ? 1.0f / lr : 0.0f;
      const size_t tok = size_t(w.q_tok0) + size_t(row);
      uint4* dst = reinterpret_cast<uint4*>(O + (tok * p.Hq + w.h) * D);
      const uint32_t tm_o = tmem + lane_off + uint32_t(256 + t * D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (has) {
          tmem_ld32(tm_o + c * 32, r);
          tmem_ld_wait();
          tmem_ld_fence(r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (valid) {
          // 32 columns of this row: 64 contiguous bytes, as two 32-byte
          // stores (whole L2 sectors) when O allows it, else four 16-byte
          // ones.  Each store instruction of a warp touches 32 rows, so their
          // number sets the epilogue's length, which the next unit's first
          // PV product waits for (clock64 probe, dense S = 1024: the two
          // tiles' epilogue 6,700 -> 4,900 cycles; forward +1% to +4%).
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
          if (p.o_st32) {
            st_global_v8(dst + c * 4, pk);
            st_global_v8(dst + c * 4 + 2, pk + 8);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[c * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      if (valid) {
        const float lse = (l > 0.0f) ? (m + log2f(l)) * 0.693147180559945309f : -INFINITY;
        const size_t li = VARLEN ? size_t(w.h) * total_tok + tok
                                 : (size_t(w.b) * p.Hq + w.h) * p.Sq + size_t(row);
        p.lse[li] = lse;
      }
      if (has) tc_fence_before();
    }
  }
}

// Unrolled K steps of S = Q K^T (both operands K-major, 128-byte swizzle): step
// kk reads 64-element chunk kk/4 at byte offset 32*(kk%4) inside its rows.
template <int D, int CHUNK, int KK>
FA_DEV void s_steps(uint32_t d_tmem, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi, uint32_t idesc) {
  if constexpr (KK < D / 16) {
    constexpr uint32_t off = ((KK >> 2) * CHUNK + (KK & 3) * 32) >> 4;
    mma_ss_w<off, off>(d_tmem, alo, ahi, blo, bhi, idesc, KK > 0 ? 1u : 0u);
    s_steps<D, CHUNK, KK + 1>(d_tmem, alo, ahi, blo, bhi, idesc);
  }
}
// Unrolled K steps of O += P V: step kk takes TMEM columns 8*kk.. of P and
// key rows 16*kk.. of V (2048 bytes = 128 descriptor units further).
template <int KK, int KEND>
FA_DEV void pv_steps(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc, uint32_t acc) {
  if constexpr (KK < KEND) {
    mma_ts_w<KK * 8, KK * 128>(d_tmem, a_tmem, blo, bhi, idesc, KK > 0 ? 1u : acc);
    pv_steps<KK + 1, KEND>(d_tmem, a_tmem, blo, bhi, idesc, acc);
  }
}

// MMA issuer (one converged warp; an elected lane issues).  Issue order per unit, with tiles a = 0, b = 1:
//   S_a(0) S_b(0) | PV_a(0) S_a(1) PV_b(0) S_b(1) | PV_a(1) S_a(2) ... PV_b(n-1)
// so that while the softmax of one tile runs, the tensor cores compute the
// other tile's products.  S_t(j+1) overwrites the TMEM columns holding P_t(j)
// only after PV_t(j) was issued; tcgen05 MMAs of one thread run in order.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void mma_role(const Shared<D, VARLEN>& sh, const uint32_t tmem, const FwdParams& p,
                         const PackedSched& ps, const int total_units) {
  using L = Layout<D, VARLEN>;
  constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false, false);
  constexpr uint32_t kIdPV = idesc_bf16_f32(kBM, D, false, true);
  const uint32_t q_base = sh.sbase + L::kQ;
  const uint32_t kv_base = sh.sbase + L::kKV;
  uint32_t uit = 0;
  uint32_t sit[2] = {0u, 0u};   // phase counters per tile
  RingPos kv{0, 0u};            // next K/V tile to consume

  // S_t = Q_t K^T : M = 128 rows, N = 128 keys, K = D in steps of 16.  The
  // descriptors of the 16-wide K steps differ from the first only in the
  // start-address field, by compile-time offsets.
  auto issue_s = [&](int t, int stage) {
    const uint64_t da = sdesc_sw128(q_base + t * L::kTileBytes, 16, 1024);
    const uint64_t db = sdesc_sw128(kv_base + stage * L::kTileBytes, 16, 1024);
    s_steps<D, L::kChunkBytes, 0>(tmem + t * kBN, desc_lo(da), desc_hi(da), desc_lo(db), desc_hi(db), kIdS);
  };
  // O_t (+)= P_t V : M = 128 rows, N = D, K = 128 keys in steps of 16;
  // P from TMEM (8 columns per 16 keys), V MN-major (64-wide D chunks;
  // 16 keys = 16 rows of 128 B = 2048 B further into the V tile)
  // Keys 0-63 once the correction warpgroup has released O (it has seen
  // the first half of P), keys 64-127 once the second half is signalled.
  // Without split_p the correction warpgroup released O only after all of
  // P was signalled, so the second half needs no wait of its own.
  auto issue_pv = [&](int t, int stage, bool acc, uint32_t ph) -> bool {
    const uint64_t db = sdesc_sw128(kv_base + stage * L::kTileBytes, L::kChunkBytes, 1024);
    pv_steps<0, 4>(tmem + 256 + t * D, tmem + t * kBN, desc_lo(db), desc_hi(db), kIdPV, acc ? 1u : 0u);
    if (p.split_p) {
      if (!mbar_wait_bounded(sh.p_hi(t), ph, sh.abort(), &g_err, kSiteMmaO, p.wait_limit_ns)) return false;
      tc_fence_after();
    }
    pv_steps<4, 8>(tmem + 256 + t * D, tmem + t * kBN, desc_lo(db), desc_hi(db), kIdPV, 1u);
    return true;
  };
  const int stages = p.stages;
  auto take_kv = [&]() {
    const RingPos r = kv;
    kv = ring_next(kv, stages);
    return r;
  };
  auto wait_kv = [&](RingPos r) -> bool {
    if (!mbar_wait_bounded(sh.kv_full(r.stage), r.phase, sh.abort(), &g_err, kSiteMmaKV, p.wait_limit_ns))
      return false;
    tc_fence_after();
    return true;
  };

  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const Unit w = decode_unit<CAUSAL, VARLEN>(u, p, ps);
    if (w.n == 0) continue;
    const int n0 = w.nt[0], n1 = w.nt[1];
    if (!mbar_wait_bounded(sh.q_full(), uit & 1, sh.abort(), &g_err, kSiteMmaQ, p.wait_limit_ns)) return;
    tc_fence_after();
    // prologue: S of both tiles for block 0 (a tile that sees no key is
    // skipped throughout)
    RingPos kp = take_kv();
    if (!wait_kv(kp)) return;
    if (n0 > 0) {
      issue_s(0, kp.stage);
      mma_commit_w(sh.s_full(0));
    }
    if (n1 > 0) {
      issue_s(1, kp.stage);
      mma_commit_w(sh.s_full(1));
    }
    mma_commit_w(sh.kv_empty(kp.stage));
    if (w.n == 1) mma_commit_w(sh.q_empty());
    for (int j = 0; j < w.n; ++j) {
      const RingPos vp = take_kv();
      if (!wait_kv(vp)) return;
      const bool more = j + 1 < w.n;
      bool k_ready = false;
      if (more) kp = take_kv();
      // tile 0: PV(j), then S(j+1) if it sees block j + 1
      if (j < n0) {
        const uint32_t ph = sit[0] & 1;
        ++sit[0];
        if (!mbar_wait_bounded(sh.o_ready(0), ph, sh.abort(), &g_err, kSiteMmaO, p.wait_limit_ns)) return;
        tc_fence_after();
        if (!issue_pv(0, vp.stage, j > 0, ph)) return;
        if (j + 1 < n0) {
          if (!wait_kv(kp)) return;
          k_ready = true;
          issue_s(0, kp.stage);
          mma_commit_w(sh.s_full(0));
        } else {
          mma_commit_w(sh.o_full(0));
        }
      }
      // tile 1: PV(j), then S(j+1) if it sees block j + 1
      if (j < n1) {
        const uint32_t ph = sit[1] & 1;
        ++sit[1];
        if (!mbar_wait_bounded(sh.o_ready(1), ph, sh.abort(), &g_err, kSiteMmaO, p.wait_limit_ns)) return;
        tc_fence_after();
        if (!issue_pv(1, vp.stage, j > 0, ph)) return;
        if (j + 1 == n1) mma_commit_w(sh.o_full(1));
      }
      mma_commit_w(sh.kv_empty(vp.stage));
      if (more) {
        if (j + 1 < n1) {
          if (!k_ready && !wait_kv(kp)) return;
          issue_s(1, kp.stage);
          mma_commit_w(sh.s_full(1));
        }
        mma_commit_w(sh.kv_empty(kp.stage));
        if (j + 1 == w.n - 1) mma_commit_w(sh.q_empty());
      }
    }
    ++uit;
  }
}

// TMA producer (one thread): Q of both tiles once per unit, then K_j, V_j in
// order through the stage ring.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void producer_role(const Shared<D, VARLEN>& sh, const CUtensorMap* tq, const CUtensorMap* tk,
                              const CUtensorMap* tv, const FwdParams& p, const PackedSched& ps,
                              const int total_units) {
  using L = Layout<D, VARLEN>;
  uint32_t uit = 0;
  RingPos kv{0, 0u};   // next K/V tile to fill
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const Unit w = decode_unit<CAUSAL, VARLEN>(u, p, ps);
    if (w.n == 0) continue;
    const int hk = w.h / p.group;
    if (!mbar_wait_bounded(sh.q_empty(), (uit & 1) ^ 1, sh.abort(), &g_err, kSiteProdQ, p.wait_limit_ns)) return;
    mbar_arrive_expect_tx(sh.q_full(), 2 * L::kTileBytes);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_3d(sh.sbase + L::kQ + t * L::kTileBytes + c * L::kChunkBytes, tq, sh.q_full(), c * 64, w.h,
                    w.q_tok0 + w.pair * kPairRows + t * kBM);
    for (int j = 0; j < w.n; ++j) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const int stage = kv.stage;
        if (!mbar_wait_bounded(sh.kv_empty(stage), kv.phase ^ 1u, sh.abort(), &g_err, kSiteProdKV, p.wait_limit_ns))
          return;
        mbar_arrive_expect_tx(sh.kv_full(stage), L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sh.sbase + L::kKV + stage * L::kTileBytes + c * L::kChunkBytes, which ? tv : tk,
                      sh.kv_full(stage), c * 64, hk, w.k_tok0 + j * kBN);
        kv = ring_next(kv, p.stages);
      }
    }
    ++uit;
  }
}

template <int D, bool CAUSAL, bool VARLEN, int EMU>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Layout<D, VARLEN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32;
  Shared<D, VARLEN> sh;
  sh.base = smem;
  sh.sbase = smem_u32(smem);

  if (threadIdx.x == 0) {
    mbar_init(sh.q_full(), 1);
    mbar_init(sh.q_empty(), 1);
    for (int s = 0; s < L::kMaxStages; ++s) {
      mbar_init(sh.kv_full(s), 1);
      mbar_init(sh.kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sh.s_full(t), 1);
      mbar_init(sh.p_lo(t), kBM);      // one arrival per softmax thread
      mbar_init(sh.p_hi(t), kBM);
      mbar_init(sh.o_ready(t), kBM);   // one per correction thread
      mbar_init(sh.o_full(t), 1);
    }
    st_shared(sh.abort(), 0);
    fence_barrier_init();
  }
  if (warp == 12 && (threadIdx.x % 32) == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 13) {
    tmem_alloc(sh.tmem_slot(), 512);
    tmem_relinquish();
  }
  PackedSched ps{};
  int total_units;
  if (VARLEN) {
    total_units = qs::build_packed_sched(p, ps, smem + L::kSched, &g_err);
  } else {
    total_units = qs::dense_units(p);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();

  if (warp < 8) {
    reg_alloc<192>();
    softmax_role<D, CAUSAL, VARLEN, EMU>(warp / 4, sh, tmem, p, ps, total_units);
  } else if (warp < 12) {
    reg_dealloc<80>();
    correction_role<D, CAUSAL, VARLEN>(sh, tmem, p, ps, total_units);
  } else {
    reg_dealloc<48>();
    const int lane = threadIdx.x % 32;
    if (warp == 12 && lane == 0)
      producer_role<D, CAUSAL, VARLEN>(sh, &tm_q, &tm_k, &tm_v, p, ps, total_units);
    else if (warp == 13)   // the whole warp, converged; one elected lane issues
      mma_role<D, CAUSAL, VARLEN>(sh, tmem, p, ps, total_units);
  }

  // After a give-up, let copies and MMAs already in flight land before the
  // shared and tensor memory they target are released.
  if (ld_shared_volatile(sh.abort())) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool VARLEN, int EMU>
fa_status launch_inst(const FwdLaunch& L, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      cudaStream_t stream) {
  using Lay = Layout<D, VARLEN>;
  auto kern = fwd_kernel<D, CAUSAL, VARLEN, EMU>;
  if (L.p.stages < 2 || L.p.stages > Lay::kMaxStages) return FA_ERR_INVALID_ARG;
  const fa_status st = prepare_kernel(reinterpret_cast<const void*>(kern), Lay::kMaxDynamic);
  if (st != FA_OK) return st;
  int grid = L.num_sms;
  if (!VARLEN) {
    const long long units = (long long)((L.p.Sq + kPairRows - 1) / kPairRows) * L.p.B * L.p.Hq;
    if (units < grid) grid = (int)units;
  }
  if (grid < 1) grid = 1;
  kern<<<grid, kThreads, Lay::dynamic_bytes(L.p.stages), stream>>>(tq, tk, tv, L.p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, bool CAUSAL, bool VARLEN>
fa_status launch_emu(const FwdLaunch& L, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t s) {
  switch (L.emu_per_16) {
    case 0: return launch_inst<D, CAUSAL, VARLEN, 0>(L, tq, tk, tv, s);
    case 2: return launch_inst<D, CAUSAL, VARLEN, 2>(L, tq, tk, tv, s);
    case 3: return launch_inst<D, CAUSAL, VARLEN, 3>(L, tq, tk, tv, s);
    case 4: return launch_inst<D, CAUSAL, VARLEN, 4>(L, tq, tk, tv, s);
    default: return FA_ERR_INVALID_ARG;
  }
}

template <int D>
fa_status launch_d(const FwdLaunch& L, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   cudaStream_t s) {
  const bool varlen = L.p.cu_seqlens != nullptr;
  if (L.causal)
    return varlen ? launch_emu<D, true, true>(L, tq, tk, tv, s) : launch_emu<D, true, false>(L, tq, tk, tv, s);
  return varlen ? launch_emu<D, false, true>(L, tq, tk, tv, s) : launch_emu<D, false, false>(L, tq, tk, tv, s);
}

}  // namespace fwd

fa_status launch_fwd(const FwdLaunch& L, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const int rows_q = L.p.cu_seqlens ? L.p.Sq : L.p.B * L.p.Sq;
  const int rows_k = L.p.cu_seqlens ? L.p.Sk : L.p.B * L.p.Sk;
  fa_status st;
  if ((st = make_tmap_rows_heads_d(&tq, L.q, rows_q, L.p.Hq, L.D, fwd::kBM)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&tk, L.k, rows_k, L.p.Hkv, L.D, fwd::kBN)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&tv, L.v, rows_k, L.p.Hkv, L.D, fwd::kBN)) != FA_OK) return st;
  if (L.D == 128) return fwd::launch_d<128>(L, tq, tk, tv, stream);
  if (L.D == 64) return fwd::launch_d<64>(L, tq, tk, tv, stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status fwd_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, fwd::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(fwd::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

}  // namespace fa
