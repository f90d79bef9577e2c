// dQ kernel of the backward pass (sm_103a, dense and packed layouts, head
// dimension D = 64 or 128): the query-side half of the split backward that
// the deterministic mode runs.
//
// A dQ tile of 128 query rows of one (sequence, query head) is computed whole
// by one CTA, summing over the key blocks it sees in ascending order inside
// tensor memory, so the result is the same bit for bit on every run and
// needs no accumulator in global memory nor any ordering between CTAs
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", fdeinterviews.com summary, paragraph after
// the bullets: the deterministic backward mode).  Per block of 64 keys:
//     S  = Q K_j^T,  dP = dO V_j^T            (M = 128 queries, N = 64 keys)
//     P  = exp2(S * scale * log2 e - LSE2),  dS = P * (dP - Delta)
//     dQ += dS K_j                            (M = 128, N = D, K = 64 keys)
// with the score products of the next blocks issued while the elementwise
// pass of block j runs (two score buffers in tensor memory at D = 128, three
// at D = 64), and dQ written as BF16 (times scale) at the end of the tile.
// Q and dO, the A operands of every score product of the tile, are copied
// once per tile from shared into tensor memory (tcgen05.cp), so the score
// products read only K_j and V_j from shared memory: per block of 64 keys
// that is 384 operand wavefronts of 128 bytes instead of 896, under the
// shared-memory bandwidth that bounds this kernel otherwise.  Its companion,
// the main backward kernel without its dQ product, accumulates dK and dV.
//
// Thread layout (320 threads, one CTA per SM):
//   warps 0-3   elementwise for key columns 0-31 of each block, and the dQ
//               epilogue for features [0, D/2)  (thread = query row)
//   warps 4-7   the same for key columns 32-63 and features [D/2, D)
//   warp  8     TMA producer (one lane)
//   warp  9     TMEM owner + MMA issuer (converged warp, one elected lane)
//
// Tensor memory: score buffers b < kSB with S at 128 b (64 columns) and dP
// at 128 b + 64; dS as BF16 pairs over columns 0-15 and 32-47 of the S
// region (one half per warpgroup, each inside the columns it has read); dQ
// in [128 kSB, 128 kSB + D); Q and dO of the tile as BF16 pairs (row per
// lane) in the D columns after it.
//
// Shared memory: Q and dO of the next tile (TMA lands them while the current
// tile runs from its tensor-memory copy), a ring of K_j blocks (held from the
// score product to the dQ product of a block) and a ring of V_j blocks (read
// by the dP product only), barriers, and for packed layouts the
// longest-first schedule tables.
#include <cuda_runtime.h>

#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"
#include "q_sched.cuh"
#include "softmax_math.cuh"

namespace fa {
namespace bdq {

__device__ DeviceError g_err;

constexpr int kThreads = 320;
constexpr int kBM = qs::kTileRows;   // query rows per tile
constexpr int kBN = 64;              // keys per block
constexpr int kPairRows = qs::kPairRows;

enum Site { kSiteEs = 1, kSiteEpi, kSiteMmaQ, kSiteMmaKV, kSiteMmaP, kSiteMmaDq, kSiteProdQ, kSiteProdKV };

// Parameters of the dQ kernel (the fields q_sched.cuh reads, plus its own).
struct DqParams {
  const int* cu_seqlens;   // packed layout: device [B + 1]; nullptr for dense
  const int* plan;         // packed layout: padded-row prefix at plan[B + 1 ...] (written by the plan kernel)
  const float* ndelta;     // -Delta, row-term layout of the pre pass
  const float* nlse2;      // -LSE * log2(e), same layout
  void* dq;                // BF16 output, Q's layout
  int B, Hq, Hkv, Sq, Sk;  // packed: Sq = Sk = total rows
  int group;               // Hq / Hkv
  int sched_group;         // dense causal: heads per longest-first group
  int sq_pad;              // row-term floats per (batch, head) (dense) / per head (packed)
  int snake;               // deal the units boustrophedon-wise (q_sched.cuh)
  int dq_st32;             // dQ is 32-byte aligned: its rows are written with 32-byte stores
  float scale;
  float scale_log2;
  unsigned long long wait_limit_ns;
};

template <int D, bool VARLEN>
struct Layout {
  static constexpr int kTileBytes = kBM * D * 2;      // Q or dO tile: 128 rows x D BF16
  static constexpr int kQChunk = kBM * 128;           // 128 rows x 64 features
  static constexpr int kKTile = kBN * D * 2;          // K_j or V_j: 64 keys x D
  static constexpr int kKChunk = kBN * 128;           // 64 keys x 64 features (8 KB)
  static constexpr int kSB = (D == 128) ? 2 : 3;         // score buffers in tensor memory
  static constexpr int kKSt = (D == 128) ? 5 : 6;        // K ring: blocks j .. j + kSB - 1 held, the rest loading
  static constexpr int kVSt = (D == 128) ? 3 : 4;        // V ring
  static constexpr int kQ = 0;                                      // [Q | dO] of the next tile
  static constexpr int kK = kQ + 2 * kTileBytes;                    // [kKSt] K_j
  static constexpr int kV = kK + kKSt * kKTile;                     // [kVSt] V_j
  static constexpr int kBars = kV + kVSt * kKTile;
  // tensor-memory columns of dQ, Q and dO
  static constexpr uint32_t kColDQ = 128 * kSB;
  static constexpr uint32_t kColQ = kColDQ + D;
  static constexpr uint32_t kColDO = kColQ + D / 2;
  // qd_full, qd_free, qd_tfree, k_full[kKSt], k_empty[kKSt], v_full[kVSt], v_empty[kVSt],
  // s_full[kSB], p_ready[kSB], dq_full, dq_empty
  static constexpr int kNumBars = 3 + 2 * kKSt + 2 * kVSt + 2 * kSB + 2;
  static constexpr int kMisc = kBars + kNumBars * 8;                // tmem slot, abort flag
  static constexpr int kSched = kMisc + 64;
  static constexpr int kTotal = kSched + (VARLEN ? qs::kSchedBytes : 0);
  static constexpr int kDynamic = kTotal + kSmemAlignSlack;
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kBars % 1024 == 0, "tile alignment");
  static_assert(kColDO + D / 2 <= 512, "tensor memory");
  static_assert(kDynamic <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

template <int D, bool VARLEN>
struct Shared {
  using L = Layout<D, VARLEN>;
  uint8_t* base;
  uint32_t sbase;
  FA_DEV uint32_t bar(int i) const { return sbase + L::kBars + 8 * i; }
  FA_DEV uint32_t qd_full() const { return bar(0); }    // Q and dO of the next tile landed in shared memory
  FA_DEV uint32_t qd_free() const { return bar(1); }    // copied on into tensor memory: the buffer is free
  FA_DEV uint32_t qd_tfree() const { return bar(2); }   // the tile's last score products done: its copy is free
  FA_DEV uint32_t k_full(int s) const { return bar(3 + s); }
  FA_DEV uint32_t k_empty(int s) const { return bar(3 + L::kKSt + s); }
  FA_DEV uint32_t v_full(int s) const { return bar(3 + 2 * L::kKSt + s); }
  FA_DEV uint32_t v_empty(int s) const { return bar(3 + 2 * L::kKSt + L::kVSt + s); }
  static constexpr int kB2 = 3 + 2 * L::kKSt + 2 * L::kVSt;
  FA_DEV uint32_t s_full(int b) const { return bar(kB2 + b); }
  FA_DEV uint32_t p_ready(int b) const { return bar(kB2 + L::kSB + b); }   // dS of buffer b in TMEM
  FA_DEV uint32_t dq_full() const { return bar(kB2 + 2 * L::kSB); }
  FA_DEV uint32_t dq_empty() const { return bar(kB2 + 2 * L::kSB + 1); }
  FA_DEV uint32_t abort() const { return sbase + L::kMisc + 4; }
  FA_DEV uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + L::kMisc); }
  FA_DEV uint32_t q_tile() const { return sbase + L::kQ; }
  FA_DEV uint32_t do_tile() const { return sbase + L::kQ + L::kTileBytes; }
  FA_DEV uint32_t k_tile(int s) const { return sbase + L::kK + s * L::kKTile; }
  FA_DEV uint32_t v_tile(int s) const { return sbase + L::kV + s * L::kKTile; }
};

constexpr uint32_t kColBuf = 128, kColDPoff = 64;   // score buffer stride; dP within a buffer

// One query tile of a unit (a unit is a pair of tiles, see q_sched.cuh).
struct Tile {
  int row0;   // first query row of the tile inside the sequence
  int nblk;   // 64-key blocks it sees (0: no valid row, or no visible key)
};

template <bool CAUSAL>
FA_DEV Tile tile_of(const qs::QUnit& w, int t) {
  Tile x;
  x.row0 = w.pair * kPairRows + t * kBM;
  x.nblk = 0;
  if (x.row0 < w.seq_q) {
    int kv_end = w.seq_k;
    if (CAUSAL) {
      const int last = min(x.row0 + kBM, w.seq_q) - 1;
      kv_end = min(w.seq_k, last + 1 + (w.seq_k - w.seq_q));
    }
    x.nblk = kv_end <= 0 ? 0 : (kv_end + kBN - 1) / kBN;
  }
  return x;
}

// Row-term index of row `row` of the unit's sequence, head h.
template <bool VARLEN>
FA_DEV size_t row_term(const qs::QUnit& w, int row, const DqParams& p) {
  if (VARLEN) return size_t(w.h) * p.sq_pad + size_t(p.plan[p.B + 1 + w.b]) + size_t(row);
  return (size_t(w.b) * p.Hq + w.h) * p.sq_pad + size_t(row);
}

// Unrolled K steps (K = D in 16-wide steps) of S = Q K_j^T or dP = dO V_j^T:
// A (Q or dO) in tensor memory, 8 columns per step; B (K_j or V_j) K-major
// in shared memory, step kk reading 64-wide chunk kk / 4 (chunks 64 rows =
// 8 KB apart) at byte 32 (kk % 4).
template <int D, int KK>
FA_DEV void score_steps(uint32_t d, uint32_t a, uint32_t blo, uint32_t bhi, uint32_t idesc) {
  if constexpr (KK < D / 16) {
    constexpr uint32_t ob = ((KK >> 2) * (kBN * 128) + (KK & 3) * 32) >> 4;
    mma_ts_w<KK * 8, ob>(d, a, blo, bhi, idesc, KK > 0 ? 1u : 0u);
    score_steps<D, KK + 1>(d, a, blo, bhi, idesc);
  }
}
// Warp-collective copy of a 128-row x 256-bit block from shared memory
// (matrix descriptor, as for an MMA operand) into tensor memory: row i to
// lane i, 8 columns from column t + TOFF; SOFF is added to the descriptor's
// start-address field.  Copies run before the tcgen05.mma the same thread
// issues after them.
template <uint32_t TOFF, uint32_t SOFF>
FA_DEV void tmem_cp_w(uint32_t t, uint32_t s_lo, uint32_t s_hi) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 tt, sl;\n\t.reg .b64 sd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.u32 tt, %0, %3;\n\t"
      "add.u32 sl, %1, %4;\n\t"
      "mov.b64 sd, {sl, %2};\n\t"
      "@e tcgen05.cp.cta_group::1.128x256b [tt], sd;\n\t}\n" ::"r"(t),
      "r"(s_lo), "r"(s_hi), "n"(TOFF), "n"(SOFF)
      : "memory");
}
// Copies a 128-row tile (Q or dO: K-major, 64-wide chunks 128 rows = 16 KB
// apart, 128-byte swizzle) from shared into tensor memory, 16 features (8
// columns, 256 bits per row) per copy: the layout the score products read
// their A operand in (row per lane, feature pairs per column).
template <int D, int KK>
FA_DEV void copy_steps(uint32_t t, uint32_t slo, uint32_t shi) {
  if constexpr (KK < D / 16) {
    constexpr uint32_t os = ((KK >> 2) * (kBM * 128) + (KK & 3) * 32) >> 4;
    tmem_cp_w<KK * 8, os>(t, slo, shi);
    copy_steps<D, KK + 1>(t, slo, shi);
  }
}
// Unrolled K steps (64 keys in 16-wide steps) of dQ += dS K_j: A = dS in
// TMEM (8 columns per step; keys 0-31 in columns 0-15, keys 32-63 in
// columns 32-47 of the S region, as the two warpgroups write them), B = K_j
// MN-major (16 key rows = 2048 B per step).
template <int KK>
FA_DEV void dq_steps(uint32_t d, uint32_t a, uint32_t blo, uint32_t bhi, uint32_t idesc, uint32_t acc) {
  if constexpr (KK < kBN / 16) {
    constexpr uint32_t ca = KK * 8 + (KK >= 2 ? 16 : 0);
    mma_ts_w<ca, KK * 128>(d, a, blo, bhi, idesc, KK > 0 ? 1u : acc);
    dq_steps<KK + 1>(d, a, blo, bhi, idesc, acc);
  }
}

// Ring position: stage and the parity of its barriers' current phase.
struct RingPos {
  int stage;
  uint32_t phase;
};
template <int S>
FA_DEV RingPos ring_next(RingPos r) {
  return (r.stage + 1 == S) ? RingPos{0, r.phase ^ 1u} : RingPos{r.stage + 1, r.phase};
}

// TMA producer (one thread): per tile Q and dO into their buffer (once the
// previous tile's have been copied into tensor memory), then K_j, V_j
// through the rings.
template <int D, bool CAUSAL, bool VARLEN>
__device__ void producer_role(const Shared<D, VARLEN>& sh, const CUtensorMap* tq, const CUtensorMap* tdo,
                              const CUtensorMap* tk, const CUtensorMap* tv, const DqParams& p,
                              const qs::PackedSched& ps, int total_units) {
  using L = Layout<D, VARLEN>;
  uint32_t tit = 0;
  RingPos kr{0, 0u}, vr{0, 0u};
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const qs::QUnit w = qs::decode_pair_unit<CAUSAL, VARLEN>(u, p, ps);
    const int hk = w.h / p.group;
    for (int t = 0; t < 2; ++t) {
      const Tile x = tile_of<CAUSAL>(w, t);
      if (x.nblk == 0) continue;
      if (!mbar_wait_bounded(sh.qd_free(), (tit & 1) ^ 1, sh.abort(), &g_err, kSiteProdQ, p.wait_limit_ns)) return;
      mbar_arrive_expect_tx(sh.qd_full(), 2 * L::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sh.q_tile() + c * L::kQChunk, tq, sh.qd_full(), c * 64, w.h, w.q_tok0 + x.row0);
        tma_load_3d(sh.do_tile() + c * L::kQChunk, tdo, sh.qd_full(), c * 64, w.h, w.q_tok0 + x.row0);
      }
      ++tit;
      for (int j = 0; j < x.nblk; ++j) {
        const int krow = w.k_tok0 + j * kBN;
        if (!mbar_wait_bounded(sh.k_empty(kr.stage), kr.phase ^ 1u, sh.abort(), &g_err, kSiteProdKV,
                               p.wait_limit_ns))
          return;
        mbar_arrive_expect_tx(sh.k_full(kr.stage), L::kKTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sh.k_tile(kr.stage) + c * L::kKChunk, tk, sh.k_full(kr.stage), c * 64, hk, krow);
        kr = ring_next<L::kKSt>(kr);
        if (!mbar_wait_bounded(sh.v_empty(vr.stage), vr.phase ^ 1u, sh.abort(), &g_err, kSiteProdKV,
                               p.wait_limit_ns))
          return;
        mbar_arrive_expect_tx(sh.v_full(vr.stage), L::kKTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sh.v_tile(vr.stage) + c * L::kKChunk, tv, sh.v_full(vr.stage), c * 64, hk, krow);
        vr = ring_next<L::kVSt>(vr);
      }
    }
  }
}

// MMA issuer (whole warp, converged; an elected lane issues).
template <int D, bool CAUSAL, bool VARLEN>
__device__ void mma_role(const Shared<D, VARLEN>& sh, const uint32_t tmem, const DqParams& p,
                         const qs::PackedSched& ps, int total_units) {
  using L = Layout<D, VARLEN>;
  constexpr int kSB = L::kSB;
  constexpr uint32_t kColDQ = L::kColDQ;
  constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, false, false);   // S, dP: 128 queries x 64 keys
  constexpr uint32_t kIdQ = idesc_bf16_f32(kBM, D, false, true);      // dQ: A in TMEM, B MN-major
  uint32_t tit = 0, sit = 0;
  RingPos kr{0, 0u}, vr{0, 0u};
  // every step takes the next K block of the ring, so step t's block sits
  // in K stage t mod kKSt
  auto wait = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    if (!mbar_wait_bounded(bar, parity, sh.abort(), &g_err, site, p.wait_limit_ns)) return false;
    tc_fence_after();
    return true;
  };
  // S and dP of global step t (the next K and V blocks of the rings) into
  // buffer t mod kSB; V_j is released as soon as its one product is issued
  auto scores = [&](uint32_t t) -> bool {
    if (!wait(sh.k_full(kr.stage), kr.phase, kSiteMmaKV)) return false;
    const int buf = t % kSB;
    const uint64_t dk = sdesc_sw128(sh.k_tile(kr.stage), 16, 1024);
    score_steps<D, 0>(tmem + kColBuf * buf, tmem + L::kColQ, desc_lo(dk), desc_hi(dk), kIdS);
    kr = ring_next<L::kKSt>(kr);
    if (!wait(sh.v_full(vr.stage), vr.phase, kSiteMmaKV)) return false;
    const uint64_t dv = sdesc_sw128(sh.v_tile(vr.stage), 16, 1024);
    score_steps<D, 0>(tmem + kColBuf * buf + kColDPoff, tmem + L::kColDO, desc_lo(dv), desc_hi(dv), kIdS);
    mma_commit_w(sh.v_empty(vr.stage));
    vr = ring_next<L::kVSt>(vr);
    mma_commit_w(sh.s_full(buf));
    return true;
  };
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const qs::QUnit w = qs::decode_pair_unit<CAUSAL, VARLEN>(u, p, ps);
    for (int t = 0; t < 2; ++t) {
      const Tile x = tile_of<CAUSAL>(w, t);
      if (x.nblk == 0) continue;
      // Q and dO of the tile into tensor memory, once they have landed and
      // the previous tile's score products (the readers of the copy there)
      // are done; the copies run before the products issued after them
      if (!wait(sh.qd_full(), tit & 1, kSiteMmaQ)) return;
      if (tit > 0 && !wait(sh.qd_tfree(), (tit - 1) & 1, kSiteMmaQ)) return;
      {
        const uint64_t dq_s = sdesc_sw128(sh.q_tile(), 16, 1024);
        const uint64_t do_s = sdesc_sw128(sh.do_tile(), 16, 1024);
        copy_steps<D, 0>(tmem + L::kColQ, desc_lo(dq_s), desc_hi(dq_s));
        copy_steps<D, 0>(tmem + L::kColDO, desc_lo(do_s), desc_hi(do_s));
        mma_commit_w(sh.qd_free());   // the shared-memory buffer may take the next tile
      }
      // prologue: scores of the first kSB - 1 blocks
      const int pro = min(kSB - 1, x.nblk);
      for (int j = 0; j < pro; ++j)
        if (!scores(sit + j)) return;
      if (pro == x.nblk) mma_commit_w(sh.qd_tfree());   // every score product of the tile issued
      for (int j = 0; j < x.nblk; ++j, ++sit) {
        const int buf = sit % kSB;
        // scores kSB - 1 blocks ahead, into the buffer the previous step's
        // dQ product has just read (products run in issue order)
        if (j + kSB - 1 < x.nblk) {
          if (!scores(sit + kSB - 1)) return;
          if (j + kSB == x.nblk) mma_commit_w(sh.qd_tfree());
        }
        if (!wait(sh.p_ready(buf), (sit / kSB) & 1, kSiteMmaP)) return;
        // the previous tile's dQ has been read out before this tile's first
        // (overwriting) dQ product; its score products have run meanwhile
        if (j == 0 && tit > 0 && !wait(sh.dq_empty(), (tit - 1) & 1, kSiteMmaDq)) return;
        // dQ += dS K_j (K_j MN-major: D contiguous, 64-wide chunks 8 KB apart)
        const int kstage = sit % L::kKSt;
        const uint64_t dk = sdesc_sw128(sh.k_tile(kstage), L::kKChunk, 1024);
        dq_steps<0>(tmem + kColDQ, tmem + kColBuf * buf, desc_lo(dk), desc_hi(dk), kIdQ, j > 0 ? 1u : 0u);
        mma_commit_w(sh.k_empty(kstage));
      }
      mma_commit_w(sh.dq_full());
      ++tit;
    }
  }
}

// Elementwise warpgroup H (key columns [32 H, 32 H + 32) of each block;
// thread = query row of the tile), and the dQ epilogue of features
// [H D/2, (H + 1) D/2).
template <int D, bool CAUSAL, bool VARLEN, int H>
__device__ void elementwise_role(const Shared<D, VARLEN>& sh, const uint32_t tmem, const DqParams& p,
                                 const qs::PackedSched& ps, int total_units) {
  constexpr int kC0 = 32 * H;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r_in_tile = (warp & 3) * 32 + lane;
  const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = pk2(sl2, sl2);
  __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq);
  constexpr int kSB = Layout<D, VARLEN>::kSB;
  constexpr uint32_t kColDQ = Layout<D, VARLEN>::kColDQ;
  uint32_t tit = 0, sit = 0;
  for (int u = blockIdx.x, d = qs::first_step(p.snake); u < total_units; u += d, d = qs::next_step(d, p.snake)) {
    const qs::QUnit w = qs::decode_pair_unit<CAUSAL, VARLEN>(u, p, ps);
    const int diag = w.seq_k - w.seq_q;
    for (int t = 0; t < 2; ++t) {
      const Tile x = tile_of<CAUSAL>(w, t);
      const int row = x.row0 + r_in_tile;
      const bool valid = row < w.seq_q;
      if (x.row0 >= w.seq_q) continue;   // no valid row in the tile
      if (x.nblk > 0) {
        // this row's terms: weights exp2(s * scale * log2 e - LSE2), dS =
        // P (dP - Delta); a padding row gets weight 0
        float nl = -INFINITY, nd = 0.0f;
        if (valid) {
          const size_t ri = row_term<VARLEN>(w, row, p);
          nl = p.nlse2[ri];
          nd = p.ndelta[ri];
        }
        const uint64_t nl2 = pk2(nl, nl), nd2 = pk2(nd, nd);
        for (int j = 0; j < x.nblk; ++j, ++sit) {
          const int buf = sit % kSB;
          if (!mbar_wait_bounded(sh.s_full(buf), (sit / kSB) & 1, sh.abort(), &g_err, kSiteEs, p.wait_limit_ns))
            return;
          tc_fence_after();
          const uint32_t tb = tl + kColBuf * buf;
          uint32_t sr[32], dr[32];
          tmem_ld32(tb + kC0, sr);
          tmem_ld32(tb + kColDPoff + kC0, dr);
          tmem_ld_wait();
          tmem_ld_fence(sr);
          tmem_ld_fence(dr);
          // keys of this warpgroup's columns: k0 + c; masked from column
          // cmax on (past the sequence's keys, or after the row's diagonal)
          const int k0 = kBN * j + kC0;
          int cmax = w.seq_k - k0;
          if (CAUSAL) cmax = min(cmax, row + diag - k0 + 1);
          uint32_t dd[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t xs = fma2(pk2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, nl2);
            float x0, x1;
            up2(xs, x0, x1);
            float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
            if (c >= cmax) p0 = 0.0f;
            if (c + 1 >= cmax) p1 = 0.0f;
            const uint64_t g = add2(pk2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), nd2);
            float s0, s1;
            up2(mul2(pk2(p0, p1), g), s0, s1);
            dd[c / 2] = pack_bf16x2(s0, s1);
          }
          // dS as BF16 pairs (keys k0 + 2q, k0 + 2q + 1 in column kC0 + q of
          // the S region): inside the columns this warpgroup has just read
          tmem_st16(tb + kC0, dd);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(sh.p_ready(buf));
        }
        if (!mbar_wait_bounded(sh.dq_full(), tit & 1, sh.abort(), &g_err, kSiteEpi, p.wait_limit_ns)) return;
        tc_fence_after();
      }
      // epilogue: scale * dQ in BF16 (zero when the tile sees no key)
      const size_t tok = size_t(w.q_tok0) + size_t(row);
      __nv_bfloat16* dst = dq + (tok * p.Hq + w.h) * D + H * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
        if (x.nblk > 0) {
          tmem_ld32(tl + kColDQ + H * (D / 2) + 32 * c, r);
          tmem_ld_wait();
          tmem_ld_fence(r);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        if (valid) {
          // 32 features of this row: 64 contiguous bytes, as two 32-byte
          // stores (whole L2 sectors) when dQ allows it, else four 16-byte ones
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * p.scale, __uint_as_float(r[2 * e + 1]) * p.scale);
          if (p.dq_st32) {
            st_global_v8(dst + 32 * c, pk);
            st_global_v8(dst + 32 * c + 16, pk + 8);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              reinterpret_cast<uint4*>(dst + 32 * c)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
      if (x.nblk > 0) {
        tc_fence_before();
        mbar_arrive(sh.dq_empty());
        ++tit;
      }
    }
  }
}

template <int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const DqParams p) {
  using L = Layout<D, VARLEN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32;
  Shared<D, VARLEN> sh;
  sh.base = smem;
  sh.sbase = smem_u32(smem);
  if (threadIdx.x == 0) {
    mbar_init(sh.qd_full(), 1);
    mbar_init(sh.qd_free(), 1);
    mbar_init(sh.qd_tfree(), 1);
    for (int s = 0; s < L::kKSt; ++s) {
      mbar_init(sh.k_full(s), 1);
      mbar_init(sh.k_empty(s), 1);
    }
    for (int s = 0; s < L::kVSt; ++s) {
      mbar_init(sh.v_full(s), 1);
      mbar_init(sh.v_empty(s), 1);
    }
    for (int b = 0; b < L::kSB; ++b) {
      mbar_init(sh.s_full(b), 1);
      mbar_init(sh.p_ready(b), 256);
    }
    mbar_init(sh.dq_full(), 1);
    mbar_init(sh.dq_empty(), 256);
    st_shared(sh.abort(), 0);
    fence_barrier_init();
  }
  if (warp == 8 && (threadIdx.x % 32) == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 9) {
    tmem_alloc(sh.tmem_slot(), 512);
    tmem_relinquish();
  }
  qs::PackedSched ps{};
  int total_units;
  if (VARLEN) total_units = qs::build_packed_sched(p, ps, smem + L::kSched, &g_err);
  else total_units = qs::dense_units(p);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();
  if (warp < 4) {
    elementwise_role<D, CAUSAL, VARLEN, 0>(sh, tmem, p, ps, total_units);
  } else if (warp < 8) {
    elementwise_role<D, CAUSAL, VARLEN, 1>(sh, tmem, p, ps, total_units);
  } else if (warp == 8) {
    if ((threadIdx.x % 32) == 0) producer_role<D, CAUSAL, VARLEN>(sh, &tm_q, &tm_do, &tm_k, &tm_v, p, ps, total_units);
  } else {
    mma_role<D, CAUSAL, VARLEN>(sh, tmem, p, ps, total_units);   // converged warp; one elected lane issues
  }
  // after a give-up, let copies and products already in flight land before
  // the memory they target is released
  if (ld_shared_volatile(sh.abort())) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool VARLEN>
fa_status launch_inst(const BwdLaunch& L, const DqParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                      const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using Lay = Layout<D, VARLEN>;
  auto kern = dq_kernel<D, CAUSAL, VARLEN>;
  const fa_status st = prepare_kernel(reinterpret_cast<const void*>(kern), Lay::kDynamic);
  if (st != FA_OK) return st;
  int grid = L.num_sms;
  if (!VARLEN) {
    const long long units = (long long)((p.Sq + kPairRows - 1) / kPairRows) * p.B * p.Hq;
    if (units < grid) grid = (int)units;
  }
  if (grid < 1) grid = 1;
  kern<<<grid, kThreads, Lay::kDynamic, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D>
fa_status launch_d(const BwdLaunch& L, const DqParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                   const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  const bool varlen = p.cu_seqlens != nullptr;
  if (L.p.causal)
    return varlen ? launch_inst<D, true, true>(L, p, tq, tdo, tk, tv, s)
                  : launch_inst<D, true, false>(L, p, tq, tdo, tk, tv, s);
  return varlen ? launch_inst<D, false, true>(L, p, tq, tdo, tk, tv, s)
                : launch_inst<D, false, false>(L, p, tq, tdo, tk, tv, s);
}

}  // namespace bdq

// dQ of the split backward: reads Q, K, V, dO and the pre pass's row terms,
// writes dQ (BF16) directly.
fa_status launch_bwd_dq(const BwdLaunch& L, cudaStream_t stream) {
  const BwdParams& b = L.p;
  bdq::DqParams p{};
  p.cu_seqlens = b.cu_seqlens;
  p.plan = b.plan;
  p.ndelta = b.ndelta;
  p.nlse2 = b.nlse2;
  p.dq = b.dq;
  p.B = b.B;
  p.Hq = b.Hq;
  p.Hkv = b.Hkv;
  p.Sq = b.Sq;
  p.Sk = b.Sk;
  p.group = b.group;
  p.sched_group = b.B * b.Hq;   // dense causal: all heads in one longest-first group
  p.snake = (b.causal && b.cu_seqlens == nullptr && b.Sq >= 4096) ? 1 : 0;
  p.dq_st32 = (reinterpret_cast<uintptr_t>(b.dq) & 31u) == 0;
  p.sq_pad = b.sq_pad;
  p.scale = b.scale;
  p.scale_log2 = b.scale_log2;
  p.wait_limit_ns = b.wait_limit_ns;
  const bool packed = b.cu_seqlens != nullptr;
  const int rows_q = packed ? b.Sq : b.B * b.Sq;
  const int rows_k = packed ? b.Sk : b.B * b.Sk;
  CUtensorMap tq, tdo, tk, tv;
  fa_status st;
  if ((st = make_tmap_rows_heads_d(&tq, L.q, rows_q, b.Hq, b.D, bdq::kBM)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&tdo, b.dout, rows_q, b.Hq, b.D, bdq::kBM)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&tk, L.k, rows_k, b.Hkv, b.D, bdq::kBN)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&tv, L.v, rows_k, b.Hkv, b.D, bdq::kBN)) != FA_OK) return st;
  if (b.D == 128) return bdq::launch_d<128>(L, p, tq, tdo, tk, tv, stream);
  if (b.D == 64) return bdq::launch_d<64>(L, p, tq, tdo, tk, tv, stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status bwd_dq_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, bdq::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(bdq::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

}  // namespace fa
