// Main kernel of the backward pass on CTA pairs (sm_103a, dense layout,
// D = 128): every tensor-core product is a paired (cta_group::2) tcgen05 MMA
// issued by one thread of the even CTA of a two-CTA cluster.
//
// A work unit is a pair of adjacent key blocks 2m (even CTA) and 2m + 1 (odd
// CTA), 128 keys each, of one (batch, key/value head).  For every query head
// of the group and every 64-row query block i that sees the pair's keys:
//     S^T  = K Q_i^T,  dP^T = V dO_i^T        M = 256 keys, N = 64 queries
//     P^T  = exp2(S^T * scale * log2 e - LSE2_i),  dS^T = P^T * (dP^T - Delta_i)
//     dV  += P^T dO_i, dK += dS^T Q_i          M = 256 keys, N = 128 features
//     dQ_i^T = K^T dS^T                        M = 128 features, N = 64
//                                              queries, K = the pair's 256 keys
// In the first two products each CTA supplies its own 128 keys (A) and half
// of the query block (B: rows 32 r .. 32 r + 31); in dV / dK it supplies the
// 64-feature half r of dO_i / Q_i.  So each CTA reads half of every B operand
// from shared memory, which is the point of pairing ("FlashAttention-4:
// Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
// fdeinterviews.com summary, bullet "Paired-CTA backward pass": one matrix
// multiply over two thread blocks, each holding half an operand, less
// shared-memory operand traffic and half the dQ atomic adds).  The dQ product
// sums over both key blocks, so CTA r ends with features [64 r, 64 r + 64) of
// a partial dQ_i that already covers 256 keys and adds 16 KB per step into
// the FP32 accumulator instead of 32 KB: the pair adds each dQ element once
// where two unpaired CTAs would add it twice.  Its B operand, dS^T of all 256
// keys for the CTA's 32 queries, is written half by the CTA itself and half by
// the other CTA of the pair through distributed shared memory.
//
// Thread layout (384 threads, 12 warps, one CTA per SM, clusters of two):
//   warps 0-3   P / dS elementwise warpgroup (thread = key row of this CTA)
//   warps 4-7   dQ warpgroup (TMEM -> FP32 staging tiles) and dK/dV epilogue
//   warp  8     TMA producer of this CTA's tiles (one lane)
//   warp  9     TMEM (allocated for the pair); in the even CTA the MMA issuer
//   warp  10    dQ reduce issuer (one lane; deterministic-mode tickets)
//   warp  11    odd CTA: forwards the completion of its TMA loads to the even
//               CTA's barriers (one lane); even CTA: idle
//
// Tensor memory of each CTA (512 columns): score buffers b = 0, 1 with S^T at
// 128 b and dP^T at 128 b + 64 (P^T / dS^T as BF16 over their first 32
// columns; the 32-column dQ^T result is written over S^T once the dV product
// has read P^T), dV [256, 384), dK [384, 512).
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "fa_internal.h"
#include "ptx.cuh"
#include "softmax_math.cuh"

namespace fa {
namespace bwdp {

__device__ DeviceError g_err;

constexpr int kD = 128;       // head dimension
constexpr int kBN = 128;      // keys per CTA (256 per pair)
constexpr int kBM = 64;       // query rows per step
constexpr int kHalf = 32;     // query rows (B operand of S^T, dP^T) and dQ^T tile rows per CTA
constexpr int kThreads = 384;
constexpr int kStages = 3;    // Q / dO ring depth

enum Site { kSiteEsS = 1, kSiteEsQ, kSiteEsDs, kSiteDqFull, kSiteDqTicket, kSiteAcc, kSiteMmaKV, kSiteMmaQ,
            kSiteMmaP, kSiteMmaDq, kSiteMmaAcc, kSiteProdKV, kSiteProdQ, kSiteRelay, kSiteRed };

struct Layout {
  static constexpr int kKTile = kBN * kD * 2;        // 32 KB: 2 chunks [128 keys][128 B]
  static constexpr int kKChunk = kBN * 128;          // 16 KB
  static constexpr int kHalfChunk = kHalf * 128;     // 4 KB: 32 rows x 128 B
  // one Q / dO stage (32 KB): the CTA's 32 query rows, both 64-feature
  // chunks (K-major B of S^T / dP^T), then all 64 rows of its feature chunk
  // (MN-major B of dK / dV)
  static constexpr int kQK = 0;
  static constexpr int kQM = 2 * kHalfChunk;
  static constexpr int kGK = kQM + kBM * 128;
  static constexpr int kGM = kGK + 2 * kHalfChunk;
  static constexpr int kStageBytes = kGM + kBM * 128;
  static constexpr int kK = 0;                                    // own key block, K-major
  static constexpr int kV = kK + kKTile;
  static constexpr int kX = kV + kKTile;                          // keys of block 2m, feature half r
  static constexpr int kY = kX + kKChunk;                         // keys of block 2m + 1, feature half r
  static constexpr int kStage0 = kY + kKChunk;
  static constexpr int kDs = kStage0 + kStages * kStageBytes;     // dS^T [256 keys][32 queries], 64-byte swizzle
  static constexpr int kDsBytes = 2 * kBN * kHalf * 2;
  static constexpr int kDqStage = kDs + kDsBytes;                 // 2 FP32 tiles [32 queries][64 features]
  static constexpr int kDqTile = kHalf * 64 * 4;
  static constexpr int kRowTerms = kDqStage + 2 * kDqTile;        // [kStages][-LSE2 | -Delta][64]
  static constexpr int kRowTermBytes = 2 * kBM * 4;
  static constexpr int kBars = kRowTerms + kStages * kRowTermBytes;
  static constexpr int kNumBars = 3 + 3 * kStages + 8 + 2 + 2 + 2;
  static constexpr int kMisc = kBars + kNumBars * 8;              // tmem slot, abort flag
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kDynamic = kTotal + kSmemAlignSlack;
  static_assert(kStageBytes == 32768 && kStage0 % 1024 == 0 && kDs % 1024 == 0, "tile alignment");
  static_assert(kDynamic <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// Work unit: key-block pair m of one (batch, key/value head).  Both CTAs run
// the same steps: query heads of the group x query blocks that see a key of
// block 2m (under a causal mask block 2m + 1 sees a subset of them; its
// extra rows come out as exact zeros).
struct Unit {
  int b, hk, m;
  int n;       // this CTA's key block: 2m + rank
  int i0;      // first query block
  int nq;      // query blocks per head
  int steps;   // group * nq
};

__device__ __forceinline__ int num_pairs(const BwdParams& p) { return ((p.Sk + kBN - 1) / kBN + 1) / 2; }

__device__ __forceinline__ Unit decode_unit(int u, const BwdParams& p, int rank) {
  Unit w;
  // Units in groups of g = sched_group (batch, kv head) pairs, pair index m
  // ascending within a group, each m over the group's heads: g = 1 is
  // head-major (the clusters working at one time share a head's Q / dO
  // reads and its dQ-accumulator slice in L2), used without a mask; under a
  // causal mask pair m sees the most query rows when m is small, so each
  // group runs longest first; deterministic mode uses g = all heads, which
  // puts pair m's predecessor (m - 1) of the same head in an earlier wave of
  // the grid, so the ordered dQ additions rarely wait.
  const int npair = num_pairs(p);
  const int nbh = p.B * p.Hkv;
  const int g = p.sched_group;
  const int grp = u / (g * npair), r = u % (g * npair);
  const int gh = min(g, nbh - grp * g);   // heads in this (possibly last, smaller) group
  const int bh = grp * g + r % gh;
  w.m = r / gh;
  w.b = bh / p.Hkv;
  w.hk = bh % p.Hkv;
  w.n = 2 * w.m + rank;
  const int nqb = (p.Sq + kBM - 1) / kBM;
  int i0 = 0;
  if (p.causal) {
    // query row q sees key j iff j <= q + (Sk - Sq); block i reaches key
    // 256 m (the pair's first key) iff 64 i + 63 + (Sk - Sq) >= 256 m
    const int x = kBN * (2 * w.m) - (p.Sk - p.Sq) - (kBM - 1);
    i0 = x <= 0 ? 0 : (x + kBM - 1) / kBM;
  }
  w.i0 = i0;
  w.nq = nqb > i0 ? nqb - i0 : 0;
  w.steps = p.group * w.nq;
  return w;
}

struct Shared {
  using L = Layout;
  uint8_t* base;
  uint32_t sbase;
  uint32_t rank, peer;
  FA_DEV uint32_t bar(int i) const { return sbase + L::kBars + 8 * i; }
  FA_DEV uint32_t kv_full() const { return bar(0); }    // this CTA's K, V, X, Y landed (TMA)
  FA_DEV uint32_t kv_peer() const { return bar(1); }    // even CTA: the odd CTA's K, V, X, Y landed
  FA_DEV uint32_t kv_empty() const { return bar(2); }   // the pair's unit is done with K, V, X, Y
  FA_DEV uint32_t qd_full(int s) const { return bar(3 + s); }
  FA_DEV uint32_t qd_peer(int s) const { return bar(3 + kStages + s); }
  FA_DEV uint32_t qd_empty(int s) const { return bar(3 + 2 * kStages + s); }
  static constexpr int kB2 = 3 + 3 * kStages;
  FA_DEV uint32_t s_full(int b) const { return bar(kB2 + b); }        // S^T, dP^T of buffer b in TMEM
  FA_DEV uint32_t p_ready(int b) const { return bar(kB2 + 2 + b); }   // even CTA: P^T, dS^T in both CTAs' TMEM
  FA_DEV uint32_t dq_full(int b) const { return bar(kB2 + 4 + b); }
  FA_DEV uint32_t dq_empty(int b) const { return bar(kB2 + 6 + b); }  // even CTA: dQ^T read out by both
  FA_DEV uint32_t ds_free() const { return bar(kB2 + 8); }            // the dQ product has read dS^T
  FA_DEV uint32_t acc_full() const { return bar(kB2 + 9); }
  FA_DEV uint32_t acc_empty() const { return bar(kB2 + 10); }         // even CTA: dK / dV read out by both
  FA_DEV uint32_t dqs_full() const { return bar(kB2 + 11); }          // staging tiles written (128 arrivals)
  FA_DEV uint32_t dqs_free() const { return bar(kB2 + 12); }          // staging tiles read by the TMA unit
  FA_DEV uint32_t ds_ready() const { return bar(kB2 + 13); }          // even CTA: dS^T exchanged (both CTAs)
  FA_DEV uint32_t abort() const { return sbase + L::kMisc + 4; }
  FA_DEV uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + L::kMisc); }
  FA_DEV uint32_t stage(int s) const { return sbase + L::kStage0 + s * L::kStageBytes; }
  FA_DEV uint32_t row_terms(int s) const { return sbase + L::kRowTerms + s * L::kRowTermBytes; }
  FA_DEV const float* stage_nlse2(int s) const {
    return reinterpret_cast<const float*>(base + L::kRowTerms + s * L::kRowTermBytes);
  }
  FA_DEV const float* stage_ndelta(int s) const { return stage_nlse2(s) + kBM; }
  FA_DEV float* dq_stage(int j) const { return reinterpret_cast<float*>(base + L::kDqStage + j * L::kDqTile); }
  FA_DEV uint32_t dq_stage_addr(int j) const { return sbase + L::kDqStage + j * L::kDqTile; }
  // a barrier of the even CTA, by its shared::cluster address
  FA_DEV uint32_t at_leader(uint32_t bar_addr) const { return mapa_shared(bar_addr, 0); }
};

// TMEM columns (see the file comment).
constexpr uint32_t kColBuf = 128, kColDPoff = 64, kColDV = 256, kColDK = 384;

// Gives up on a wait: the other CTA of the pair is told to stop as well.
FA_DEV void stop_pair(const Shared& sh) {
  st_shared(sh.abort(), 1);
  st_cluster_u32(mapa_shared(sh.abort(), sh.peer), 1);
}
// Bounded wait on a barrier of this CTA (cluster-scope acquire: some of them
// receive arrivals from the other CTA or from the pair's MMAs).
FA_DEV bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity, int site, const BwdParams& p) {
  if (mbar_wait_bounded_cluster(bar, parity, sh.abort(), &g_err, site, p.wait_limit_ns)) return true;
  stop_pair(sh);
  return false;
}

struct Maps {
  CUtensorMap q64, q32, g64, g32, k, v, dq;   // g = dO; 64 / 32 = rows per box
};

// TMA producer of this CTA: its K / V block, the feature-half-r columns of
// both key blocks of the pair (A operand of dQ^T), and per step its pieces of
// Q_i / dO_i and the block's row terms.
__device__ void producer_role(const Shared& sh, const Maps& mp, const BwdParams& p, const int total_units) {
  using L = Layout;
  const int r = (int)sh.rank;
  uint32_t sit = 0, ukv = 0;
  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, r);
    if (w.steps == 0) continue;
    if (!wait_bar(sh, sh.kv_empty(), (ukv & 1) ^ 1, kSiteProdKV, p)) return;
    mbar_arrive_expect_tx(sh.kv_full(), 2 * L::kKTile + 2 * L::kKChunk);
    const int krow = w.b * p.Sk + kBN * w.n;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_load_3d(sh.sbase + L::kK + c * L::kKChunk, &mp.k, sh.kv_full(), c * 64, w.hk, krow);
      tma_load_3d(sh.sbase + L::kV + c * L::kKChunk, &mp.v, sh.kv_full(), c * 64, w.hk, krow);
    }
    tma_load_3d(sh.sbase + L::kX, &mp.k, sh.kv_full(), 64 * r, w.hk, w.b * p.Sk + kBN * (2 * w.m));
    tma_load_3d(sh.sbase + L::kY, &mp.k, sh.kv_full(), 64 * r, w.hk, w.b * p.Sk + kBN * (2 * w.m + 1));
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int h = w.hk * p.group + s / w.nq;
      const int i = w.i0 + s % w.nq;
      const int st = sit % kStages;
      if (!wait_bar(sh, sh.qd_empty(st), ((sit / kStages) & 1) ^ 1, kSiteProdQ, p)) return;
      mbar_arrive_expect_tx(sh.qd_full(st), L::kStageBytes + 2 * kBM * 4);
      const int qrow = w.b * p.Sq + kBM * i;
      const uint32_t sb = sh.stage(st);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sb + L::kQK + c * L::kHalfChunk, &mp.q32, sh.qd_full(st), c * 64, h, qrow + kHalf * r);
        tma_load_3d(sb + L::kGK + c * L::kHalfChunk, &mp.g32, sh.qd_full(st), c * 64, h, qrow + kHalf * r);
      }
      tma_load_3d(sb + L::kQM, &mp.q64, sh.qd_full(st), 64 * r, h, qrow);
      tma_load_3d(sb + L::kGM, &mp.g64, sh.qd_full(st), 64 * r, h, qrow);
      const size_t roff = (size_t(w.b) * p.Hq + h) * p.sq_pad + size_t(kBM) * i;
      bulk_load(sh.row_terms(st), p.nlse2 + roff, kBM * 4, sh.qd_full(st));
      bulk_load(sh.row_terms(st) + kBM * 4, p.ndelta + roff, kBM * 4, sh.qd_full(st));
    }
    ++ukv;
  }
}

// Odd CTA: forwards "my tiles have landed" to the even CTA, whose MMAs read
// them.  The odd CTA's producer cannot refill a buffer before the even CTA's
// MMAs have released it, so the forwarded phases never run ahead.
__device__ void relay_role(const Shared& sh, const BwdParams& p, const int total_units) {
  uint32_t sit = 0, ukv = 0;
  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, 1);
    if (w.steps == 0) continue;
    if (!wait_bar(sh, sh.kv_full(), ukv & 1, kSiteRelay, p)) return;
    mbar_arrive_cluster(sh.at_leader(sh.kv_peer()));
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int st = sit % kStages;
      if (!wait_bar(sh, sh.qd_full(st), (sit / kStages) & 1, kSiteRelay, p)) return;
      mbar_arrive_cluster(sh.at_leader(sh.qd_peer(st)));
    }
    ++ukv;
  }
}

// Unrolled K steps of S^T = K Q^T and dP^T = V dO^T (K = 128 features in
// 16-wide steps; K-major operands, step kk in 64-wide chunk kk / 4 at byte
// 32 (kk % 4)).
template <int KK>
FA_DEV void sdp_steps(uint32_t d_s, uint32_t d_dp, uint32_t klo, uint32_t khi, uint32_t vlo, uint32_t vhi,
                      uint32_t qlo, uint32_t qhi, uint32_t glo, uint32_t ghi, uint32_t idesc) {
  if constexpr (KK < kD / 16) {
    constexpr uint32_t oa = ((KK >> 2) * Layout::kKChunk + (KK & 3) * 32) >> 4;
    constexpr uint32_t ob = ((KK >> 2) * Layout::kHalfChunk + (KK & 3) * 32) >> 4;
    mma_pair_ss_w<oa, ob>(d_s, klo, khi, qlo, qhi, idesc, KK > 0 ? 1u : 0u);
    mma_pair_ss_w<oa, ob>(d_dp, vlo, vhi, glo, ghi, idesc, KK > 0 ? 1u : 0u);
    sdp_steps<KK + 1>(d_s, d_dp, klo, khi, vlo, vhi, qlo, qhi, glo, ghi, idesc);
  }
}
// dV += P^T dO, dK += dS^T Q: A in TMEM (8 columns per 16 queries), B
// MN-major (16 query rows = 2048 B per step).
template <int KK>
FA_DEV void grad_steps(uint32_t d_dv, uint32_t d_dk, uint32_t a_p, uint32_t a_ds, uint32_t golo, uint32_t gohi,
                       uint32_t qlo, uint32_t qhi, uint32_t idesc, uint32_t acc) {
  if constexpr (KK < kBM / 16) {
    mma_pair_ts_w<KK * 8, KK * 128>(d_dv, a_p, golo, gohi, idesc, KK > 0 ? 1u : acc);
    mma_pair_ts_w<KK * 8, KK * 128>(d_dk, a_ds, qlo, qhi, idesc, KK > 0 ? 1u : acc);
    grad_steps<KK + 1>(d_dv, d_dk, a_p, a_ds, golo, gohi, qlo, qhi, idesc, acc);
  }
}
// dQ^T = K^T dS^T over the pair's 256 keys: A = K^T (MN-major, block 2m at X
// then block 2m + 1 at Y = X + 16 KB, 16 key rows = 2048 B per step), B = dS^T
// (MN-major, 64-byte swizzle, 16 key rows = 1024 B per step).
template <int KK>
FA_DEV void dq_steps(uint32_t d_dq, uint32_t xlo, uint32_t xhi, uint32_t slo, uint32_t shi, uint32_t idesc) {
  if constexpr (KK < 2 * kBN / 16) {
    constexpr uint32_t oa = ((KK >> 3) * Layout::kKChunk + (KK & 7) * 2048) >> 4;
    mma_pair_ss_w<oa, KK * 64>(d_dq, xlo, xhi, slo, shi, idesc, KK > 0 ? 1u : 0u);
    dq_steps<KK + 1>(d_dq, xlo, xhi, slo, shi, idesc);
  }
}

// MMA issuer (even CTA; the whole warp runs this converged, an elected lane
// issues).  Every commit arrives on the barrier in both CTAs.
__device__ void mma_role(const Shared& sh, const uint32_t tmem, const BwdParams& p, const int total_units) {
  using L = Layout;
  constexpr uint32_t kIdS = idesc_bf16_f32(2 * kBN, kBM, false, false);   // 256 keys x 64 queries
  constexpr uint32_t kIdG = idesc_bf16_f32(2 * kBN, kD, false, true);     // 256 keys x 128 features
  constexpr uint32_t kIdQ = idesc_bf16_f32(kD, kBM, true, true);          // 128 features x 64 queries
  const uint64_t dk_kmaj = sdesc_sw128(sh.sbase + L::kK, 16, 1024);
  const uint64_t dv_kmaj = sdesc_sw128(sh.sbase + L::kV, 16, 1024);
  const uint64_t dx_mn = sdesc_sw128(sh.sbase + L::kX, L::kKChunk, 1024);
  const uint64_t dds = sdesc_sw64(sh.sbase + L::kDs, 8192, 512);
  uint32_t sit = 0, ukv = 0;

  auto wait = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    if (!wait_bar(sh, bar, parity, site, p)) return false;
    tc_fence_after();
    return true;
  };
  // scores of global step t into buffer t & 1, once both CTAs' pieces of
  // Q_t / dO_t have landed and both have read out the dQ^T of step t - 2
  auto scores = [&](uint32_t t) -> bool {
    const int buf = t & 1, st = t % kStages;
    const uint32_t ph = (t / kStages) & 1;
    if (!wait(sh.qd_full(st), ph, kSiteMmaQ) || !wait(sh.qd_peer(st), ph, kSiteMmaQ)) return false;
    if (!wait(sh.dq_empty(buf), ((t >> 1) & 1) ^ 1, kSiteMmaDq)) return false;
    const uint64_t dq = sdesc_sw128(sh.stage(st) + L::kQK, 16, 1024);
    const uint64_t dg = sdesc_sw128(sh.stage(st) + L::kGK, 16, 1024);
    sdp_steps<0>(tmem + kColBuf * buf, tmem + kColBuf * buf + kColDPoff, desc_lo(dk_kmaj), desc_hi(dk_kmaj),
                 desc_lo(dv_kmaj), desc_hi(dv_kmaj), desc_lo(dq), desc_hi(dq), desc_lo(dg), desc_hi(dg), kIdS);
    mma_pair_commit_w(sh.s_full(buf));
    return true;
  };

  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, 0);
    if (w.steps == 0) continue;
    if (!wait(sh.kv_full(), ukv & 1, kSiteMmaKV) || !wait(sh.kv_peer(), ukv & 1, kSiteMmaKV)) return;
    if (!scores(sit)) return;
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int st = sit % kStages, buf = sit & 1;
      // next step's scores first, so they run during this step's
      // elementwise pass
      if (s + 1 < w.steps && !scores(sit + 1)) return;
      if (!wait(sh.p_ready(buf), (sit >> 1) & 1, kSiteMmaP)) return;
      if (s == 0 && ukv > 0 && !wait(sh.acc_empty(), (ukv - 1) & 1, kSiteMmaAcc)) return;
      const uint64_t dgo = sdesc_sw128(sh.stage(st) + L::kGM, L::kKChunk, 1024);
      const uint64_t dqq = sdesc_sw128(sh.stage(st) + L::kQM, L::kKChunk, 1024);
      grad_steps<0>(tmem + kColDV, tmem + kColDK, tmem + kColBuf * buf, tmem + kColBuf * buf + kColDPoff,
                    desc_lo(dgo), desc_hi(dgo), desc_lo(dqq), desc_hi(dqq), kIdG, s > 0 ? 1u : 0u);
      mma_pair_commit_w(sh.qd_empty(st));
      // dQ^T over the S^T columns of this buffer (the dV product, issued
      // before, has read P^T from them), once dS^T is exchanged
      if (!wait(sh.ds_ready(), sit & 1, kSiteMmaP)) return;
      dq_steps<0>(tmem + kColBuf * buf, desc_lo(dx_mn), desc_hi(dx_mn), desc_lo(dds), desc_hi(dds), kIdQ);
      mma_pair_commit_w(sh.dq_full(buf));
      mma_pair_commit_w(sh.ds_free());
    }
    mma_pair_commit_w(sh.acc_full());
    mma_pair_commit_w(sh.kv_empty());
    ++ukv;
  }
}

// dS^T row of one key into the B operand of dQ^T: row R of [256 keys][32
// queries], 64-byte rows, 16-byte chunk j stored at chunk j ^ ((R / 2) mod 4).
// Queries [32 H, 32 H + 32) of the thread's 64 (packed in dd[16 H .. 16 H + 15])
// go to this CTA (`remote` false) or to the other CTA of the pair.
template <int H>
FA_DEV void store_ds_half(uint32_t region, uint32_t peer, int R, const uint32_t (&dd)[32], bool remote) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a = region + R * 64 + ((j ^ ((R >> 1) & 3)) << 4);
    if (remote)
      st_cluster_v4(mapa_shared(a, peer), dd[16 * H + 4 * j], dd[16 * H + 4 * j + 1], dd[16 * H + 4 * j + 2],
                    dd[16 * H + 4 * j + 3]);
    else
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(dd[16 * H + 4 * j]),
                   "r"(dd[16 * H + 4 * j + 1]), "r"(dd[16 * H + 4 * j + 2]), "r"(dd[16 * H + 4 * j + 3])
                   : "memory");
  }
}

// P / dS warpgroup: thread = key row kr of this CTA's key block, 64 query
// columns per step.
__device__ void elementwise_role(const Shared& sh, const uint32_t tmem, const BwdParams& p,
                                 const int total_units) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kr = (warp & 3) * 32 + lane;
  const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = pk2(sl2, sl2);
  const int diag = p.Sk - p.Sq;
  const int R = kBN * (int)sh.rank + kr;   // this key's row in the pair's dS^T
  const uint32_t ds_region = sh.sbase + Layout::kDs;
  uint32_t sit = 0;
  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, (int)sh.rank);
    const int key = kBN * w.n + kr;
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int i = w.i0 + s % w.nq;
      const int st = sit % kStages, buf = sit & 1;
      if (!wait_bar(sh, sh.qd_full(st), (sit / kStages) & 1, kSiteEsQ, p)) return;
      if (!wait_bar(sh, sh.s_full(buf), (sit >> 1) & 1, kSiteEsS, p)) return;
      tc_fence_after();
      const uint32_t tb = tl + kColBuf * buf;
      uint32_t sr[2][32], dr[2][32];
      tmem_ld32(tb, sr[0]);
      tmem_ld32(tb + 32, sr[1]);
      tmem_ld32(tb + kColDPoff, dr[0]);
      tmem_ld32(tb + kColDPoff + 32, dr[1]);
      tmem_ld_wait();
      tmem_ld_fence(sr[0]);
      tmem_ld_fence(sr[1]);
      tmem_ld_fence(dr[0]);
      tmem_ld_fence(dr[1]);
      // columns c < cmin are masked: keys past Sk, or (causal) queries that
      // come before this key
      int cmin = 0;
      if (key >= p.Sk) cmin = kBM;
      else if (p.causal) cmin = min(kBM, max(0, key - diag - kBM * i));
      const float2* nl = reinterpret_cast<const float2*>(sh.stage_nlse2(st));
      const float2* nd = reinterpret_cast<const float2*>(sh.stage_ndelta(st));
      uint32_t pp[32], dd[32];
#pragma unroll
      for (int c = 0; c < kBM; c += 2) {
        const float2 l2 = nl[c / 2], d2 = nd[c / 2];
        const uint64_t x = fma2(pk2(__uint_as_float(sr[c / 32][c % 32]), __uint_as_float(sr[c / 32][c % 32 + 1])),
                                sl2x2, pk2(l2.x, l2.y));
        float x0, x1;
        up2(x, x0, x1);
        float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
        if (c < cmin) p0 = 0.0f;
        if (c + 1 < cmin) p1 = 0.0f;
        const uint64_t g = add2(pk2(__uint_as_float(dr[c / 32][c % 32]), __uint_as_float(dr[c / 32][c % 32 + 1])),
                                pk2(d2.x, d2.y));
        float s0, s1;
        up2(mul2(pk2(p0, p1), g), s0, s1);
        pp[c / 2] = pack_bf16x2(p0, p1);
        dd[c / 2] = pack_bf16x2(s0, s1);
      }
      // P^T and dS^T as BF16 into TMEM (A operands of dV and dK); the
      // paired dV / dK products may start as soon as both CTAs have them
      tmem_st32(tb, pp);
      tmem_st32(tb + kColDPoff, dd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_cluster_relaxed(sh.at_leader(sh.p_ready(buf)));
      // dS^T into the B operand of dQ^T in both CTAs, once the previous
      // step's dQ product has read it
      if (!wait_bar(sh, sh.ds_free(), (sit & 1) ^ 1, kSiteEsDs, p)) return;
      if (sh.rank == 0) {
        store_ds_half<0>(ds_region, sh.peer, R, dd, false);
        store_ds_half<1>(ds_region, sh.peer, R, dd, true);
      } else {
        store_ds_half<1>(ds_region, sh.peer, R, dd, false);
        store_ds_half<0>(ds_region, sh.peer, R, dd, true);
      }
      fence_proxy_async_cluster();
      mbar_arrive_cluster(sh.at_leader(sh.ds_ready()));
    }
  }
}

// dQ warpgroup: TMEM lane l = 64 j + f holds feature 64 r + f of queries
// [32 j, 32 j + 32) of dQ_i^T (summed over the pair's keys); it goes to FP32
// staging tile j [32 queries][64 features] for the reduce issuer.  At the end
// of a unit, lane = key row: dV and scale * dK of this CTA's keys in BF16.
__device__ void dq_role(const Shared& sh, const uint32_t tmem, const BwdParams& p, const int total_units) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int l = (warp & 3) * 32 + lane;
  const int j = l >> 6, f = l & 63;
  const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
  uint32_t sit = 0, ukv = 0;
  __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk);
  __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(p.dv);
  float* tile = sh.dq_stage(j);
  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, (int)sh.rank);
    bool stop = false;
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int buf = sit & 1;
      if (!wait_bar(sh, sh.dq_full(buf), (sit >> 1) & 1, kSiteDqFull, p)) {
        stop = true;
        break;
      }
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tl + kColBuf * buf, v);
      tmem_ld_wait();
      tmem_ld_fence(v);
      tc_fence_before();
      mbar_arrive_cluster_relaxed(sh.at_leader(sh.dq_empty(buf)));
      if (!wait_bar(sh, sh.dqs_free(), (sit & 1) ^ 1, kSiteDqFull, p)) {
        stop = true;
        break;
      }
#pragma unroll
      for (int c = 0; c < kHalf; ++c) tile[c * 64 + f] = __uint_as_float(v[c]);
      fence_proxy_async_smem();
      mbar_arrive(sh.dqs_full());
    }
    if (stop || ld_shared_volatile(sh.abort())) break;
    // epilogue of the unit: dV and scale * dK rows in BF16
    const int key = kBN * w.n + l;
    const bool valid = key < p.Sk;
    const size_t roff = ((size_t(w.b) * p.Sk + key) * p.Hkv + w.hk) * kD;
    if (w.steps > 0) {
      if (!wait_bar(sh, sh.acc_full(), ukv & 1, kSiteAcc, p)) break;
      tc_fence_after();
    }
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
      const float mul = which ? p.scale : 1.0f;
      __nv_bfloat16* dst = (which ? dk : dv) + roff;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t r[32];
        if (w.steps > 0) {
          tmem_ld32(tl + (which ? kColDK : kColDV) + c * 32, r);
          tmem_ld_wait();
          tmem_ld_fence(r);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        if (valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * mul, __uint_as_float(r[8 * e + 1]) * mul);
            o.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * mul, __uint_as_float(r[8 * e + 3]) * mul);
            o.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * mul, __uint_as_float(r[8 * e + 5]) * mul);
            o.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * mul, __uint_as_float(r[8 * e + 7]) * mul);
            reinterpret_cast<uint4*>(dst + c * 32)[e] = o;
          }
        }
      }
    }
    if (w.steps > 0) {
      tc_fence_before();
      mbar_arrive_cluster_relaxed(sh.at_leader(sh.acc_empty()));
      ++ukv;
    }
  }
}

// dQ reduce issuer (one thread): adds the two staging tiles (features
// [64 r, 64 r + 64) of the block's 64 query rows) into the FP32 accumulator
// with TMA bulk tensor reduce-adds.  Out-of-range rows are skipped by the
// unit; rows of a padded query block that belong to the next sequence receive
// exact zeros, since their weights are 0.  Deterministic mode: the pairs add
// into one (b, h, i, feature half) in ascending pair order m = 0, 1, ...; a
// step's ticket is released one step late (once at most the next step's two
// additions are pending), and never held across units, so waits point only
// from pair m to pair m - 1 of the same head.
__device__ void reduce_role(const Shared& sh, const CUtensorMap* tdq, const BwdParams& p, const int total_units) {
  const int r = (int)sh.rank;
  uint32_t sit = 0;
  int* held = nullptr;
  int held_next = 0;
  auto release_held = [&]() {
    __threadfence();
    st_release_gpu(held, held_next);
    held = nullptr;
  };
  for (int u = cluster_id_x(); u < total_units; u += nclusters_x()) {
    const Unit w = decode_unit(u, p, r);
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int h = w.hk * p.group + s / w.nq;
      const int i = w.i0 + s % w.nq;
      if (!wait_bar(sh, sh.dqs_full(), sit & 1, kSiteRed, p)) goto done;
      int* ticket = nullptr;
      if (p.deterministic) {
        ticket = p.tickets + ((size_t(w.b) * p.Hq + h) * p.nqb + i) * 2 + r;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(ticket) != w.m) {
          if (ld_shared_volatile(sh.abort()) || globaltimer_ns() - t0 > p.wait_limit_ns) {
            if (atomicCAS(&g_err.status, 0, FA_ERR_TIMEOUT) == 0) atomicExch(&g_err.site, kSiteDqTicket);
            stop_pair(sh);
            goto done;
          }
          __nanosleep(64);
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        tma_reduce_add_3d(tdq, sh.dq_stage_addr(j), 64 * r, h, w.b * p.Sq + kBM * i + kHalf * j);
        bulk_commit_group();
      }
      bulk_wait_group_read0();   // the staging tiles may be overwritten
      mbar_arrive(sh.dqs_free());
      if (p.deterministic) {
        if (held) {
          bulk_wait_group2();    // the previous step's two additions are complete
          release_held();
        }
        held = ticket;
        held_next = w.m + 1;
      }
    }
    if (held) {
      bulk_wait_group0();
      release_held();
    }
  }
done:
  bulk_wait_group0();   // outstanding reductions finish before the CTA exits
  if (held) release_held();
}

__global__ void __launch_bounds__(kThreads, 1) bwd_pair_kernel(const __grid_constant__ Maps mp, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  Shared sh;
  sh.base = smem;
  sh.sbase = smem_u32(smem);
  sh.rank = cluster_ctarank();
  sh.peer = sh.rank ^ 1u;
  if (threadIdx.x == 0) {
    mbar_init(sh.kv_full(), 1);
    mbar_init(sh.kv_peer(), 1);
    mbar_init(sh.kv_empty(), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sh.qd_full(s), 1);
      mbar_init(sh.qd_peer(s), 1);
      mbar_init(sh.qd_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.s_full(b), 1);
      mbar_init(sh.p_ready(b), 2 * 128);
      mbar_init(sh.dq_full(b), 1);
      mbar_init(sh.dq_empty(b), 2 * 128);
    }
    mbar_init(sh.ds_free(), 1);
    mbar_init(sh.acc_full(), 1);
    mbar_init(sh.acc_empty(), 2 * 128);
    mbar_init(sh.dqs_full(), 128);
    mbar_init(sh.dqs_free(), 1);
    mbar_init(sh.ds_ready(), 2 * 128);
    st_shared(sh.abort(), 0);
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&mp.q64);
    tma_prefetch_desc(&mp.q32);
    tma_prefetch_desc(&mp.g64);
    tma_prefetch_desc(&mp.g32);
    tma_prefetch_desc(&mp.k);
    tma_prefetch_desc(&mp.v);
    tma_prefetch_desc(&mp.dq);
  }
  if (warp == 9) {
    tmem_alloc_pair(sh.tmem_slot(), 512);
    tmem_relinquish_pair();
  }
  const int total_units = num_pairs(p) * p.B * p.Hkv;
  tc_fence_before();
  // both CTAs' barriers and TMEM exist before any remote arrival or MMA
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();
  if (warp < 4) {
    elementwise_role(sh, tmem, p, total_units);
  } else if (warp < 8) {
    dq_role(sh, tmem, p, total_units);
  } else if (warp == 8) {
    if (lane == 0) producer_role(sh, mp, p, total_units);
  } else if (warp == 9) {
    if (sh.rank == 0) mma_role(sh, tmem, p, total_units);   // converged warp; one elected lane issues
  } else if (warp == 10) {
    if (lane == 0) reduce_role(sh, &mp.dq, p, total_units);
  } else {
    if (lane == 0 && sh.rank == 1) relay_role(sh, p, total_units);
  }
  __syncwarp();
  if (ld_shared_volatile(sh.abort())) {
    // a wait gave up: let copies and products already issued drain
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  // neither CTA leaves (or frees TMEM) while the pair's products or remote
  // writes may still reach it
  cluster_sync();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace bwdp

// Main kernel of the paired backward; the caller has run the pre pass and
// runs the post pass.
fa_status launch_bwd_pair_main(const BwdLaunch& L, cudaStream_t stream) {
  const BwdParams& p = L.p;
  if (p.D != bwdp::kD) return FA_ERR_UNSUPPORTED;
  bwdp::Maps mp;
  fa_status st;
  if ((st = make_tmap_rows_heads_d(&mp.q64, L.q, p.B * p.Sq, p.Hq, p.D, bwdp::kBM)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&mp.q32, L.q, p.B * p.Sq, p.Hq, p.D, bwdp::kHalf)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&mp.g64, p.dout, p.B * p.Sq, p.Hq, p.D, bwdp::kBM)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&mp.g32, p.dout, p.B * p.Sq, p.Hq, p.D, bwdp::kHalf)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&mp.k, L.k, p.B * p.Sk, p.Hkv, p.D, bwdp::kBN)) != FA_OK) return st;
  if ((st = make_tmap_rows_heads_d(&mp.v, L.v, p.B * p.Sk, p.Hkv, p.D, bwdp::kBN)) != FA_OK) return st;
  if ((st = make_tmap_f32_rows_heads_d(&mp.dq, p.dq_acc, p.B * p.Sq, p.Hq, p.D, 64, bwdp::kHalf)) != FA_OK)
    return st;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(bwdp::kThreads, 1, 1);
  cfg.dynamicSmemBytes = bwdp::Layout::kDynamic;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((st = prepare_kernel(reinterpret_cast<const void*>(bwdp::bwd_pair_kernel), bwdp::Layout::kDynamic)) != FA_OK)
    return st;
  // resident clusters per device, computed once per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  constexpr int kMaxDevices = 64;
  static int resident[kMaxDevices] = {};
  static std::mutex mu;
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    if (resident[dev] == 0) {
      cfg.gridDim = dim3(2 * (L.num_sms / 2), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, bwdp::bwd_pair_kernel, &cfg) != cudaSuccess || n < 1)
        return FA_ERR_CUDA;
      resident[dev] = n;
    }
    max_clusters = resident[dev];
  }
  // as many clusters as can be resident at once: the deterministic mode's
  // ordered additions then only ever wait on running clusters
  const long long units =
      (long long)(((p.Sk + bwdp::kBN - 1) / bwdp::kBN + 1) / 2) * p.B * p.Hkv;
  const int clusters = (int)(units < max_clusters ? units : max_clusters);
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  if (cudaLaunchKernelEx(&cfg, bwdp::bwd_pair_kernel, mp, p) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status bwd_pair_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, bwdp::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(bwdp::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

}  // namespace fa
