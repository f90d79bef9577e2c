// Backward pass of exact attention on sm_103a (dense and packed layouts,
// head dimension D = 64 or 128).
//
// Three kernels per call:
//   pre   Delta_i = sum_d dO_id * O_id and LSE_i * log2(e) per query row (FP32,
//         rows padded to a multiple of 64), the FP32 dQ accumulator and the
//         deterministic-mode tickets zeroed;
//   main  one persistent, warp-specialised CTA per SM; a work unit is one block
//         of 128 keys of one (batch, key/value head).  For every query head of
//         the group and every 64-row query block it recomputes the scores and
//         runs the five products of the backward pass on the tensor cores
//         (tcgen05, accumulators in TMEM):
//             S^T  = K Q_i^T            dP^T = V dO_i^T
//             P^T  = exp2(S^T * scale * log2 e - LSE2_i)
//             dS^T = P^T * (dP^T - Delta_i)
//             dV  += P^T dO_i           dK  += dS^T Q_i
//             dQ_i^T = K^T dS^T   -> added to the FP32 accumulator
//         dK and dV stay in TMEM across the whole group and are written once
//         per unit, so they need no atomics.  dQ partial sums are added by the
//         TMA unit (bulk tensor reduce-adds of 32 x D FP32 tiles staged
//         through two shared-memory buffers, so one tile is written while the
//         other is read), in deterministic mode (when selected instead of
//         the split backward below) in ascending key-block order enforced by
//         one ticket per (batch, head, query block);
//   post  dQ = BF16(scale * accumulator).
//
// Deterministic mode runs by default as a split backward: this main kernel
// without its dQ product (dK, dV only; no accumulator, no post pass), and the
// dQ kernel of fa_bwd_dq.cu, which computes each dQ tile whole.
//
// Sources: "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling" (fdeinterviews.com summary): the paragraph on
// Blackwell's changed balance (the backward tile: five products, shared-memory
// traffic the bottleneck), bullet "Paired-CTA backward pass" (dQ through global
// atomic adds) and the paragraph on the deterministic backward mode and
// longest-first ordering.  Every product here runs on one SM's tensor core;
// the paired-CTA (2-SM) variant of that bullet is the separate kernel in
// fa_bwd_pair.cu.
//
// Schedules: a static one (CTA c takes units c, c + grid, ...) for dense
// calls -- head-major without a mask, longest-first (key-block-major) within
// groups of heads under a causal mask or in deterministic mode -- and a
// dynamic one (units claimed from an atomic counter, announced to the roles
// through a ring in shared memory) for packed calls, in the longest-first
// order the plan kernel writes.
//
// Thread layout (512 threads, 16 warps, one CTA per SM; registers per thread
// after setmaxnreg: elementwise 160, dQ 128, warps 8-11 64):
//   warps 0-3   P / dS elementwise warpgroup for query columns 0-31 (one
//               thread per key row)
//   warps 12-15 the same for query columns 32-63
//   warps 4-7   dQ warpgroup (dQ^T from TMEM to the staging tiles) and the
//               dK/dV epilogue
//   warp  8     TMA producer (one lane)
//   warp  9     TMEM owner + MMA issuer (converged warp, one elected lane issues)
//   warp  10    dQ reduce issuer (one lane; deterministic-mode tickets)
//   warp  11    idle
//
// Tensor memory (512 columns): two score buffers b = 0, 1 (steps alternate)
// with S^T at 128 b and dP^T at 128 b + 64 (P^T / dS^T as BF16 over columns
// 0-15 and 32-47 of each region, one half per elementwise warpgroup; the dQ^T
// product is written over dP^T once the dK product has read dS^T), dV
// [256, 384), dK [384, 512).
#include <cuda_runtime.h>

#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "fa_internal.h"
#include "ptx.cuh"
#include "softmax_math.cuh"

namespace fa {
namespace bwd {

__device__ DeviceError g_err;

constexpr int kBN = 128;       // keys per work unit
constexpr int kBM = 64;        // query rows per step
constexpr int kThreads = 512;
constexpr int kStages = 3;     // Q / dO ring depth
constexpr int kDqRows = 32;    // rows of the FP32 dQ staging tile (half a query block)
constexpr int kRing = 4;       // work units announced ahead by the producer
// consumers of each announced unit: two elementwise warpgroups, the dQ
// warpgroup, the MMA warp and the reduce issuer
constexpr int kRingReaders = 128 + 128 + 128 + 32 + 1;

enum Site { kSiteEsS = 1, kSiteEsQ, kSiteEsDs, kSiteDqFull, kSiteDqTicket, kSiteAcc, kSiteMmaKV, kSiteMmaQ,
            kSiteMmaP, kSiteMmaDq, kSiteMmaAcc, kSiteProdKV, kSiteProdQ };

// Shared-memory layout for head dimension kD (64 or 128): tiles of kD / 64
// chunks, each 64 features (128 bytes) wide.
template <int kD>
struct Layout {
  static constexpr int kKTile = kBN * kD * 2;        // kD = 128: 32 KB, 2 chunks of 128 rows x 128 B
  static constexpr int kKChunk = kBN * 128;          // 16 KB
  static constexpr int kQTile = kBM * kD * 2;        // kD = 128: 16 KB, 2 chunks of 64 rows x 128 B
  static constexpr int kQChunk = kBM * 128;          // 8 KB
  static constexpr int kStageStride = 2 * kQTile;                 // Q, dO (1024-aligned)
  static constexpr int kRowTermBytes = 2 * kBM * 4;               // -LSE2, -Delta of the stage's rows
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKTile;
  static constexpr int kStage0 = kV + kKTile;
  static constexpr int kDs = kStage0 + kStages * kStageStride;    // dS^T smem, 2 buffers of 16 KB
  static constexpr int kDsBytes = kBN * 128;
  static constexpr int kDqStage = kDs + 2 * kDsBytes;             // 2 FP32 dQ tiles [32 rows][128]
  static constexpr int kDqStageBytes = kDqRows * kD * 4;
  static constexpr int kRowTerms = kDqStage + 2 * kDqStageBytes;  // [kStages][2][kBM] floats
  static constexpr int kBars = kRowTerms + kStages * kRowTermBytes;
  // kv_full, kv_empty, qd_full[S], qd_empty[S], s_full[2], p_ready[2],
  // dq_full[2], dq_empty[2], ds_free[2], acc_full, acc_empty, dqs_full[2], dqs_free[2], q_full[S],
  // unit ring full[4] / empty[4]
  static constexpr int kNumBars = 2 + 2 * kStages + 10 + 2 + 4 + kStages + 2 * kRing;
  static constexpr int kMisc = kBars + kNumBars * 8;              // tmem slot, abort, check-in count
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kDynamic = kTotal + kSmemAlignSlack;
  static_assert(kDynamic <= 232448, "dynamic shared memory above the 227 KB per-CTA limit");
};

// ------------------------------------------------------------- pre / post --

// This lane's kD / 32 consecutive elements of a row: sum of dO * O, and the
// same elements of the FP32 dQ accumulator set to zero.
template <int kD>
FA_DEV float row_dot(const __nv_bfloat16* o, const __nv_bfloat16* g) {
  float acc = 0.0f;
#pragma unroll
  for (int e = 0; e < kD / 64; ++e) {
    const float2 a = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(o)[e]);
    const float2 b = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(g)[e]);
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
  }
  return acc;
}
template <int kD>
FA_DEV void zero_row_part(float* a) {
  if constexpr (kD == 128) *reinterpret_cast<float4*>(a) = make_float4(0.f, 0.f, 0.f, 0.f);
  else *reinterpret_cast<float2*>(a) = make_float2(0.f, 0.f);
}

// One warp per padded query row (b, h, q): stores -LSE * log2(e) and -Delta
// (negated so the main kernel adds them with one packed FMA / ADD) and zeroes
// the row's dQ accumulator (when there is one: the split backward writes dQ
// from its own kernel).  Rows q >= Sq (padding) and rows that saw no key
// (LSE = -inf) get -inf and 0, so their weights come out as exactly 0.
template <int kD>
__global__ void pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                           const float* __restrict__ lse, float* __restrict__ ndelta, float* __restrict__ nlse2,
                           float* __restrict__ dq_acc, int* __restrict__ tickets, long long n_tickets,
                           int* __restrict__ sched, int B, int Hq, int Sq, int sq_pad) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;   // work-unit counter of the main kernel
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)B * Hq * sq_pad;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp_id; r < rows; r += nwarps) {
    const int q = (int)(r % sq_pad);
    const long long bh = r / sq_pad;
    const int h = (int)(bh % Hq);
    const int b = (int)(bh / Hq);
    float dl = 0.0f, l2 = -INFINITY;
    if (q < Sq) {
      const size_t off = ((size_t(b) * Sq + q) * Hq + h) * kD + lane * (kD / 32);
      const float acc0 = row_dot<kD>(o + off, dout + off);
      float acc = acc0;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
      dl = -acc;
      const float lv = lse[(size_t(b) * Hq + h) * Sq + q];
      l2 = (lv == -INFINITY) ? -INFINITY : -lv * 1.4426950408889634f;
      if (dq_acc) zero_row_part<kD>(dq_acc + off);
    }
    if (lane == 0) {
      ndelta[r] = dl;
      nlse2[r] = l2;
    }
  }
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long t = tid; t < n_tickets; t += (long long)gridDim.x * blockDim.x) tickets[t] = 0;
}

// dQ = BF16(scale * accumulator), eight elements per thread.  Packed layout:
// nothing is written when the plan kernel rejected the offsets (`rejected`
// points at its status word; nullptr for the dense layout).
__global__ void post_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, long long n8,
                            float scale, const int* __restrict__ rejected) {
  if (rejected && *rejected) return;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
    const float4 c = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
    uint4 out;
    out.x = pack_bf16x2(a.x * scale, a.y * scale);
    out.y = pack_bf16x2(a.z * scale, a.w * scale);
    out.z = pack_bf16x2(c.x * scale, c.y * scale);
    out.w = pack_bf16x2(c.z * scale, c.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = out;
  }
}

// ------------------------------------------------------------ packed layout --

// One block of 1024 threads (B <= 1024 sequences): checks the offsets
// (cu_seqlens[0] = 0, non-decreasing, at most 262,144 tokens per sequence,
// cu_seqlens[B] = total) and writes the per-sequence tables of the packed
// backward: plan[0..B] = prefix sums of 128-key blocks, plan[B+1..2B+1] =
// prefix sums of the sequences' rows rounded up to 64 (where their row terms
// and tickets start), plan[2B+2] = the total number of key blocks (0 when
// the offsets are invalid, so that nothing is computed) and plan[2B+3] = 1
// for invalid offsets, which is also reported as FA_ERR_INVALID_ARG.
//
// It also writes the work order of the main kernel (one entry per key block
// and kv head), longest first ("FlashAttention-4 ...", the paragraph on
// longest-first scheduling of causal and variable-length work): the
// (sequence, kv head) pairs sorted by key-block count, most first (ties by
// sequence index, then kv head), cut into groups of `group` consecutive
// pairs; the groups in that order, and within a group key block 0 of every
// pair, then key block 1 of the pairs that have one, and so on.  Under a
// causal mask key block n of a sequence sees more query rows than block
// n + 1, so every group starts with its longest units; each pair has a few
// consecutive key blocks in flight at one time (L2 reuse of its query
// rows); and block n - 1 of a pair always comes before block n, at most
// `group` entries earlier (the deterministic mode's ordered additions wait
// only on earlier units).
__global__ void __launch_bounds__(1024) plan_kernel(const int* __restrict__ cu, int B, int total, int Hkv,
                                                    int group, int* __restrict__ plan, int2* __restrict__ order) {
  __shared__ int s_blk[1024], s_pad[1024], s_nb[1024], s_seq[1024], s_rnb[1024], s_rpre[1024];
  __shared__ int bad;
  const int t = threadIdx.x;
  if (t == 0) bad = 0;
  __syncthreads();
  int nb = 0, np = 0;
  if (t < B) {
    const int a = cu[t], c = cu[t + 1];
    const int len = c - a;
    if (len < 0 || len > kMaxPairsPerSeq * 256 || (t == 0 && a != 0) || (t == B - 1 && c != total))
      atomicOr(&bad, 1);
    const int l = len < 0 ? 0 : len;
    nb = (l + kBN - 1) / kBN;
    np = (l + kBM - 1) / kBM * kBM;
  }
  s_blk[t] = nb;
  s_pad[t] = np;
  s_nb[t] = nb;
  __syncthreads();
  // inclusive prefix sums over the 1024 entries
  for (int off = 1; off < 1024; off <<= 1) {
    const int x = t >= off ? s_blk[t - off] : 0;
    const int y = t >= off ? s_pad[t - off] : 0;
    __syncthreads();
    s_blk[t] += x;
    s_pad[t] += y;
    __syncthreads();
  }
  if (t < B) {
    plan[t] = t ? s_blk[t - 1] : 0;
    plan[B + 1 + t] = t ? s_pad[t - 1] : 0;
  }
  if (t == 0) {
    plan[B] = s_blk[B - 1];
    plan[2 * B + 1] = s_pad[B - 1];
    plan[2 * B + 2] = bad ? 0 : s_blk[B - 1];
    plan[2 * B + 3] = bad;
    if (bad && atomicCAS(&g_err.status, 0, FA_ERR_INVALID_ARG) == 0) atomicExch(&g_err.site, 0);
  }
  if (bad) return;   // block-uniform: nothing is computed

  // sequences by key-block count, most first (rank r holds sequence s_seq[r])
  if (t < B) {
    int rank = 0;
    for (int c = 0; c < B; ++c) rank += (s_nb[c] > nb) || (s_nb[c] == nb && c < t);
    s_seq[rank] = t;
    s_rnb[rank] = nb;
  }
  __syncthreads();
  // exclusive prefix of the ranked counts: pair q = r * Hkv + h starts at
  // entry Hkv * s_rpre[r] + h * s_rnb[r] of the pair-major enumeration
  s_rpre[t] = t < B ? s_rnb[t] : 0;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int x = t >= off ? s_rpre[t - off] : 0;
    __syncthreads();
    s_rpre[t] += x;
    __syncthreads();
  }
  const int incl = s_rpre[t];
  __syncthreads();
  s_rpre[t] = incl - (t < B ? s_rnb[t] : 0);
  __syncthreads();

  const long long npairs = (long long)B * Hkv;
  for (long long q = t; q < npairs; q += blockDim.x) {
    const int r = (int)(q / Hkv), h = (int)(q % Hkv);
    const int nbq = s_rnb[r];
    const long long g0 = q - q % group;
    const long long g1 = g0 + group < npairs ? g0 + group : npairs;
    // the group's first entry, and its member count at each level n (pairs
    // with more than n key blocks: a prefix of the group, counts descend)
    const int r0 = (int)(g0 / Hkv), h0 = (int)(g0 % Hkv);
    long long pos = (long long)Hkv * s_rpre[r0] + (long long)h0 * s_rnb[r0] + (q - g0);
    long long members = g1 - g0;
    for (int n = 0; n < nbq; ++n) {
      while (members > 0 && s_rnb[(int)((g0 + members - 1) / Hkv)] <= n) --members;
      order[pos] = make_int2(h * kMaxPackedSeqs + s_seq[r], n);
      pos += members;
    }
  }
}

// Packed counterpart of pre_kernel.  Row terms live per head over the padded
// rows of all sequences (sequence b from plan[B+1+b], rounded up to 64 rows);
// padding rows get -inf and 0 so their weights are exactly 0.  One warp per
// padded row; the real rows' dQ accumulator rows are zeroed.
template <int kD>
__global__ void pre_packed_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                  const float* __restrict__ lse, const int* __restrict__ cu,
                                  const int* __restrict__ plan, float* __restrict__ ndelta,
                                  float* __restrict__ nlse2, float* __restrict__ dq_acc, int* __restrict__ tickets,
                                  long long n_tickets, int* __restrict__ sched, int B, int Hq, int total,
                                  int sq_pad) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;   // work-unit counter of the main kernel
  if (plan[2 * B + 3] != 0) return;   // offsets rejected: nothing is computed
  const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)Hq * sq_pad;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int* pad = plan + B + 1;
  for (long long r = warp_id; r < rows; r += nwarps) {
    const int h = (int)(r / sq_pad);
    const int pr = (int)(r % sq_pad);
    float dl = 0.0f, l2 = -INFINITY;
    if (pr < pad[B]) {
      int lo = 0, hi = B;   // pad[lo] <= pr < pad[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pad[mid] <= pr) lo = mid;
        else hi = mid;
      }
      const int off = pr - pad[lo];
      if (off < cu[lo + 1] - cu[lo]) {
        const int tok = cu[lo] + off;
        const size_t e = ((size_t)tok * Hq + h) * kD + lane * (kD / 32);
        float acc = row_dot<kD>(o + e, dout + e);
#pragma unroll
        for (int sft = 16; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
        dl = -acc;
        const float lv = lse[(size_t)h * total + tok];
        l2 = (lv == -INFINITY) ? -INFINITY : -lv * 1.4426950408889634f;
        if (dq_acc) zero_row_part<kD>(dq_acc + e);
      }
    }
    if (lane == 0) {
      ndelta[r] = dl;
      nlse2[r] = l2;
    }
  }
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (long long t = tid; t < n_tickets; t += (long long)gridDim.x * blockDim.x) tickets[t] = 0;
}

// ------------------------------------------------------------ main kernel --

// One work unit: key block n (128 keys) of one (batch entry or packed
// sequence b, key/value head); its steps run over the query heads of the
// group and the 64-row query blocks that see at least one of its keys.
struct Unit {
  int b, hk, n;
  int i0;           // first query block
  int nq;           // query blocks per head (of the sequence, from i0)
  int steps;        // group * nq
  int qbase, kbase; // row of the sequence's first query / key in the [rows, H, D] arrays
  int lq, lk;       // query / key count of the sequence
  long long rt;     // row-term index of the sequence's first row for head 0 (+ h * sq_pad per head)
  long long tk;     // ticket index of its first query block for head 0 (+ h * nqb per head)
};

// Work units of the call.  Packed layout: the plan kernel has stored the
// number of 128-key blocks over all sequences (0 if the offsets are invalid).
template <bool PACKED>
__device__ __forceinline__ int total_units_of(const BwdParams& p) {
  if constexpr (PACKED) return p.plan[2 * p.B + 2] * p.Hkv;
  else return ((p.Sk + kBN - 1) / kBN) * p.B * p.Hkv;
}

// Per-sequence geometry of a unit.  The dense instantiation derives it from
// the call's parameters instead of carrying it in registers.
template <bool PACKED> FA_DEV int u_qbase(const Unit& w, const BwdParams& p) { return PACKED ? w.qbase : w.b * p.Sq; }
template <bool PACKED> FA_DEV int u_kbase(const Unit& w, const BwdParams& p) { return PACKED ? w.kbase : w.b * p.Sk; }
template <bool PACKED> FA_DEV int u_lq(const Unit& w, const BwdParams& p) { return PACKED ? w.lq : p.Sq; }
template <bool PACKED> FA_DEV int u_lk(const Unit& w, const BwdParams& p) { return PACKED ? w.lk : p.Sk; }
template <bool PACKED> FA_DEV size_t u_rt(const Unit& w, const BwdParams& p) {
  return PACKED ? size_t(w.rt) : size_t(w.b) * p.Hq * p.sq_pad;
}
template <bool PACKED> FA_DEV size_t u_tk(const Unit& w, const BwdParams& p) {
  return PACKED ? size_t(w.tk) : size_t(w.b) * p.Hq * p.nqb;
}

template <bool PACKED>
__device__ __forceinline__ Unit decode_unit(int u, const BwdParams& p) {
  Unit w;
  if constexpr (PACKED) {
    // the order table written by the plan kernel (longest first; block
    // n - 1 of a pair always has the smaller unit index)
    const int2 e = p.order[u];
    w.hk = e.x / kMaxPackedSeqs;
    w.b = e.x % kMaxPackedSeqs;
    w.n = e.y;
    w.qbase = w.kbase = p.cu_seqlens[w.b];
    w.lq = w.lk = p.cu_seqlens[w.b + 1] - w.qbase;
    w.rt = p.plan[p.B + 1 + w.b];   // padded-row prefix (multiple of 64)
    w.tk = w.rt / kBM;
  } else {
    // Units in groups of g = sched_group (batch, kv head) pairs; within a
    // group key block n ascends, each n over the group's heads.  Under a
    // causal mask block n sees the most query rows when n is small, so the
    // order is longest first within each group, and the few consecutive key
    // blocks of a head in flight at one time move through the same query
    // rows a few blocks apart (L2 reuse of Q / dO rows and dQ-accumulator
    // slices).  g = 1 is head-major (no mask: all units equally long);
    // deterministic mode uses g = all heads (key-block-major), which puts a
    // block's predecessor in the ordered dQ additions far ahead.
    const int nkv = (p.Sk + kBN - 1) / kBN;
    const int nbh = p.B * p.Hkv;
    const int g = p.sched_group;
    const int grp = u / (g * nkv), r = u % (g * nkv);
    const int gh = min(g, nbh - grp * g);   // heads in this (possibly last, smaller) group
    const int bh = grp * g + r % gh;
    w.n = r / gh;
    w.b = bh / p.Hkv;
    w.hk = bh % p.Hkv;
  }
  const int lq = u_lq<PACKED>(w, p), lk = u_lk<PACKED>(w, p);
  const int nqb = (lq + kBM - 1) / kBM;
  int i0 = 0;
  if (p.causal) {
    // query row q sees key j iff j <= q + (lk - lq); block i reaches key
    // 128 n iff 64 i + 63 + (lk - lq) >= 128 n
    const int x = kBN * w.n - (lk - lq) - (kBM - 1);
    i0 = x <= 0 ? 0 : (x + kBM - 1) / kBM;
  }
  w.i0 = i0;
  w.nq = nqb > i0 ? nqb - i0 : 0;
  w.steps = p.group * w.nq;
  return w;
}

// Query block of step s of a unit (steps run over the group's query heads,
// each over the unit's query blocks, first to last or last to first).
FA_DEV int step_block(const Unit& w, int s, const BwdParams& p) {
  const int r = s % w.nq;
  return w.i0 + (p.rev_blocks ? w.nq - 1 - r : r);
}

template <int kD>
struct Shared {
  using L = Layout<kD>;
  uint8_t* base;
  uint32_t sbase;
  FA_DEV uint32_t bar(int i) const { return sbase + L::kBars + 8 * i; }
  FA_DEV uint32_t kv_full() const { return bar(0); }
  FA_DEV uint32_t kv_empty() const { return bar(1); }
  FA_DEV uint32_t qd_full(int s) const { return bar(2 + s); }   // dO and the row terms landed
  FA_DEV uint32_t q_full(int s) const { return bar(18 + 2 * kStages + s); }   // Q landed
  FA_DEV uint32_t ring_full(int r) const { return bar(18 + 3 * kStages + r); }
  FA_DEV uint32_t ring_empty(int r) const { return bar(18 + 3 * kStages + kRing + r); }
  FA_DEV uint32_t ring(int r) const { return sbase + L::kMisc + 16 + 4 * r; }   // announced unit indices
  FA_DEV uint32_t qd_empty(int s) const { return bar(2 + kStages + s); }
  // per TMEM score buffer b (steps alternate buffers)
  FA_DEV uint32_t s_full(int b) const { return bar(2 + 2 * kStages + b); }
  FA_DEV uint32_t p_ready(int b) const { return bar(4 + 2 * kStages + b); }
  FA_DEV uint32_t dq_full(int b) const { return bar(6 + 2 * kStages + b); }
  FA_DEV uint32_t dq_empty(int b) const { return bar(8 + 2 * kStages + b); }
  // per shared-memory dS buffer
  FA_DEV uint32_t ds_free(int b) const { return bar(10 + 2 * kStages + b); }
  FA_DEV uint32_t acc_full() const { return bar(12 + 2 * kStages); }
  FA_DEV uint32_t acc_empty() const { return bar(13 + 2 * kStages); }
  // per dQ staging tile (half a query block each)
  FA_DEV uint32_t dqs_full(int b) const { return bar(14 + 2 * kStages + b); }   // written (128 arrivals)
  FA_DEV uint32_t dqs_free(int b) const { return bar(16 + 2 * kStages + b); }   // read by the TMA unit
  FA_DEV float* dq_stage(int b) const {
    return reinterpret_cast<float*>(base + L::kDqStage + b * L::kDqStageBytes);
  }
  FA_DEV uint32_t dq_stage_addr(int b) const { return sbase + L::kDqStage + b * L::kDqStageBytes; }
  FA_DEV uint32_t abort() const { return sbase + L::kMisc + 4; }
  FA_DEV uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + L::kMisc); }
  FA_DEV uint32_t stage(int s) const { return sbase + L::kStage0 + s * L::kStageStride; }
  FA_DEV uint32_t row_terms(int s) const { return sbase + L::kRowTerms + s * L::kRowTermBytes; }
  FA_DEV const float* stage_nlse2(int s) const {
    return reinterpret_cast<const float*>(base + L::kRowTerms + s * L::kRowTermBytes);
  }
  FA_DEV const float* stage_ndelta(int s) const { return stage_nlse2(s) + kBM; }
  FA_DEV uint32_t ds(int b) const { return sbase + L::kDs + b * L::kDsBytes; }
  FA_DEV uint8_t* ds_ptr(int b) const { return base + L::kDs + b * L::kDsBytes; }
};

// TMEM columns.  Two score buffers b = 0, 1 (steps alternate): S^T at
// 128 b, dP^T at 128 b + 64.  After a step's dS^T has been consumed by the dK
// product, its dQ^T product is written over the dP^T columns of the same
// buffer, so the next S^T into the buffer need not wait for its read-out.
constexpr uint32_t kColBuf = 128, kColDPoff = 64, kColDV = 256, kColDK = 384;

// Work schedule.  Static: CTA c takes units c, c + grid, ...  Dynamic: the
// producer claims units from a counter in global memory (atomicAdd, so SMs
// that finish early take more) and announces them, in claim order, through
// a small ring in shared memory that every other role reads.  -1 ends it.
template <int kD, bool DYN>
FA_DEV int next_unit(const Shared<kD>& sh, int k, const BwdParams& p, int site, int total_units) {
  if constexpr (!DYN) {
    const int u = (int)blockIdx.x + k * (int)gridDim.x;
    return u < total_units ? u : -1;
  }
  const int slot = k % kRing;
  if (!mbar_wait_bounded(sh.ring_full(slot), (k / kRing) & 1, sh.abort(), &g_err, site, p.wait_limit_ns)) return -1;
  const int u = ld_shared_volatile(sh.ring(slot));
  mbar_arrive(sh.ring_empty(slot));
  return u;
}

template <int kD, bool PACKED, bool DYN>
__device__ void producer_role(const Shared<kD>& sh, const CUtensorMap* tq, const CUtensorMap* tk,
                              const CUtensorMap* tv, const CUtensorMap* tdo, const BwdParams& p,
                              const int total_units) {
  uint32_t sit = 0, ukv = 0;
  for (int k = 0;; ++k) {
    int u;
    if constexpr (DYN) {
      u = atomicAdd(p.sched, 1);
      if (u < 0 || u >= total_units) u = -1;
      const int slot = k % kRing;
      if (!mbar_wait_bounded(sh.ring_empty(slot), ((k / kRing) & 1) ^ 1, sh.abort(), &g_err, kSiteProdKV,
                             p.wait_limit_ns))
        return;
      st_shared(sh.ring(slot), u);
      mbar_arrive(sh.ring_full(slot));
    } else {
      u = (int)blockIdx.x + k * (int)gridDim.x;
      if (u >= total_units) u = -1;
    }
    if (u < 0) break;
    const Unit w = decode_unit<PACKED>(u, p);
    if (w.steps == 0) continue;
    if (!mbar_wait_bounded(sh.kv_empty(), (ukv & 1) ^ 1, sh.abort(), &g_err, kSiteProdKV, p.wait_limit_ns)) return;
    mbar_arrive_expect_tx(sh.kv_full(), 2 * Layout<kD>::kKTile);
    const int krow = u_kbase<PACKED>(w, p) + kBN * w.n;
#pragma unroll
    for (int c = 0; c < kD / 64; ++c) {
      tma_load_3d(sh.sbase + Layout<kD>::kK + c * Layout<kD>::kKChunk, tk, sh.kv_full(), c * 64, w.hk, krow);
      tma_load_3d(sh.sbase + Layout<kD>::kV + c * Layout<kD>::kKChunk, tv, sh.kv_full(), c * 64, w.hk, krow);
    }
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int h = w.hk * p.group + s / w.nq;
      const int i = step_block(w, s, p);
      const int st = sit % kStages;
      if (!mbar_wait_bounded(sh.qd_empty(st), ((sit / kStages) & 1) ^ 1, sh.abort(), &g_err, kSiteProdQ,
                             p.wait_limit_ns))
        return;
      // Q on its own barrier (the S^T product needs nothing else), then dO
      // and the row terms
      mbar_arrive_expect_tx(sh.q_full(st), Layout<kD>::kQTile);
      mbar_arrive_expect_tx(sh.qd_full(st), Layout<kD>::kQTile + 2 * kBM * 4);
      const int qrow = u_qbase<PACKED>(w, p) + kBM * i;
      const uint32_t sb = sh.stage(st);
#pragma unroll
      for (int c = 0; c < kD / 64; ++c) tma_load_3d(sb + c * Layout<kD>::kQChunk, tq, sh.q_full(st), c * 64, h, qrow);
#pragma unroll
      for (int c = 0; c < kD / 64; ++c)
        tma_load_3d(sb + Layout<kD>::kQTile + c * Layout<kD>::kQChunk, tdo, sh.qd_full(st), c * 64, h, qrow);
      const size_t roff = u_rt<PACKED>(w, p) + size_t(h) * p.sq_pad + size_t(kBM) * i;
      bulk_load(sh.row_terms(st), p.nlse2 + roff, kBM * 4, sh.qd_full(st));
      bulk_load(sh.row_terms(st) + kBM * 4, p.ndelta + roff, kBM * 4, sh.qd_full(st));
    }
    ++ukv;
  }
}

// Unrolled K steps (K = D in 16-wide steps) of S^T = K Q^T or dP^T = V dO^T;
// both operands K-major: step kk reads 64-wide chunk kk/4 at byte 32*(kk%4).
template <int kD, int KK>
FA_DEV void score_steps(uint32_t d, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi, uint32_t idesc) {
  if constexpr (KK < kD / 16) {
    constexpr uint32_t oa = ((KK >> 2) * Layout<kD>::kKChunk + (KK & 3) * 32) >> 4;
    constexpr uint32_t ob = ((KK >> 2) * Layout<kD>::kQChunk + (KK & 3) * 32) >> 4;
    mma_ss_w<oa, ob>(d, alo, ahi, blo, bhi, idesc, KK > 0 ? 1u : 0u);
    score_steps<kD, KK + 1>(d, alo, ahi, blo, bhi, idesc);
  }
}
// Unrolled K steps (64 queries in 16-wide steps) of dV += P^T dO and
// dK += dS^T Q: A in TMEM (8 columns per step; queries 0-31 in columns
// 0-15 and queries 32-63 in columns 32-47 of the region, as the two
// elementwise warpgroups write them), B MN-major (2048 B per step).
template <int KK>
FA_DEV void grad_steps(uint32_t d_dv, uint32_t d_dk, uint32_t a_p, uint32_t a_ds, uint32_t golo, uint32_t gohi,
                       uint32_t qlo, uint32_t qhi, uint32_t idesc, uint32_t acc) {
  if constexpr (KK < kBM / 16) {
    constexpr uint32_t ca = KK * 8 + (KK >= 2 ? 16 : 0);
    mma_ts_w<ca, KK * 128>(d_dv, a_p, golo, gohi, idesc, KK > 0 ? 1u : acc);
    mma_ts_w<ca, KK * 128>(d_dk, a_ds, qlo, qhi, idesc, KK > 0 ? 1u : acc);
    grad_steps<KK + 1>(d_dv, d_dk, a_p, a_ds, golo, gohi, qlo, qhi, idesc, acc);
  }
}
// Unrolled K steps (128 keys in 16-wide steps) of dQ^T = K^T dS^T: both
// operands MN-major, 16 key rows = 2048 B per step.
template <int KK>
FA_DEV void dq_steps(uint32_t d_dq, uint32_t klo, uint32_t khi, uint32_t slo, uint32_t shi, uint32_t idesc) {
  if constexpr (KK < kBN / 16) {
    mma_ss_w<KK * 128, KK * 128>(d_dq, klo, khi, slo, shi, idesc, KK > 0 ? 1u : 0u);
    dq_steps<KK + 1>(d_dq, klo, khi, slo, shi, idesc);
  }
}

// MMA issuer: the whole warp runs this, converged; an elected lane issues.
template <int kD, bool PACKED, bool DYN, bool DQ>
__device__ void mma_role(const Shared<kD>& sh, const uint32_t tmem, const BwdParams& p, const int total_units) {
  constexpr uint32_t kIdS = idesc_bf16_f32(kBN, kBM, false, false);   // S^T, dP^T: 128 keys x 64 queries
  constexpr uint32_t kIdG = idesc_bf16_f32(kBN, kD, false, true);     // dV, dK: A in TMEM, B MN-major
  // dQ^T: A = K^T, B = dS^T; always M = 128 rows: with kD = 64 the second
  // 64 rows read the next tile in shared memory (V) and are never used
  constexpr uint32_t kIdQ = idesc_bf16_f32(128, kBM, true, true);
  const uint32_t kb = sh.sbase + Layout<kD>::kK, vb = sh.sbase + Layout<kD>::kV;
  const uint64_t dk_kmaj = sdesc_sw128(kb, 16, 1024), dv_kmaj = sdesc_sw128(vb, 16, 1024);
  const uint64_t dk_mn = sdesc_sw128(kb, Layout<kD>::kKChunk, 1024);
  uint32_t sit = 0, ukv = 0;

  auto wait = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    if (!mbar_wait_bounded(bar, parity, sh.abort(), &g_err, site, p.wait_limit_ns)) return false;
    tc_fence_after();
    return true;
  };
  // Scores of global step t into buffer t & 1.  S^T may go first, before the
  // dQ^T that step t - 2 wrote over the dP^T columns has been read out (the
  // S^T product then covers that read-out), or after that wait (when the dQ
  // warpgroup is paced by the additions, queueing S^T ahead of it can delay
  // the dQ product of the current step); dP^T always waits for it.
  auto scores = [&](uint32_t t) -> bool {
    const int buf = t & 1, st = t % kStages;
    const uint32_t ph = (t / kStages) & 1;
    if (!wait(sh.q_full(st), ph, kSiteMmaQ)) return false;
    if (DQ && !p.scores_first && !wait(sh.dq_empty(buf), ((t >> 1) & 1) ^ 1, kSiteMmaDq)) return false;
    const uint64_t dq = sdesc_sw128(sh.stage(st), 16, 1024);
    score_steps<kD, 0>(tmem + kColBuf * buf, desc_lo(dk_kmaj), desc_hi(dk_kmaj), desc_lo(dq), desc_hi(dq), kIdS);
    if (DQ && p.scores_first && !wait(sh.dq_empty(buf), ((t >> 1) & 1) ^ 1, kSiteMmaDq)) return false;
    if (!wait(sh.qd_full(st), ph, kSiteMmaQ)) return false;
    const uint64_t dg = sdesc_sw128(sh.stage(st) + Layout<kD>::kQTile, 16, 1024);
    score_steps<kD, 0>(tmem + kColBuf * buf + kColDPoff, desc_lo(dv_kmaj), desc_hi(dv_kmaj), desc_lo(dg), desc_hi(dg),
                   kIdS);
    mma_commit_w(sh.s_full(buf));
    return true;
  };

  for (int k = 0;; ++k) {
    const int u = next_unit<kD, DYN>(sh, k, p, kSiteMmaKV, total_units);
    if (u < 0) break;
    const Unit w = decode_unit<PACKED>(u, p);
    if (w.steps == 0) continue;
    if (!wait(sh.kv_full(), ukv & 1, kSiteMmaKV)) return;
    if (!scores(sit)) return;
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int st = sit % kStages, buf = sit & 1;
      // next step's scores first, so they are computed while the
      // elementwise pass of this step runs
      if (s + 1 < w.steps && !scores(sit + 1)) return;
      if (!wait(sh.p_ready(buf), (sit >> 1) & 1, kSiteMmaP)) return;
      if (s == 0 && ukv > 0 && !wait(sh.acc_empty(), (ukv - 1) & 1, kSiteMmaAcc)) return;
      // dV += P^T dO_i, dK += dS^T Q_i (B MN-major: D contiguous, 64-wide
      // chunks 8 KB apart)
      const uint64_t dgo = sdesc_sw128(sh.stage(st) + Layout<kD>::kQTile, Layout<kD>::kQChunk, 1024);
      const uint64_t dqq = sdesc_sw128(sh.stage(st), Layout<kD>::kQChunk, 1024);
      grad_steps<0>(tmem + kColDV, tmem + kColDK, tmem + kColBuf * buf, tmem + kColBuf * buf + kColDPoff,
                    desc_lo(dgo), desc_hi(dgo), desc_lo(dqq), desc_hi(dqq), kIdG, s > 0 ? 1u : 0u);
      mma_commit_w(sh.qd_empty(st));
      if constexpr (DQ) {
        // dQ_i^T = K^T dS^T over the dP^T columns of this buffer (its dS^T
        // has just been read by the dK product, issued before): M = D (K
        // MN-major, chunks 16 KB apart), N = 64 queries (dS^T MN-major),
        // K = 128 keys
        const uint64_t dsd = sdesc_sw128(sh.ds(buf), Layout<kD>::kDsBytes, 1024);
        dq_steps<0>(tmem + kColBuf * buf + kColDPoff, desc_lo(dk_mn), desc_hi(dk_mn), desc_lo(dsd), desc_hi(dsd),
                    kIdQ);
        mma_commit_w(sh.dq_full(buf));
        mma_commit_w(sh.ds_free(buf));
      }
    }
    mma_commit_w(sh.acc_full());
    mma_commit_w(sh.kv_empty());
    ++ukv;
  }
}

// P / dS warpgroups: thread = key row kr of the unit's key block; warpgroup
// H handles query columns [32 H, 32 H + 32) of each 64-row step, so two
// warpgroups (one warp per scheduler each) share the elementwise work.
template <int kD, bool PACKED, bool DYN, bool DQ, int H>
__device__ void elementwise_role(const Shared<kD>& sh, const uint32_t tmem, const BwdParams& p,
                                 const int total_units) {
  constexpr int kC0 = 32 * H;   // first query column of this warpgroup
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kr = (warp & 3) * 32 + lane;
  const uint32_t tl = tmem + (uint32_t((warp & 3) * 32) << 16);
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = pk2(sl2, sl2);
  uint32_t sit = 0;
  for (int k = 0;; ++k) {
    const int u = next_unit<kD, DYN>(sh, k, p, kSiteEsQ, total_units);
    if (u < 0) break;
    const Unit w = decode_unit<PACKED>(u, p);
    const int key = kBN * w.n + kr;
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int i = step_block(w, s, p);
      const int st = sit % kStages, buf = sit & 1;
      if (!mbar_wait_bounded(sh.qd_full(st), (sit / kStages) & 1, sh.abort(), &g_err, kSiteEsQ, p.wait_limit_ns))
        return;
      if (!mbar_wait_bounded(sh.s_full(buf), (sit >> 1) & 1, sh.abort(), &g_err, kSiteEsS, p.wait_limit_ns))
        return;
      tc_fence_after();
      const uint32_t tb = tl + kColBuf * buf;
      uint32_t sr[32], dr[32];
      tmem_ld32(tb + kC0, sr);
      tmem_ld32(tb + kColDPoff + kC0, dr);
      tmem_ld_wait();
      tmem_ld_fence(sr);
      tmem_ld_fence(dr);
      // columns c < cmin are masked: keys past the sequence's keys, or
      // (causal) queries that come before this key
      int cmin = 0;
      if (key >= u_lk<PACKED>(w, p)) cmin = kBM;
      else if (p.causal) cmin = min(kBM, max(0, key - (u_lk<PACKED>(w, p) - u_lq<PACKED>(w, p)) - kBM * i));
      // row terms of the 32 columns: 16-byte broadcast loads (every lane
      // reads the same address), four columns per shared-memory wavefront
      const float4* nl = reinterpret_cast<const float4*>(sh.stage_nlse2(st) + kC0);
      const float4* nd = reinterpret_cast<const float4*>(sh.stage_ndelta(st) + kC0);
      uint32_t pp[16], dd[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float4 l4 = nl[c / 4], d4 = nd[c / 4];
        const float2 l2 = (c & 2) ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
        const float2 d2 = (c & 2) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
        const uint64_t x = fma2(pk2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2x2, pk2(l2.x, l2.y));
        float x0, x1;
        up2(x, x0, x1);
        float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
        if (kC0 + c < cmin) p0 = 0.0f;
        if (kC0 + c + 1 < cmin) p1 = 0.0f;
        const uint64_t g = add2(pk2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), pk2(d2.x, d2.y));
        float s0, s1;
        up2(mul2(pk2(p0, p1), g), s0, s1);
        pp[c / 2] = pack_bf16x2(p0, p1);
        dd[c / 2] = pack_bf16x2(s0, s1);
      }
      // P^T and dS^T as BF16 into TMEM (A operands of dV and dK): this
      // warpgroup's query pairs (32 H + 2 q, 32 H + 2 q + 1) in column 32 H + q
      // of the S^T / dP^T region -- inside the columns this warpgroup has
      // just read, never in the other warpgroup's
      tmem_st16(tb + kC0, pp);
      tmem_st16(tb + kColDPoff + kC0, dd);
      // dS^T into shared memory (B operand of dQ^T): row kr, 128-byte rows,
      // 16-byte chunk j (queries 8 j .. 8 j + 7) stored at chunk j ^ (kr mod 8)
      if constexpr (DQ) {
        if (!mbar_wait_bounded(sh.ds_free(buf), ((sit >> 1) & 1) ^ 1, sh.abort(), &g_err, kSiteEsDs,
                               p.wait_limit_ns))
          return;
        uint8_t* row = sh.ds_ptr(buf) + kr * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(row + (((4 * H + j) ^ (kr & 7)) << 4)) =
              make_uint4(dd[4 * j], dd[4 * j + 1], dd[4 * j + 2], dd[4 * j + 3]);
      }
      tmem_st_wait();
      if constexpr (DQ) fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(sh.p_ready(buf));
    }
  }
}

// dQ warpgroup: thread = feature d.  Per step it moves dQ_i^T from TMEM to the
// two row-major FP32 staging tiles in shared memory (queries 0-31 and 32-63
// of the block, 32 x 128 each); the reduce issuer adds each into the FP32
// accumulator.  At the end of a unit it writes dK (scaled) and dV.
template <int kD, bool PACKED, bool DYN, bool DQ>
__device__ void dq_role(const Shared<kD>& sh, const uint32_t tmem, const BwdParams& p, const int total_units) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wq = warp & 3;
  const int d = wq * 32 + lane;           // dQ^T lane = feature; dK/dV lane = key row
  const uint32_t tl = tmem + (uint32_t(wq * 32) << 16);
  uint32_t sit = 0, ukv = 0;
  __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk);
  __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(p.dv);
  for (int k = 0;; ++k) {
    const int u = next_unit<kD, DYN>(sh, k, p, kSiteDqFull, total_units);
    if (u < 0) break;
    const Unit w = decode_unit<PACKED>(u, p);
    bool stop = false;
    for (int s = 0; DQ && s < w.steps; ++s, ++sit) {
      const int buf = sit & 1;
      if (!mbar_wait_bounded(sh.dq_full(buf), (sit >> 1) & 1, sh.abort(), &g_err, kSiteDqFull, p.wait_limit_ns)) {
        stop = true;
        break;
      }
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(tl + kColBuf * buf + kColDPoff, v[0]);
      tmem_ld32(tl + kColBuf * buf + kColDPoff + 32, v[1]);
      tmem_ld_wait();
      tmem_ld_fence(v[0]);
      tmem_ld_fence(v[1]);
      tc_fence_before();
      mbar_arrive(sh.dq_empty(buf));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // tile `half` of step sit is the sit-th use of that buffer
        if (!mbar_wait_bounded(sh.dqs_free(half), (sit & 1) ^ 1, sh.abort(), &g_err, kSiteDqFull,
                               p.wait_limit_ns)) {
          stop = true;
          break;
        }
        float* stage = sh.dq_stage(half);
#pragma unroll
        for (int c = 0; c < kDqRows; ++c)
          if (d < kD) stage[c * kD + d] = __uint_as_float(v[half][c]);   // lanes >= kD: padding rows
        fence_proxy_async_smem();
        mbar_arrive(sh.dqs_full(half));
      }
      if (stop) break;
    }
    if (stop || ld_shared_volatile(sh.abort())) break;
    // epilogue of the unit: dV and scale * dK rows in BF16
    const int key = kBN * w.n + d;
    const bool valid = key < u_lk<PACKED>(w, p);
    const size_t roff = ((size_t(u_kbase<PACKED>(w, p)) + key) * p.Hkv + w.hk) * kD;
    if (w.steps > 0) {
      if (!mbar_wait_bounded(sh.acc_full(), ukv & 1, sh.abort(), &g_err, kSiteAcc, p.wait_limit_ns)) break;
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
          // 32 columns of this key row: 64 contiguous bytes, as two 32-byte
          // stores (whole L2 sectors) when dK and dV allow it, else four
          // 16-byte ones
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
          if (p.dkv_st32) {
            st_global_v8(dst + c * 32, pk);
            st_global_v8(dst + c * 32 + 16, pk + 8);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              reinterpret_cast<uint4*>(dst + c * 32)[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      }
    }
    if (w.steps > 0) {
      tc_fence_before();
      mbar_arrive(sh.acc_empty());
      ++ukv;
    }
  }
}

// dQ reduce issuer (one thread): adds each staging tile into the FP32
// accumulator with one TMA bulk tensor reduce-add.  Tile b of step t is freed
// once the unit has read it, which is known when at most one later group is
// still reading (the other tile), so one tile is always being written while
// the other is read.  Out-of-range rows are skipped by the unit; rows of a
// padded query block that belong to the next sequence receive exact zeros,
// since their weights are 0.
//
// Deterministic mode: key blocks add into each (b, h, i) in ascending order
// n = 0, 1, ..., one ticket per (b, h, i) holding the next block allowed to
// add.  A step's ticket is released one step late, once the next step's two
// reductions are issued and at most those two are still pending, so the
// completion latency of the additions is not paid per step.  Waits point
// only from key block n to block n - 1 of the same head, which has the
// smaller unit index in every schedule, and no ticket is held across units,
// so the waits cannot form a cycle.
template <int kD, bool PACKED, bool DYN, bool DQ>
__device__ void reduce_role(const Shared<kD>& sh, const CUtensorMap* tdq, const BwdParams& p, const int total_units) {
  if constexpr (!DQ) {
    // dQ is computed by its own kernel: only the unit announcements of the
    // dynamic schedule are acknowledged here
    if constexpr (DYN)
      for (int k = 0;; ++k)
        if (next_unit<kD, DYN>(sh, k, p, kSiteDqFull, total_units) < 0) break;
    return;
  }
  uint32_t sit = 0;
  bool pending1 = false;   // tile 1 of the previous step is still being read
  int* held = nullptr;     // deterministic mode: ticket of the previous step, not yet released
  int held_next = 0;
  // The bulk wait before a release returns only once the additions are
  // complete, a proxy fence orders them (made by the TMA unit) before the
  // release store, and the next block's additions are issued only after an
  // acquire load has seen that store and a proxy fence; so the additions to
  // an address are applied in ticket order.  A full fence before the store
  // measured 13% slower; the proxy fences cost nothing measurable.
  auto release_held = [&]() {
    fence_proxy_async_global();
    st_release_gpu(held, held_next);
    held = nullptr;
  };
  for (int k = 0;; ++k) {
    const int u = next_unit<kD, DYN>(sh, k, p, kSiteDqFull, total_units);
    if (u < 0) break;
    const Unit w = decode_unit<PACKED>(u, p);
    for (int s = 0; s < w.steps; ++s, ++sit) {
      const int h = w.hk * p.group + s / w.nq;
      const int i = step_block(w, s, p);
      int* ticket = nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (!mbar_wait_bounded(sh.dqs_full(half), sit & 1, sh.abort(), &g_err, kSiteDqFull, p.wait_limit_ns))
          goto done;
        if (p.deterministic && half == 0) {
          ticket = p.tickets + u_tk<PACKED>(w, p) + size_t(h) * p.nqb + i;
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(ticket) != w.n) {
            if (ld_shared_volatile(sh.abort()) || globaltimer_ns() - t0 > p.wait_limit_ns) {
              if (atomicCAS(&g_err.status, 0, FA_ERR_TIMEOUT) == 0) atomicExch(&g_err.site, kSiteDqTicket);
              st_shared(sh.abort(), 1);
              goto done;
            }
            __nanosleep(64);
          }
          fence_proxy_async_global();
        }
        tma_reduce_add_3d(tdq, sh.dq_stage_addr(half), 0, h, u_qbase<PACKED>(w, p) + kBM * i + kDqRows * half);
        bulk_commit_group();
        bulk_wait_group_read1();   // every group but this one has been read
        if (half == 0) {
          if (pending1) mbar_arrive(sh.dqs_free(1));
          pending1 = false;
        } else {
          mbar_arrive(sh.dqs_free(0));
          pending1 = true;
        }
      }
      if (p.deterministic) {
        if (held) {
          bulk_wait_group2();   // the previous step's two additions are complete
          release_held();
        }
        held = ticket;
        held_next = w.n + 1;
      }
    }
    if (held) {
      // end of the unit: no ticket is held while waiting on another head's
      bulk_wait_group0();
      release_held();
    }
  }
done:
  bulk_wait_group0();   // outstanding reductions finish before the CTA exits
  if (held) release_held();
}

template <int kD, bool PACKED, bool DYN, bool DQ>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqacc, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x / 32;
  Shared<kD> sh;
  sh.base = smem;
  sh.sbase = smem_u32(smem);
  if (threadIdx.x == 0) {
    mbar_init(sh.kv_full(), 1);
    mbar_init(sh.kv_empty(), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sh.qd_full(s), 1);
      mbar_init(sh.q_full(s), 1);
      mbar_init(sh.qd_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.s_full(b), 1);
      mbar_init(sh.p_ready(b), 256);
      mbar_init(sh.dq_full(b), 1);
      mbar_init(sh.dq_empty(b), 128);
      mbar_init(sh.ds_free(b), 1);
    }
    mbar_init(sh.acc_full(), 1);
    mbar_init(sh.acc_empty(), 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(sh.dqs_full(b), 128);
      mbar_init(sh.dqs_free(b), 1);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(sh.ring_full(r), 1);
      mbar_init(sh.ring_empty(r), kRingReaders);
    }
    st_shared(sh.abort(), 0);
    fence_barrier_init();
  }
  if (warp == 8 && (threadIdx.x % 32) == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dqacc);
  }
  if (warp == 9) {
    tmem_alloc(sh.tmem_slot(), 512);
    tmem_relinquish();
  }
  const int total_units = total_units_of<PACKED>(p);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot();
  // register split (sums to the 512 x 128 the block was launched with)
  if (warp < 4) {
    reg_alloc<160>();
    elementwise_role<kD, PACKED, DYN, DQ, 0>(sh, tmem, p, total_units);
  } else if (warp < 8) {
    dq_role<kD, PACKED, DYN, DQ>(sh, tmem, p, total_units);
  } else if (warp < 12) {
    reg_dealloc<64>();
    if (warp == 8) {
      if ((threadIdx.x % 32) == 0) producer_role<kD, PACKED, DYN>(sh, &tm_q, &tm_k, &tm_v, &tm_do, p, total_units);
    } else if (warp == 9) {
      mma_role<kD, PACKED, DYN, DQ>(sh, tmem, p, total_units);   // converged warp; one elected lane issues
    } else if (warp == 10) {
      if ((threadIdx.x % 32) == 0) reduce_role<kD, PACKED, DYN, DQ>(sh, &tm_dqacc, p, total_units);
    }
  } else {
    reg_alloc<160>();
    elementwise_role<kD, PACKED, DYN, DQ, 1>(sh, tmem, p, total_units);
  }
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

}  // namespace bwd

namespace {

// The main kernel, with (DQ) or without its dQ product.
template <int kD, bool DQ>
fa_status launch_main(const BwdLaunch& L, bool packed, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq, cudaStream_t stream) {
  const BwdParams& p = L.p;
  fa_status st;
  if ((st = prepare_kernel(reinterpret_cast<const void*>(bwd::bwd_kernel<kD, false, false, DQ>),
                           bwd::Layout<kD>::kDynamic)) != FA_OK ||
      (st = prepare_kernel(reinterpret_cast<const void*>(bwd::bwd_kernel<kD, false, true, DQ>),
                           bwd::Layout<kD>::kDynamic)) != FA_OK ||
      (st = prepare_kernel(reinterpret_cast<const void*>(bwd::bwd_kernel<kD, true, true, DQ>),
                           bwd::Layout<kD>::kDynamic)) != FA_OK)
    return st;
  // packed: the number of key blocks is only known on the device; this
  // bound (every sequence adds at most one partial block) sizes the grid
  const long long units = packed ? ((long long)p.Sk / bwd::kBN + p.B) * p.Hkv
                                 : (long long)((p.Sk + bwd::kBN - 1) / bwd::kBN) * p.B * p.Hkv;
  const int grid = (int)(units < L.num_sms ? units : L.num_sms);
  constexpr int kSmem = bwd::Layout<kD>::kDynamic;
  // packed layouts always use the dynamic schedule (their units differ in
  // length); dense ones as chosen by the caller (sched_dynamic)
  if (packed)
    bwd::bwd_kernel<kD, true, true, DQ><<<grid, bwd::kThreads, kSmem, stream>>>(tq, tk, tv, tdo, tdq, p);
  else if (p.sched_dynamic)
    bwd::bwd_kernel<kD, false, true, DQ><<<grid, bwd::kThreads, kSmem, stream>>>(tq, tk, tv, tdo, tdq, p);
  else
    bwd::bwd_kernel<kD, false, false, DQ><<<grid, bwd::kThreads, kSmem, stream>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int kD>
fa_status launch_bwd_d(const BwdLaunch& L, cudaStream_t stream) {
  const BwdParams& p = L.p;
  const bool packed = p.cu_seqlens != nullptr;
  // rows of the [rows, H, D] arrays
  const int rows_q = packed ? p.Sq : p.B * p.Sq;
  const int rows_k = packed ? p.Sk : p.B * p.Sk;
  fa_status st;

  // pre: (packed: offsets and per-sequence tables,) Delta, LSE2, zero
  // accumulator and tickets
  const long long heads_rt = packed ? (long long)p.Hq : (long long)p.B * p.Hq;
  const long long rows = heads_rt * p.sq_pad;
  // split: dK / dV from the main kernel without its dQ product, dQ from its
  // own kernel (no accumulator, no tickets, no post pass)
  const bool split = L.split_dq && !L.pair;
  float* acc = split ? nullptr : p.dq_acc;
  const long long n_tickets = (p.deterministic && !split) ? heads_rt * p.nqb * 2 : 0;
  long long pre_blocks = (rows * 32 + 255) / 256;
  if (pre_blocks > 16 * L.num_sms) pre_blocks = 16 * L.num_sms;
  if (pre_blocks < 1) pre_blocks = 1;
  if (packed) {
    bwd::plan_kernel<<<1, 1024, 0, stream>>>(p.cu_seqlens, p.B, p.Sq, p.Hkv, p.sched_group, p.plan, p.order);
    bwd::pre_packed_kernel<kD><<<(unsigned)pre_blocks, 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(p.o), reinterpret_cast<const __nv_bfloat16*>(p.dout), p.lse,
        p.cu_seqlens, p.plan, p.ndelta, p.nlse2, acc, p.tickets, n_tickets, p.sched, p.B, p.Hq, p.Sq,
        p.sq_pad);
  } else {
    bwd::pre_kernel<kD><<<(unsigned)pre_blocks, 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(p.o), reinterpret_cast<const __nv_bfloat16*>(p.dout), p.lse,
        p.ndelta, p.nlse2, acc, p.tickets, n_tickets, p.sched, p.B, p.Hq, p.Sq, p.sq_pad);
  }
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;

  if (L.pair && !packed && kD == 128) {
    if ((st = launch_bwd_pair_main(L, stream)) != FA_OK) return st;
  } else {
    CUtensorMap tq, tk, tv, tdo, tdq;
    if ((st = make_tmap_f32_rows_heads_d(&tdq, p.dq_acc, rows_q, p.Hq, p.D, p.D, bwd::kDqRows)) != FA_OK)
      return st;
    if ((st = make_tmap_rows_heads_d(&tq, L.q, rows_q, p.Hq, p.D, bwd::kBM)) != FA_OK) return st;
    if ((st = make_tmap_rows_heads_d(&tdo, p.dout, rows_q, p.Hq, p.D, bwd::kBM)) != FA_OK) return st;
    if ((st = make_tmap_rows_heads_d(&tk, L.k, rows_k, p.Hkv, p.D, bwd::kBN)) != FA_OK) return st;
    if ((st = make_tmap_rows_heads_d(&tv, L.v, rows_k, p.Hkv, p.D, bwd::kBN)) != FA_OK) return st;
    if (split) st = launch_main<kD, false>(L, packed, tq, tk, tv, tdo, tdq, stream);
    else st = launch_main<kD, true>(L, packed, tq, tk, tv, tdo, tdq, stream);
    if (st != FA_OK) return st;
  }
  if (split) return launch_bwd_dq(L, stream);

  // post: dQ = BF16(scale * accumulator)
  const long long n8 = (long long)rows_q * p.Hq * p.D / 8;
  long long post_blocks = (n8 + 255) / 256;
  if (post_blocks > 16 * L.num_sms) post_blocks = 16 * L.num_sms;
  bwd::post_kernel<<<(unsigned)post_blocks, 256, 0, stream>>>(p.dq_acc, reinterpret_cast<__nv_bfloat16*>(p.dq),
                                                              n8, p.scale, packed ? p.plan + 2 * p.B + 3 : nullptr);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

fa_status launch_bwd(const BwdLaunch& L, cudaStream_t stream) {
  if (L.p.D == 128) return launch_bwd_d<128>(L, stream);
  if (L.p.D == 64) return launch_bwd_d<64>(L, stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status bwd_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, bwd::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(bwd::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

// ------------------------------------------------- allocation-free entry --

// Scratch of fa_bwd_noalloc(): a fixed buffer in the library's own device
// memory, so that callers who may not allocate still get a backward pass.
namespace bwd {
static __device__ __align__(256) unsigned char g_static_scratch[FA_BWD_STATIC_SCRATCH_BYTES];
}

// Device address of the buffer in the current CUDA context.  The symbol's
// host-side name is not a device address, and the address belongs to the
// context that loaded the module: it is looked up once per context (with that
// context current) and cached under the context's unique id, so that a
// context created later (after cudaDeviceReset, or a non-primary context made
// current by the caller) gets its own lookup instead of a stale address.
static CUresult current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (!get_current || !get_id) return CUDA_ERROR_NOT_FOUND;
  CUcontext ctx = nullptr;
  const CUresult r = get_current(&ctx);
  if (r != CUDA_SUCCESS) return r;
  if (ctx == nullptr) return CUDA_ERROR_INVALID_CONTEXT;
  return get_id(ctx, id);
}

static fa_status static_scratch_address(void** out) {
  constexpr int kMaxContexts = 64;
  static unsigned long long ids[kMaxContexts] = {};
  static void* addr[kMaxContexts] = {};
  static int n = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  if (current_context_id(&id) == CUDA_SUCCESS) {
    for (int i = 0; i < n; ++i)
      if (ids[i] == id) {
        *out = addr[i];
        return FA_OK;
      }
  }
  // first call in this context (the lookup also initialises the runtime's
  // context when none is current yet)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, bwd::g_static_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
  if (current_context_id(&id) != CUDA_SUCCESS) return FA_ERR_CUDA;
  if (n < kMaxContexts) {
    ids[n] = id;
    addr[n] = p;
    ++n;
  }
  *out = p;
  return FA_OK;
}

}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                    int Sq, int Sk, int D, int causal, float scale, const int* cu_seqlens,
                                    int deterministic, fa_stream_t stream) {
  try {
    const size_t need = fa_bwd_workspace_size(B, Hq, Hkv, Sq, Sk, D, nullptr, cu_seqlens ? Sq : 0, deterministic);
    if (need > FA_BWD_STATIC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {  // need == 0: fa_bwd rejects the arguments below, before any launch
      const fa_status st = fa::static_scratch_address(&scratch);
      if (st != FA_OK) return st;
    }
    // fa_bwd's pre-pass zeroes the accumulator and tickets on every call, so
    // what an earlier call left in the buffer does not matter.
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, causal, scale, cu_seqlens,
                  deterministic, scratch, scratch ? FA_BWD_STATIC_SCRATCH_BYTES : 0, stream);
  } catch (...) {
    return FA_ERR_CUDA;
  }
}
