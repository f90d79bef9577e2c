// Work units over query rows, shared by the forward kernel and the backward's
// dQ kernel: a unit is a pair of 128-row query tiles (256 rows) of one
// (sequence, query head), and the units of a call are visited longest first
// under a causal mask and for packed variable-length batches
// ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", fdeinterviews.com summary, the paragraph on
// longest-first scheduling).
//
// The parameter type Prm needs: B, Hq, Sq, Sk (packed: Sq = Sk = total rows),
// sched_group (dense causal: heads per longest-first group) and cu_seqlens.
#pragma once

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace qs {

constexpr int kTileRows = 128;
constexpr int kPairRows = 2 * kTileRows;

// One work unit.
struct QUnit {
  int h;          // query head
  int pair;       // pair index inside the sequence
  int q_tok0;     // token index (row of the [rows, H, D] view) of the sequence's first query
  int k_tok0;     // same for keys
  int seq_q, seq_k;
  int b;          // batch / sequence index
};

// Packed-length schedule tables (shared memory).  Sequences are sorted by
// length, longest first (ties by index).
struct PackedSched {
  int* start;      // [nseq] first token of the i-th longest sequence
  int* len;        // [nseq] its length
  int* seq;        // [nseq] its index
  int* uprefix;    // [nseq+1] non-causal: units before the i-th longest sequence
  int* gprefix;    // [P+1]   causal: units before pair group k (pair index P-1-k)
  int* header;     // [0] total units, [1] max pairs P, [2] total tokens, [3] bad input
};

// Shared-memory bytes of the packed-length tables.
constexpr int kSchedInts = 3 * kMaxPackedSeqs + (kMaxPackedSeqs + 1) + (kMaxPairsPerSeq + 1) + 4;
constexpr int kSchedBytes = 4 * kSchedInts;

// Units of this CTA: the unit order (longest first) is dealt over the
// persistent grid in rows of G = gridDim.x units, left to right on even rows
// and right to left on odd ones, so a CTA that takes one of the longest units
// of a row takes one of the shortest of the next.  CTA c's units are c,
// 2G - 1 - c, 2G + c, 4G - 1 - c, ...: steps that alternate between
// 2 (G - 1 - c) + 1 and 2 c + 1 (first_unit / next_unit_step below).
// Dealing every row left to right instead leaves CTA 0 with the longest unit
// of every row: on the causal dense workloads that is 4-14% above the mean
// load (training shape B = 2, S = 8192: 14%), against 0-2% for this order
// (computed over the sweep's unit costs).  Measured on GB300 (forward,
// same box): causal B=4 S=4096 +4%, training shape B=2 S=8192 +6%, S=32768
// +6%, but S=1024 (B=32) -3.5% and S=2048 (B=16) -1.1%; so the host asks
// for it (`snake`) for dense causal calls with S >= 4096 only, and otherwise
// every step is G.
FA_DEV int first_step(bool snake) { return snake ? 2 * (int)(gridDim.x - 1 - blockIdx.x) + 1 : (int)gridDim.x; }
FA_DEV int next_step(int d, bool snake) { return snake ? 2 * (int)gridDim.x - d : d; }

// Dense layout: number of units of the call.
template <class Prm>
FA_DEV int dense_units(const Prm& p) {
  return ((p.Sq + kPairRows - 1) / kPairRows) * p.B * p.Hq;
}

template <bool CAUSAL, bool VARLEN, class Prm>
FA_DEV QUnit decode_pair_unit(int u, const Prm& p, const PackedSched& ps) {
  QUnit w;
  if (!VARLEN) {
    const int npairs = (p.Sq + kPairRows - 1) / kPairRows;
    const int BH = p.B * p.Hq;
    int bh;
    if (CAUSAL) {
      // longest first within groups of sched_group (batch, head) pairs: a
      // group's pairs near the end of the sequence (the most key blocks)
      // first, every head of the group at each level, group after group.
      // The groups bound how many heads' K/V are in flight at once, so that
      // the key blocks a head's pairs share stay in L2.
      const int G = p.sched_group;
      const int grp = u / (G * npairs), r = u % (G * npairs);
      const int gh = min(G, BH - grp * G);   // heads of this (possibly last, smaller) group
      w.pair = npairs - 1 - r / gh;
      bh = grp * G + r % gh;
    } else {       // every pair costs the same: keep a head's pairs together
      bh = u / npairs;
      w.pair = u % npairs;
    }
    w.b = bh / p.Hq;
    w.h = bh % p.Hq;
    w.q_tok0 = w.b * p.Sq;
    w.k_tok0 = w.b * p.Sk;
    w.seq_q = p.Sq;
    w.seq_k = p.Sk;
  } else {
    const int nseq = p.B;
    int i;
    if (CAUSAL) {
      // groups of equal pair index, highest first; group k holds pair P-1-k of
      // every sequence that has it (a prefix of the longest-first order)
      const int P = ps.header[1];
      int lo = 0, hi = P - 1;
      while (lo < hi) {  // last k with gprefix[k] <= u
        const int mid = (lo + hi + 1) >> 1;
        if (ps.gprefix[mid] <= u) lo = mid; else hi = mid - 1;
      }
      w.pair = P - 1 - lo;
      const int idx = u - ps.gprefix[lo];
      i = idx / p.Hq;
      w.h = idx % p.Hq;
    } else {
      int lo = 0, hi = nseq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ps.uprefix[mid] <= u) lo = mid; else hi = mid - 1;
      }
      i = lo;
      const int rem = u - ps.uprefix[i];
      const int np = (ps.len[i] + kPairRows - 1) / kPairRows;
      w.h = rem / np;
      w.pair = rem % np;
    }
    w.b = ps.seq[i];
    w.q_tok0 = ps.start[i];
    w.k_tok0 = ps.start[i];
    w.seq_q = ps.len[i];
    w.seq_k = ps.len[i];
  }
  return w;
}

// Builds the packed-length tables cooperatively (all threads of the CTA) and
// returns the number of work units.  Invalid offsets are recorded as
// FA_ERR_INVALID_ARG in `err` (by block 0) and leave the CTA with no work.
template <class Prm>
__device__ int build_packed_sched(const Prm& p, PackedSched& ps, uint8_t* base, DeviceError* err) {
  const int nseq = p.B;
  ps.start = reinterpret_cast<int*>(base);
  ps.len = ps.start + kMaxPackedSeqs;
  ps.seq = ps.len + kMaxPackedSeqs;
  ps.uprefix = ps.seq + kMaxPackedSeqs;
  ps.gprefix = ps.uprefix + kMaxPackedSeqs + 1;
  ps.header = ps.gprefix + kMaxPairsPerSeq + 1;
  if (threadIdx.x == 0) ps.header[3] = 0;
  __syncthreads();
  // validate: cu[0] == 0, non-decreasing, cu[B] == total, lengths <= limit
  for (int b = threadIdx.x; b < nseq; b += blockDim.x) {
    const int s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
    bool bad = s1 < s0 || (s1 - s0) > kMaxPairsPerSeq * kPairRows;
    if (b == 0) bad |= s0 != 0;
    if (b == nseq - 1) bad |= s1 != p.Sq;
    if (bad) ps.header[3] = 1;
  }
  __syncthreads();
  if (ps.header[3]) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicCAS(&err->status, 0, FA_ERR_INVALID_ARG);
    return 0;
  }
  // rank of each sequence in longest-first order (ties by index)
  for (int b = threadIdx.x; b < nseq; b += blockDim.x) {
    const int Lb = p.cu_seqlens[b + 1] - p.cu_seqlens[b];
    int rank = 0;
    for (int c = 0; c < nseq; ++c) {
      const int Lc = p.cu_seqlens[c + 1] - p.cu_seqlens[c];
      rank += (Lc > Lb) || (Lc == Lb && c < b);
    }
    ps.start[rank] = p.cu_seqlens[b];
    ps.len[rank] = Lb;
    ps.seq[rank] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < nseq; ++i) {
      ps.uprefix[i] = acc;
      acc += ((ps.len[i] + kPairRows - 1) / kPairRows) * p.Hq;
    }
    ps.uprefix[nseq] = acc;
    const int P = nseq ? (ps.len[0] + kPairRows - 1) / kPairRows : 0;
    // causal groups: pair index P-1-k for k = 0..P-1; members are the
    // sequences with more than that many pairs (a prefix of the order)
    int g = 0, members = 0;
    for (int k = 0; k < P; ++k) {
      const int pi = P - 1 - k;   // descending, so the member prefix only grows
      while (members < nseq && (ps.len[members] + kPairRows - 1) / kPairRows > pi) ++members;
      ps.gprefix[k] = g;
      g += members * p.Hq;
    }
    ps.gprefix[P] = g;
    ps.header[0] = acc;   // both orders enumerate the same units
    ps.header[1] = P;
    ps.header[2] = p.Sq;
  }
  __syncthreads();
  return ps.header[0];
}

}  // namespace qs
}  // namespace fa
