// Host-side plumbing shared by the C ABI (fa_api.cu) and the kernel
// translation units: launch descriptors, tensor-map construction and the
// per-translation-unit device error records.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "fa.h"

namespace fa {

// Upper bounds of the packed-length scheduler tables kept in shared memory.
constexpr int kMaxPackedSeqs = 1024;
constexpr int kMaxPairsPerSeq = 1024;   // 256 query rows per pair -> 262,144 tokens

struct FwdParams {
  void* o;                 // BF16 output, same layout as q
  float* lse;              // FP32 log-sum-exp
  const int* cu_seqlens;   // device [B+1] or nullptr
  int B, Hq, Hkv, Sq, Sk;  // packed: Sq = Sk = total tokens
  int group;               // Hq / Hkv
  float scale_log2;        // scale * log2(e)
  float thr;               // lazy-rescale threshold in log2 units
  int stages;              // K/V ring depth (2 .. the kernel's maximum)
  int split_p;             // 1: each half of P (64 keys) is signalled to the MMA warp on its own
  int sched_group;         // dense causal: (batch, head) pairs per group of the longest-first unit order
  int snake;               // deal the units over the grid boustrophedon-wise (q_sched.cuh)
  int o_st32;              // O is 32-byte aligned: its rows are written with 32-byte stores
  unsigned long long wait_limit_ns;
};

struct FwdLaunch {
  const void* q;
  const void* k;
  const void* v;
  FwdParams p;
  int D;
  bool causal;
  int emu_per_16;
  int num_sms;
};

struct BwdParams {
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;     // [B, Sq, Hq, D] fp32
  float* ndelta;     // [B, Hq, sq_pad]  -sum_d dO * O
  float* nlse2;      // [B, Hq, sq_pad]  -lse * log2(e)
  int* tickets;      // [B, Hq, nqb, 2] (packed: [Hq, nqb, 2]) or nullptr
  const int* cu_seqlens;   // packed layout: device [B + 1]; nullptr for dense
  int* plan;         // packed: key-block prefix [B + 1], padded-row prefix [B + 1], total key blocks, status
  int2* order;       // packed: work units in schedule order, {kv head * 1024 + sequence, key block}
  int* sched;        // work-unit counter of the dynamic scheduler (zeroed by the pre pass)
  int sched_group;   // (batch, kv head) / (sequence, kv head) pairs per group of the longest-first unit order
  int sched_dynamic; // 1: units claimed from the counter; 0: CTA c takes units c, c + grid, ...
  int rev_blocks;    // 1: a unit visits its query blocks last to first
  int dkv_st32;      // dK and dV are 32-byte aligned: their rows are written with 32-byte stores
  int scores_first;  // 1: the next step's S^T is issued before waiting for the dQ read-out of its buffer
  int B, Hq, Hkv, Sq, Sk, D;   // packed: Sq = Sk = total rows
  int sq_pad;        // row-term floats per head: dense Sq rounded up to 64, packed Sq rounded up + 64 B
  int nqb;           // tickets per head: sq_pad / 64
  int group;
  int causal;
  int deterministic;
  float scale;
  float scale_log2;
  unsigned long long wait_limit_ns;
};

struct BwdLaunch {
  const void* q;
  const void* k;
  const void* v;
  BwdParams p;
  int num_sms;
  bool pair;       // main kernel on CTA pairs (paired MMAs) rather than single CTAs
  bool split_dq;   // dK / dV from the main kernel without its dQ product, dQ from its own kernel
};

// Workspace carve-up of the backward pass (all offsets 256-byte aligned).
struct BwdWorkspace {
  size_t dq_acc, ndelta, nlse2, plan, order, sched, tickets, total;
  int sq_pad;
};
// Dense: rows = Sq per batch entry; packed: Sq = total rows of B sequences.
BwdWorkspace bwd_workspace_layout(int B, int Hq, int Hkv, int Sq, int D, int deterministic, bool packed);

// 3-D tiled tensor map over a [rows, heads, D] BF16 array (D contiguous) with
// a box of 64 x 1 x box_rows and 128-byte swizzle.
fa_status make_tmap_rows_heads_d(CUtensorMap* map, const void* base, int rows, int heads, int D, int box_rows);
// Same view over an FP32 [rows, heads, D] array, box box_d x 1 x box_rows, no
// swizzle (a row-major staging tile).
fa_status make_tmap_f32_rows_heads_d(CUtensorMap* map, const void* base, int rows, int heads, int D, int box_d,
                                     int box_rows);

// Raises the dynamic shared-memory limit of kernel `func` to `bytes` the
// first time it is launched on the current device (the attribute is per
// device); thread-safe.
fa_status prepare_kernel(const void* func, int bytes);

// Kernel launchers (defined in their translation units).
fa_status launch_fwd(const FwdLaunch& L, cudaStream_t stream);
fa_status launch_bwd(const BwdLaunch& L, cudaStream_t stream);
fa_status launch_bwd_pair_main(const BwdLaunch& L, cudaStream_t stream);
fa_status launch_bwd_dq(const BwdLaunch& L, cudaStream_t stream);
fa_status launch_diag_exp2(const float* x, float* y_emu, float* y_hw, long long n, cudaStream_t stream);
fa_status launch_diag_wait(unsigned long long limit_ns, cudaStream_t stream);

// Each translation unit keeps its own device error record; these read and
// clear it (returning FA_OK when clean).
fa_status fwd_take_device_error();
fa_status bwd_take_device_error();
fa_status bwd_pair_take_device_error();
fa_status bwd_dq_take_device_error();
fa_status diag_take_device_error();

// Shared-memory alignment slack added to every dynamic allocation.
constexpr int kSmemAlignSlack = 1024;

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s

}  // namespace fa
