// C ABI of the library (include/fa.h, include/fa_diag.h): argument
// validation, tensor-map construction, device-error plumbing and dispatch to
// the kernel translation units.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "fa.h"
#include "fa_diag.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Forward knobs the library picks per configuration when the caller leaves
// them at -1.
struct FwdChoice {
  int emu_per_16;   // exponentials of every 16 on the FMA-pipe polynomial
  int split_p;      // P handed to the tensor cores in two halves
  int kv_stages;    // K/V ring depth
  int head_group;   // dense causal: (batch, head) pairs per longest-first group
};

// The table of per-configuration choices, from a measured sweep on GB300
// (forward TFLOPS, B*S = 32768 tokens, H = 16, S = 1K ... 32K; the full
// sweep is in the design notes).  Handing P over in two halves (split_p)
// paid everywhere, and with it moving 2 of every 16 exponentials to the FMA
// pipe did too (D = 128, S = 4096: 1294 with neither, 1336 split, 1405 split
// with 2/16; causal 1058 / 1058 / 1128; D = 64 non-causal 709 / 714 / 772);
// 4/16 on the FMA pipe was slower than 2/16 everywhere.  The K/V ring: D = 128
// keeps its maximum of 4 stages (2: -5 to -10%; 3: equal or within noise);
// D = 64 is flat from 4 to 8 stages and loses a little at 10 under a causal
// mask; it takes 6.
FwdChoice default_fwd_choice(int D, int causal, int Sk, int BH) {
  FwdChoice c;
  c.emu_per_16 = 2;
  c.split_p = 1;
  c.kv_stages = D == 128 ? 4 : 6;
  // all heads in one longest-first group: groups of 8 / 32 heads measured
  // 1-4% slower at S = 1024 and 4096 (causal D = 128)
  c.head_group = BH;
  (void)causal;
  (void)Sk;
  return c;
}
constexpr float kDefaultThreshold = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Current device's SM count; FA_ERR_UNSUPPORTED unless it is compute 10.3.
fa_status device_info(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Shape checks common to both passes.  Packed inputs: Sq == Sk == total.
fa_status check_shapes(int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, const int* cu_seqlens) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (cu_seqlens != nullptr) {
    if (Sq != Sk) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return FA_ERR_INVALID_ARG;
    if (B > kMaxPackedSeqs) return FA_ERR_UNSUPPORTED;
  }
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  // token indices must fit the kernels' 32-bit index arithmetic
  const long long rows_q = cu_seqlens ? (long long)Sq : (long long)B * Sq;
  const long long rows_k = cu_seqlens ? (long long)Sk : (long long)B * Sk;
  if (rows_q > INT32_MAX - 512 || rows_k > INT32_MAX - 512) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

fa_status prepare_kernel(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (kernel, device)
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : done)
    if (e.first == func && e.second == dev) return FA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return FA_ERR_CUDA;
  done.emplace_back(func, dev);
  return FA_OK;
}

fa_status make_tmap_rows_heads_d(CUtensorMap* map, const void* base, int rows, int heads, int D, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

fa_status make_tmap_f32_rows_heads_d(CUtensorMap* map, const void* base, int rows, int heads, int D, int box_d,
                                     int box_rows) {
  auto fn = encode_fn();
  if (!fn) return FA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)heads * D * 4};
  const cuuint32_t box[3] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

BwdWorkspace bwd_workspace_layout(int B, int Hq, int Hkv, int Sq, int D, int deterministic, bool packed) {
  BwdWorkspace w{};
  // row terms per head: dense, Sq rounded up to 64 per batch entry; packed,
  // every sequence rounded up to 64 rows, bounded by total + 64 per sequence
  const size_t sq_pad = packed ? (size_t(Sq) + 63) / 64 * 64 + 64 * size_t(B) : (size_t(Sq) + 63) / 64 * 64;
  const size_t rows = packed ? size_t(Sq) : size_t(B) * Sq;       // rows of the accumulator
  const size_t heads_rt = packed ? size_t(Hq) : size_t(B) * Hq;  // row-term arrays of sq_pad floats
  size_t off = 0;
  w.dq_acc = off;
  off = align256(off + rows * Hq * D * sizeof(float));
  w.ndelta = off;
  off = align256(off + heads_rt * sq_pad * sizeof(float));
  w.nlse2 = off;
  off = align256(off + heads_rt * sq_pad * sizeof(float));
  w.plan = off;
  if (packed) off = align256(off + (2 * size_t(B) + 4) * sizeof(int));
  // packed: the unit order table, one entry per (key block, kv head); every
  // sequence adds at most one partial key block
  w.order = off;
  if (packed) off = align256(off + (size_t(Sq) / 128 + size_t(B)) * size_t(Hkv) * sizeof(int2));
  w.sched = off;
  off = align256(off + sizeof(int));
  w.tickets = off;
  if (deterministic) off = align256(off + heads_rt * (sq_pad / 64) * 2 * sizeof(int));
  w.total = off;
  w.sq_pad = (int)sq_pad;
  return w;
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_fwd_tuning fa_fwd_default_tuning(void) {
  fa_fwd_tuning t;
  t.rescale_threshold = kDefaultThreshold;
  t.emu_per_16 = -1;
  t.split_p = -1;
  t.kv_stages = -1;
  t.head_group = -1;
  return t;
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                    int Sq, int Sk, int D, int causal, float scale, const int* cu_seqlens,
                    const fa_fwd_tuning* t, fa_stream_t stream) {
  try {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
      return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shapes(B, Hq, Hkv, Sq, Sk, D, scale, cu_seqlens);
    if (st != FA_OK) return st;
    fa_fwd_tuning tune = fa_fwd_default_tuning();
    if (t) {
      if (!(t->rescale_threshold >= 0.0f && t->rescale_threshold <= 16.0f)) return FA_ERR_INVALID_ARG;
      tune.rescale_threshold = t->rescale_threshold;
      if (t->emu_per_16 >= 0) {
        if (t->emu_per_16 != 0 && t->emu_per_16 != 2 && t->emu_per_16 != 3 && t->emu_per_16 != 4)
          return FA_ERR_INVALID_ARG;
        tune.emu_per_16 = t->emu_per_16;
      }
      if (t->split_p > 1) return FA_ERR_INVALID_ARG;
      tune.split_p = t->split_p;
      if (t->kv_stages > 0) {
        if (t->kv_stages < 2 || t->kv_stages > (D == 128 ? 4 : 10)) return FA_ERR_INVALID_ARG;
        tune.kv_stages = t->kv_stages;
      }
      tune.head_group = t->head_group;
    }
    const FwdChoice def = default_fwd_choice(D, causal, Sk, B * Hq);
    int num_sms = 0;
    if ((st = device_info(&num_sms)) != FA_OK) return st;
    FwdLaunch L{};
    L.q = q;
    L.k = k;
    L.v = v;
    L.p.o = o;
    L.p.lse = lse;
    L.p.o_st32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    L.p.cu_seqlens = cu_seqlens;
    L.p.B = B;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.Sq = Sq;
    L.p.Sk = Sk;
    L.p.group = Hq / Hkv;
    L.p.scale_log2 = scale * kLog2e;
    L.p.thr = tune.rescale_threshold;
    L.p.stages = tune.kv_stages > 0 ? tune.kv_stages : def.kv_stages;
    L.p.split_p = tune.split_p >= 0 ? tune.split_p : def.split_p;
    {
      const long long bh = (long long)B * Hq;
      long long g = tune.head_group > 0 ? tune.head_group : def.head_group;
      if (g > bh) g = bh;
      if (g < 1) g = 1;
      L.p.sched_group = (int)g;
    }
    L.p.snake = (causal && cu_seqlens == nullptr && Sq >= 4096) ? 1 : 0;
    L.p.wait_limit_ns = kDefaultWaitLimitNs;
    L.D = D;
    L.causal = causal != 0;
    L.emu_per_16 = tune.emu_per_16 >= 0 ? tune.emu_per_16 : def.emu_per_16;
    L.num_sms = num_sms;
    return launch_fwd(L, reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return FA_ERR_CUDA;
  }
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                 int Sq, int Sk, int D, int causal, float scale, const int* cu_seqlens, fa_stream_t stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, cu_seqlens, nullptr, stream);
}

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, const int* cu_seqlens_host,
                             int total_q, int deterministic) {
  if (deterministic != 0 && deterministic != 1) return 0;
  if ((D != 64 && D != 128) || total_q < 0) return 0;
  const bool packed = cu_seqlens_host != nullptr || total_q > 0;
  if (!packed) {
    if (check_shapes(B, Hq, Hkv, Sq, Sk, D, 1.0f, nullptr) != FA_OK) return 0;
    return bwd_workspace_layout(B, Hq, Hkv, Sq, D, deterministic, false).total;
  }
  // packed: Sq = Sk = total_q rows (any 4-aligned non-null marker passes the
  // pointer checks of check_shapes; the offsets themselves are checked below)
  static const int kMarker[1] = {0};
  if (Sq != total_q || Sk != total_q) return 0;
  if (check_shapes(B, Hq, Hkv, Sq, Sk, D, 1.0f, kMarker) != FA_OK) return 0;
  if (cu_seqlens_host) {
    if (cu_seqlens_host[0] != 0 || cu_seqlens_host[B] != total_q) return 0;
    for (int b = 0; b < B; ++b)
      if (cu_seqlens_host[b + 1] < cu_seqlens_host[b] || cu_seqlens_host[b + 1] - cu_seqlens_host[b] > 262144)
        return 0;
  }
  return bwd_workspace_layout(B, Hq, Hkv, Sq, D, deterministic, true).total;
}

fa_bwd_tuning fa_bwd_default_tuning(void) {
  fa_bwd_tuning t;
  t.paired = 0;
  t.schedule = -1;
  t.head_group = -1;
  t.reverse_blocks = -1;
  t.scores_first = -1;
  t.split_dq = -1;
  return t;
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                    int causal, float scale, const int* cu_seqlens, int deterministic, void* workspace,
                    size_t workspace_bytes, const fa_bwd_tuning* t, fa_stream_t stream) {
  try {
    fa_bwd_tuning tune = fa_bwd_default_tuning();
    if (t) {
      if (t->paired > 1 || t->schedule > 1 || t->reverse_blocks > 1 || t->scores_first > 1 || t->split_dq > 1 ||
          t->head_group == 0)
        return FA_ERR_INVALID_ARG;
      if (t->paired >= 0) tune.paired = t->paired;
      tune.schedule = t->schedule;
      tune.head_group = t->head_group;
      tune.reverse_blocks = t->reverse_blocks;
      tune.scores_first = t->scores_first;
      tune.split_dq = t->split_dq;
    }
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (const void* p : ptrs)
      if (!aligned16(p)) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shapes(B, Hq, Hkv, Sq, Sk, D, scale, cu_seqlens);
    if (st != FA_OK) return st;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const bool packed = cu_seqlens != nullptr;
    // the paired kernel is for the dense layout at D = 128 only
    if ((packed || D != 128) && tune.paired == 1) return FA_ERR_UNSUPPORTED;
    const BwdWorkspace ws = bwd_workspace_layout(B, Hq, Hkv, Sq, D, deterministic, packed);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < ws.total)
      return FA_ERR_WORKSPACE;
    int num_sms = 0;
    if ((st = device_info(&num_sms)) != FA_OK) return st;
    uint8_t* wb = static_cast<uint8_t*>(workspace);
    BwdLaunch L{};
    L.q = q;
    L.k = k;
    L.v = v;
    L.p.o = o;
    L.p.dout = dout;
    L.p.lse = lse;
    L.p.dq = dq;
    L.p.dk = dk;
    L.p.dv = dv;
    L.p.dkv_st32 = ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31u) == 0;
    L.p.dq_acc = reinterpret_cast<float*>(wb + ws.dq_acc);
    L.p.ndelta = reinterpret_cast<float*>(wb + ws.ndelta);
    L.p.nlse2 = reinterpret_cast<float*>(wb + ws.nlse2);
    L.p.sq_pad = ws.sq_pad;
    L.p.nqb = ws.sq_pad / 64;
    L.p.tickets = deterministic ? reinterpret_cast<int*>(wb + ws.tickets) : nullptr;
    L.p.cu_seqlens = cu_seqlens;
    L.p.plan = packed ? reinterpret_cast<int*>(wb + ws.plan) : nullptr;
    L.p.order = packed ? reinterpret_cast<int2*>(wb + ws.order) : nullptr;
    L.p.sched = reinterpret_cast<int*>(wb + ws.sched);
    // Work schedule of the main kernel (see its decode_unit and
    // producer_role).  Units are claimed dynamically for packed sequences
    // (lengths vary without a pattern); otherwise CTA c takes units c,
    // c + grid, ..., which measured faster on dense inputs even under a
    // causal mask (causal S = 1024 / 2048: 567 / 770 TFLOPS static against
    // 469 / 617 claimed; deterministic causal S = 8192 B = 2: 717 against
    // 696).  In either schedule a unit waits only on units with smaller
    // indices, which are running or done.  Dense order: head-major
    // (g = 1) without a causal mask (all units equally long; a head's key
    // blocks run together and share its Q / dO rows in L2).  With one,
    // key-block-major within groups of g = 32 heads: the longest blocks start
    // first, and each head has a few consecutive key blocks in flight, which
    // move through the same query rows a few blocks apart (measured over
    // g = 5 ... 512: 32 is within 2% of the best at S = 1K ... 32K, and
    // causal S = 8192 B = 2 runs 914 -> 1018 TFLOPS against the former
    // L2-footprint rule).  Deterministic mode: key-block-major over all
    // heads, so that a block's predecessor in the ordered dQ additions was
    // claimed as far ahead as possible, and each unit visits its query
    // blocks last to first, so that it meets its predecessor's additions in
    // the order they were made (causal S = 8192 B = 2: 607 -> 616 TFLOPS;
    // packed varlen: 265 -> 317).
    // Packed layouts: (sequence, kv head) pairs sorted longest first, in
    // groups of 16 pairs (deterministic: 32), key-block-major within a group
    // (the plan kernel writes the order; varlen GQA workload, 64 sequences:
    // groups of 8 / 16 / 32 / 64 / 512 pairs: 1013 / 1006 / 988 / 740 / 661
    // TFLOPS, deterministic 591 / - / 717 / 632 / 569).
    // The split backward (the deterministic default) has no ordered
    // additions, so its main kernel takes the schedule of the atomic mode.
    // Measured on GB300, deterministic mode, split (dQ kernel with Q and dO
    // held in tensor memory) against the ticket-ordered fused kernel: dense
    // B=4 H=16 S=4096 D=128 927 vs 717 TFLOPS, causal 798 vs 657, training
    // shape (B=2 S=8192 causal) 888 vs 716, packed varlen GQA (64 sequences,
    // 128..8192 tokens) 852 vs 728.
    const bool split = tune.paired != 1 &&
                       (tune.split_dq >= 0 ? tune.split_dq == 1 : deterministic == 1);
    const bool tickets = deterministic && !split;
    {
      const long long bh = (long long)B * Hkv;
      const bool dynamic = tune.schedule >= 0 ? tune.schedule == 1 : packed;
      long long g = 1;
      if (tune.head_group > 0) g = tune.head_group;
      else if (packed) g = tickets ? 32 : 16;
      else if (tickets) g = bh;
      else if (causal) g = 32;
      if (g > bh) g = bh;
      L.p.sched_group = (int)g;
      L.p.sched_dynamic = dynamic ? 1 : 0;
      L.p.rev_blocks = tune.reverse_blocks >= 0 ? tune.reverse_blocks : (tickets ? 1 : 0);
      L.p.scores_first = tune.scores_first >= 0 ? tune.scores_first : (tickets ? 0 : 1);
    }
    L.p.B = B;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.Sq = Sq;
    L.p.Sk = Sk;
    L.p.D = D;
    L.p.group = Hq / Hkv;
    L.p.causal = causal;
    L.p.deterministic = deterministic;
    L.p.scale = scale;
    L.p.scale_log2 = scale * kLog2e;
    L.p.wait_limit_ns = kDefaultWaitLimitNs;
    L.num_sms = num_sms;
    L.pair = tune.paired == 1 && !packed && D == 128;
    L.split_dq = split;
    return launch_bwd(L, reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return FA_ERR_CUDA;
  }
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                 float scale, const int* cu_seqlens, int deterministic, void* workspace,
                 size_t workspace_bytes, fa_stream_t stream) {
  return fa_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, D, causal, scale, cu_seqlens,
                   deterministic, workspace, workspace_bytes, nullptr, stream);
}

fa_status fa_get_device_error(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  fa_status first = FA_OK;
  const fa_status all[5] = {fwd_take_device_error(), bwd_take_device_error(), bwd_pair_take_device_error(),
                            bwd_dq_take_device_error(), diag_take_device_error()};
  for (fa_status s : all)
    if (first == FA_OK && s != FA_OK) first = s;
  return first;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_diag_exp2(const float* x, float* y_emu, float* y_hw, long long n, fa_stream_t stream) {
  if (n < 0) return FA_ERR_INVALID_ARG;
  if (n > 0 && (!x || !y_emu || !y_hw)) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  int num_sms = 0;
  fa_status st = device_info(&num_sms);
  if (st != FA_OK) return st;
  return launch_diag_exp2(x, y_emu, y_hw, n, reinterpret_cast<cudaStream_t>(stream));
}

fa_status fa_diag_wait_timeout(unsigned long long limit_ns, fa_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  int num_sms = 0;
  fa_status st = device_info(&num_sms);
  if (st != FA_OK) return st;
  return launch_diag_wait(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
