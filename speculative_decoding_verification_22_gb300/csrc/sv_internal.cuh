// sv_internal.cuh -- definitions shared by the kernels of the verify step:
// workspace layout, status handling, bounded waits, and thin inline-PTX
// wrappers for mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (Blackwell
// tensor cores with TMEM accumulators) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace sv {

// ---------------------------------------------------------------------------
// Problem geometry
// ---------------------------------------------------------------------------
constexpr int kSub = 32;        // vocab entries per softmax partial (one warp)
constexpr int kTileM = 128;     // vocab rows per tensor-core tile (MMA M)
constexpr int kChunk = 4096;    // vocab entries per residual-mass chunk
constexpr int kTailThreads = 512;
constexpr int kChunkPerThread = kChunk / kTailThreads;  // 8
constexpr int kTailWarps = kTailThreads / 32;
constexpr int kMaxCand = 64;    // greedy: near-maximal subtiles listed per row

// Per-sequence state handed from the decision pass to the residual and
// selection passes.
// kModeResidualPoint: the residual of a draft proposed with certainty (q =
// the point mass at the proposed token): p without that token, whose id
// is held in q_row.
enum : int { kModeSkip = 0, kModeResidual = 1, kModeP = 2, kModeResidualPoint = 3 };

struct SeqState {
  int mode;      // kModeSkip: nothing to draw (greedy, invalid, error)
  int p_row;     // logits row of the final draw
  int q_row;     // q_logits row (kModeResidual)
  int n_acc;     // accepted draft tokens
  float p_max;   // p(v) = expf(L[v] * inv_t - p_max) * p_corr
  float p_corr;
  float q_max;   // q(v) = expf(ql[v] * inv_t - q_max) * q_corr
  float q_corr;
  float u_final; // the final uniform
  float p_tau;   // truncated sampling: p(v) = 0 where L[v] < p_tau (-inf: no cut)
  float q_tau;   // likewise q(v) = 0 where ql[v] < q_tau
  int pad;
};

struct Dims {
  int64_t V, d;
  int B, K;
  int R;        // B * (K + 1) target rows
  int RQ;       // B * K draft rows
  int nsub;     // ceil(V / 32)
  int ntile;    // ceil(V / 128)
  int nchunk;   // ceil(V / 4096)
};

// Device workspace (owned by the handle).
struct Work {
  float *logits;       // [R, V]
  float2 *part_p;      // [R, nsub]   (max, sum-exp) of logits / T; T == 0: (max, 0)
  float2 *part_q;      // [RQ, nsub]  (max, sum-exp) of q_logits / T
  float *row_m;        // [R + RQ]    row maximum M of logits / T (then of q_logits / T)
  float2 *row_s;       // [R + RQ]    row sum S = sum exp(x - M) as float-float (hi, lo);
                       //             LSE = M + log S
  SeqState *seq;       // [B]
  float2 *chunk_mass;  // [B, nchunk]  float-float residual masses
  float *split_buf;    // [grid, 2, 128 * npad]  partial tiles (tensor-core path)
  int *split_cnt;      // [grid, 4]
  int *status;         // [1]   first device-side error since last read
  unsigned *abort_epoch;  // [1] epoch of the last run whose contraction gave up
  unsigned *ticket;    // [1]   tail-kernel CTA order (rewound by its last CTA)
  unsigned *finished;  // [1]
  int *row_count;      // [B]   row CTAs finished per sequence
  int *chunk_count;    // [B]   chunk CTAs finished per sequence
  unsigned *seq_flag;  // [B]   epoch of the sequence's published decision
  int *seq_final;      // [B]   decision + chunk-phase arrivals, poison bit
  int *cand;           // [R, 1 + kMaxCand] greedy: count, then subtile ids
  float *row_tau;      // [R + RQ] truncated sampling: the row's cut logit
  float2 *draft_logit; // [RQ]  exact logit of each draft token (float-float)
  float4 *rowpart;     // [R + RQ, grid] per contraction CTA and row: (max M,
                       //   sum S = sum exp(x - M) as hi, lo, 1 if a NaN/+inf
                       //   entry was seen) of logits / T and q_logits / T
  float *draft_q;      // [RQ]  q_logits at each draft token (contraction)
  int *chunk_done;     // [B]   chunk CTAs past the cooperative selection
  int *never;          // [1]   0, never written: the flag of the test stall
};

// ---------------------------------------------------------------------------
// Status word: the first device-side error wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int *status, int code) {
  atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier among the first-come nthreads threads (whole warps) that use
// barrier id (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed.  Gives up
// (returns false) after limit_ns nanoseconds or as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns,
                                          const volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 >= limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
               : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled load of box {c0 .. c0+box0, c1 .. c1+box1} into shared memory,
// completing `bar` with the box's byte count.  c0 (innermost) must be a
// multiple of 16 bytes' worth of elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m,
                                            int32_t c0, int32_t c1, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// 3-D tiled load: box {c0.., c1.., c2..}; same alignment rule on c0.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled store from shared memory (bulk async-group of the issuing
// thread); c0 follows the load's alignment rule, and parts of the box past
// the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until none of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA) before a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (TMEM + tensor cores), cta_group::1
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 out).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc,
                                          uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with FP8 E4M3 operands (kind::f8f6f4, K = 32 per instruction:
// the 32 bytes of a row that one bf16 instruction reads).
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when all tcgen05.mma issued so far by this thread
// have completed.
// One lane of the (converged) warp; the same lane every time.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}
// 32 lanes x 16 consecutive fp32 columns: thread i of the warp receives lane
// (quadrant base + i).  The registers are valid only after tmem_ld_wait()
// and then tmem_reg_fence(), which ties every later use to the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_reg_fence(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand written by TMA with
// 128-byte swizzling: rows of 128 bytes (64 bf16), 8-row groups 1024 bytes
// apart (stride byte offset), leading byte offset unused (1), descriptor
// version 1 (bit 46), swizzle mode 2 = 128B (bits 61-63).  The buffer must be
// 1024-byte aligned; the k-th 16-element slice starts 32*k bytes further.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  desc |= static_cast<uint64_t>(1) << 16;
  desc |= static_cast<uint64_t>(1024 >> 4) << 32;
  desc |= static_cast<uint64_t>(1) << 46;
  desc |= static_cast<uint64_t>(2) << 61;
  return desc;
}
// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// kind::f8f6f4 with A and B in E4M3 (type code 0) and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// (max, sum-exp) partial of one 32-entry vocab subtile held one entry per
// lane.  `valid` masks entries past V.  T == 0 (greedy) keeps only the max.
// -inf entries are allowed (probability zero); a NaN or +inf entry makes the
// whole partial (NaN, NaN), which the decision pass reports.  All lanes
// return the result.
__device__ __forceinline__ float2 subtile_partial(float logit, bool valid, float inv_t,
                                                  bool greedy) {
  if (__any_sync(0xffffffffu, valid && (isnan(logit) || logit == INFINITY)))
    return make_float2(NAN, NAN);
  if (greedy) {
    const float m = warp_max(valid ? logit : -INFINITY);
    return make_float2(m, 0.0f);
  }
  const float a = valid ? logit * inv_t : -INFINITY;
  const float m = warp_max(a);
  const float e = (valid && m > -INFINITY) ? expf(a - m) : 0.0f;
  return make_float2(m, warp_sum(e));
}

// Reduce-scatter over a warp of a 32 x 16 block held as 16 values per lane:
// every exchange halves the columns a lane keeps (8 + 4 + 2 + 1 shuffles,
// one more pairs the lanes), so on return lanes 2c and 2c+1 hold column c's
// reduction.  16 shuffles for 16 columns, against 80 for one butterfly per
// column, and the shuffles of each stage are independent of one another.
template <class Op>
__device__ __forceinline__ float reduce_scatter16(const float (&a)[16], int lane, Op op) {
  float v8[8], v4[4], v2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float give = b4 ? a[j] : a[j + 8];
    const float keep = b4 ? a[j + 8] : a[j];
    v8[j] = op(keep, __shfl_xor_sync(0xffffffffu, give, 16));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float give = b3 ? v8[j] : v8[j + 4];
    const float keep = b3 ? v8[j + 4] : v8[j];
    v4[j] = op(keep, __shfl_xor_sync(0xffffffffu, give, 8));
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float give = b2 ? v4[j] : v4[j + 2];
    const float keep = b2 ? v4[j + 2] : v4[j];
    v2[j] = op(keep, __shfl_xor_sync(0xffffffffu, give, 4));
  }
  const float give = b1 ? v2[0] : v2[1];
  const float keep = b1 ? v2[1] : v2[0];
  const float v1 = op(keep, __shfl_xor_sync(0xffffffffu, give, 2));
  return op(v1, __shfl_xor_sync(0xffffffffu, v1, 1));
}

// Subtile partials of 16 columns at once (the same values subtile_partial
// gives column by column): a[i] is this lane's entry of column i, already
// divided by T (or the raw logit for greedy), -inf where the entry is past
// V; bit i of `bad` marks a NaN or +inf entry.  Lanes 2c and 2c+1 return
// column c's (max, sum-exp), or (NaN, NaN).
__device__ __forceinline__ float2 column_partials16(const float (&a)[16], unsigned bad,
                                                   bool greedy, int lane) {
  const unsigned any_bad = __reduce_or_sync(0xffffffffu, bad);
  const float m = reduce_scatter16(a, lane, [](float x, float y) { return fmaxf(x, y); });
  float s = 0.0f;
  if (!greedy) {
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float mi = __shfl_sync(0xffffffffu, m, 2 * i);
      e[i] = mi > -INFINITY ? expf(a[i] - mi) : 0.0f;
    }
    s = reduce_scatter16(e, lane, [](float x, float y) { return x + y; });
  }
  if ((any_bad >> (lane >> 1)) & 1u) return make_float2(NAN, NAN);
  return make_float2(m, s);
}

// Error-free sum of two floats (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// ---------------------------------------------------------------------------
// Float-float ("double-float") numbers: value = hi + lo with |lo| <= ulp(hi)/2,
// about 48 significant bits, on the fp32 pipe (GB300's fp64 rate is a small
// fraction of its fp32 rate).  Addition uses TwoSum, so its result does not
// depend on the order of the operands.
// ---------------------------------------------------------------------------
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_make(float x) { return ff{x, 0.0f}; }
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, e);
  return ff{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.hi, -a.lo}; }
// a * b for a float b, exact product of the heads via FMA
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  const float p = __fmul_rn(a.hi, b);
  const float pe = fmaf(a.hi, b, -p);
  const float e = fmaf(a.lo, b, pe);
  const float hi = __fadd_rn(p, e);
  return ff{hi, __fsub_rn(e, __fsub_rn(hi, p))};
}
// a / b for a float b (one correction step)
__device__ __forceinline__ ff ff_div_f(ff a, float b) {
  const float q = __fdiv_rn(a.hi, b);
  const float r = __fadd_rn(fmaf(-q, b, a.hi), a.lo);
  const float ql = __fdiv_rn(r, b);
  const float hi = __fadd_rn(q, ql);
  return ff{hi, __fsub_rn(ql, __fsub_rn(hi, q))};
}
// a / b, both float-float, to float-float accuracy
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q = __fdiv_rn(a.hi, b.hi);
  // r = a - q * b
  const ff qb = ff_mul_f(b, q);
  const ff r = ff_add(a, ff_neg(qb));
  const float ql = __fdiv_rn(r.hi, b.hi);
  const float hi = __fadd_rn(q, ql);
  return ff{hi, __fsub_rn(ql, __fsub_rn(hi, q))};
}
__device__ __forceinline__ bool ff_lt(ff a, ff b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
__device__ __forceinline__ float ff_to_f(ff a) { return __fadd_rn(a.hi, a.lo); }
__device__ __forceinline__ ff ff_shfl_xor(ff a, int o) {
  return ff{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ ff ff_shfl_up(ff a, int o) {
  return ff{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ ff ff_shfl(ff a, int src) {
  return ff{__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
// butterfly sum: every lane ends with the same value
__device__ __forceinline__ ff warp_sum_ff(ff x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = ff_add(x, ff_shfl_xor(x, o));
  return x;
}

// Folds the (max, sum-exp) pair (m, s) of some entries into the running
// pair (M, S) of a row: M becomes max(M, m) and both sums are taken relative
// to it.  A pair with m = -inf holds no mass (so does a NaN m: callers track
// NaN and +inf entries separately).  The result does not depend on which
// pair is the running one.
__device__ __forceinline__ void lse_fold(float m, ff s, float &M, ff &S) {
  if (!(m > -INFINITY)) return;
  if (m > M) {
    S = M > -INFINITY ? ff_add(ff_mul_f(S, expf(M - m)), s) : s;
    M = m;
  } else {
    S = ff_add(S, m == M ? s : ff_mul_f(s, expf(m - M)));
  }
}

// Accumulates a * b exactly into the pair (s, c): the product's rounding
// error comes from an FMA (zero when the product is exact, as for bf16) and
// the sum's from TwoSum.
__device__ __forceinline__ void acc_product(float a, float b, float &s, float &c) {
  const float p = __fmul_rn(a, b);
  const float pe = fmaf(a, b, -p);
  float t, e;
  two_sum(s, p, t, e);
  s = t;
  c = __fadd_rn(c, __fadd_rn(e, pe));
}

// Exact-product, TwoSum-compensated dot product of two bf16 rows of length
// d (a multiple of 8; 16-byte aligned) by one warp, over the 16-byte vectors
// [lo, hi) of the rows, 4 vectors in flight per lane.  Returns a float-float
// (every lane the same value).
__device__ __forceinline__ ff dot_bf16_warp(const uint4 *h, const uint4 *w, int64_t lo,
                                            int64_t hi, int lane) {
  float s = 0.0f, c = 0.0f;
  constexpr int kBatch = 4;
  for (int64_t k0 = lo; k0 < hi; k0 += 32 * kBatch) {
    uint4 hv[kBatch], wv[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t k = k0 + j * 32 + lane;
      hv[j] = k < hi ? __ldg(&h[k]) : make_uint4(0, 0, 0, 0);
      wv[j] = k < hi ? __ldg(&w[k]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const uint32_t hw[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
      const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // a bf16 value is the top half of an fp32; the widening is exact
        acc_product(__uint_as_float(hw[e] << 16), __uint_as_float(ww[e] << 16), s, c);
        acc_product(__uint_as_float(hw[e] & 0xffff0000u), __uint_as_float(ww[e] & 0xffff0000u),
                    s, c);
      }
    }
  }
  const float hi2 = __fadd_rn(s, c);
  return warp_sum_ff(ff{hi2, __fsub_rn(c, __fsub_rn(hi2, s))});
}

// The same for two FP8 E4M3 rows of length d (a multiple of 16): E4M3
// values are exact in fp32, and so are products of two of them.
__device__ __forceinline__ ff dot_e4m3_warp(const uint4 *h, const uint4 *w, int64_t lo,
                                            int64_t hi, int lane) {
  float s = 0.0f, c = 0.0f;
  constexpr int kBatch = 4;
  for (int64_t k0 = lo; k0 < hi; k0 += 32 * kBatch) {
    uint4 hv[kBatch], wv[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int64_t k = k0 + j * 32 + lane;
      hv[j] = k < hi ? __ldg(&h[k]) : make_uint4(0, 0, 0, 0);
      wv[j] = k < hi ? __ldg(&w[k]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const uint32_t hw[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
      const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const __nv_fp8x2_storage_t h2 = static_cast<__nv_fp8x2_storage_t>(hw[e] >> (16 * hh));
          const __nv_fp8x2_storage_t w2 = static_cast<__nv_fp8x2_storage_t>(ww[e] >> (16 * hh));
          const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
          const float2 wf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(w2, __NV_E4M3)));
          acc_product(hf.x, wf.x, s, c);
          acc_product(hf.y, wf.y, s, c);
        }
      }
    }
  }
  const float hi2 = __fadd_rn(s, c);
  return warp_sum_ff(ff{hi2, __fsub_rn(c, __fsub_rn(hi2, s))});
}

// ---------------------------------------------------------------------------
// Block-level helpers (kTailThreads threads)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void st_ff_raw(float2 *p, ff v) { *p = make_float2(v.hi, v.lo); }

__device__ __forceinline__ ff block_sum_ff(ff x, ff *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  x = warp_sum_ff(x);
  __syncthreads();
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    ff t = lane < kTailWarps ? s_warp[lane] : ff_make(0.0f);
    t = warp_sum_ff(t);
    if (lane == 0) s_warp[0] = t;
  }
  __syncthreads();
  return s_warp[0];
}

__device__ __forceinline__ float block_max_f(float x, float *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  x = warp_max(x);
  __syncthreads();
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float t = lane < kTailWarps ? s_warp[lane] : -INFINITY;
    t = warp_max(t);
    if (lane == 0) s_warp[0] = t;
  }
  __syncthreads();
  return s_warp[0];
}

}  // namespace sv
