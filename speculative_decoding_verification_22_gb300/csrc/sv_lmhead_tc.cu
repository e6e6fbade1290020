// sv_lmhead_tc.cu -- kernel (a) of the verify step, bf16 path: the
// weight-streaming skinny contraction L = H * W^T on Blackwell tensor cores.
//
// The verify pass multiplies the [positions x d] block of final hidden
// states against the LM-head matrix, which is read from memory once
// ("What Actually Happens During Speculative Decoding in LLMs", memory-bound
// section; "Speculative Decoding: Guess Several Tokens, Check Them in One
// Pass", Step 1).  With R = B*(K+1) rows (5..384) the step is HBM-bound, so
// the kernel is built around streaming W exactly once:
//
//  * swap-AB: the vocabulary is the MMA M dimension (128 W rows per tile)
//    and the R hidden rows, padded to npad (multiple of 16), are N;
//  * persistent grid, one CTA per SM, stream-K split of the
//    (tile, 64-wide k block) units so every SM streams the same number of
//    bytes; a tile cut between two CTAs is finished by whichever CTA
//    completes its part second (drain mode: always by the CTA holding its
//    first k block);
//  * warp 0 issues TMA loads (128B swizzle, W evict-first in L2) into a
//    ring of shared-memory stages; warp 1 issues tcgen05.mma (kind::f16,
//    M=128, K=16) into TMEM; warps 2..5 drain TMEM and run the epilogue;
//  * drain mode (npad <= 64): each group of k blocks (one, or four at 32
//    and 64 columns) accumulates into its own TMEM slot of a ring and the
//    epilogue adds it into fp32 registers with round-to-nearest adds, so no
//    long tensor-core accumulation chain can bias the logits; direct mode
//    (npad > 64): up to four TMEM accumulators per tile (contiguous k
//    ranges) summed in registers, two tiles in TMEM up to 256 columns;
//    above 256 columns the two CTAs of a pair take the same tiles, each
//    for half of the columns (half mode), so two tiles fit again;
//  * the epilogue stages each 16-column group in shared memory, writes the
//    fp32 logits with a TMA store, and computes the per-32-entry (max,
//    sum-exp) partials of logits / T (or the max for T == 0); four more
//    warps stream the draft logits q / T of the tile for the same partials.
//    They run on the two warp schedulers that host neither the TMA
//    producer nor the MMA issuer (warps 6, 7, 10, 11; warps 8 and 9 have
//    no role): sharing a scheduler with those two latency-critical loops
//    cost up to 11 us per launch at 64 columns.
#include <atomic>

#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {
namespace tc {

// Ring depth and TMEM drain-ring length (tuning parameters).
#ifndef SV_TC_MAX_STAGES
#define SV_TC_MAX_STAGES 8
#endif
#ifndef SV_TC_DRAIN_SLOTS
#define SV_TC_DRAIN_SLOTS 32
#endif
#ifndef SV_TC_STAGES_C2
#define SV_TC_STAGES_C2 6
#endif
#ifndef SV_TC_STAGES_C4
#define SV_TC_STAGES_C4 2
#endif
#ifndef SV_TC_MAX_CHUNKS
#define SV_TC_MAX_CHUNKS 2
#endif
// direct-mode widths above which CTA pairs split the columns.  Each SM of a
// pair still takes in the whole W tile for twice as many k blocks, and at
// large widths the kernel is bound by the bytes each SM takes in from L2
// (about 70 GB/s per SM measured, with or without a multicast of W inside a
// 2-CTA cluster), so splitting pays only where one tile no longer fits
// TMEM twice (above 256 columns).
#ifndef SV_TC_HALF_MIN
#define SV_TC_HALF_MIN 256
#endif

constexpr int kWSlabBytes = kTileM * 128;          // 16 KB: 128 rows x 128 bytes
constexpr int kMaxStages = SV_TC_MAX_STAGES;
constexpr int kNumEpiWarps = 4;
constexpr int kNumQWarps = 4;
// warp w runs on scheduler w % 4; the draft-logit warps take schedulers 2
// and 3 only (see the top of the file), so the block has two idle warps
constexpr int kThreads = 64 + 32 * (kNumEpiWarps + kNumQWarps + 2);  // 384
__device__ __forceinline__ bool is_q_warp(int warp) {
  return warp >= 2 + kNumEpiWarps && (warp & 3) >= 2;
}
// 0 .. kNumQWarps - 1 for warps 6, 7, 10, 11
__device__ __forceinline__ int q_warp_index(int warp) {
  return ((warp - 2 - kNumEpiWarps) >> 2) * 2 + (warp & 1);
}
constexpr int kMaxDrainSlots = 32;
// TMEM slots of the drain ring for a column capacity NCOL (<= 512 columns)
// (direct mode: the two tile buffers)
template <int NCOL>
constexpr int drain_slots() {
  return NCOL == 0 ? 2 : (512 / NCOL < SV_TC_DRAIN_SLOTS ? 512 / NCOL : SV_TC_DRAIN_SLOTS);
}
// 64-wide k blocks accumulated into one drain slot.  Every drain costs the
// epilogue a TMEM read and an add per column, so at 32 and 64 columns four
// blocks share a slot: the tensor cores sum 16 MMAs of K=16 before each
// round-to-nearest add (a chain of all 64 blocks in TMEM was measured at
// about four times the logit error: the tensor-core sum drifts toward zero
// as the chain grows), and the MMA can run 32 (64 columns) or 64 blocks
// ahead of a draining tile end.
#ifndef SV_TC_KPS
#define SV_TC_KPS 4
#endif
#ifndef SV_TC_KPS16
#define SV_TC_KPS16 1
#endif
template <int NCOL>
constexpr int kblocks_per_slot() {
  return NCOL >= 32 ? SV_TC_KPS : SV_TC_KPS16;
}
#ifndef SV_TC_TEMPTY_BATCH
#define SV_TC_TEMPTY_BATCH 4
#endif
// Drain slots the MMA issuer takes per wait on the epilogue (long rings
// only): the epilogue frees slots in order, so once the last of a batch is
// free the whole batch is.
template <int NCOL>
constexpr int tempty_batch() {
  return drain_slots<NCOL>() >= 16 ? SV_TC_TEMPTY_BATCH : 1;
}
constexpr uint64_t kCleanupLimitNs = 2000000000ull;
// Epilogue staging: one 2 KB box ([16 columns][32 entries] fp32) per
// epilogue warp, after the stage ring (1024-byte aligned: the box uses the
// TMA 128-byte swizzle).
constexpr int kBoxFloats = 16 * 32;
constexpr int kEpiBytes = kNumEpiWarps * kBoxFloats * 4;

// Draft rows whose per-CTA (max, sum-exp) the draft-logit warps keep in
// shared memory (drain mode: fewer than 64 rows).
constexpr int kQaccRows = 64;

struct Ctl {
  float4 qacc[kQaccRows];  // (M, S hi, S lo, bad) of this CTA's entries per draft row
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[kMaxDrainSlots];
  uint64_t tempty[kMaxDrainSlots];
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
  int issued;
  int consumed;
};

// The k-block range [kb0, kb1) of tile t inside this CTA's unit range
// [u0, u1); a unit is a group of `chunks` k blocks (ngr groups per tile).
__device__ __forceinline__ void tile_range(int t, int64_t u0, int64_t u1, int ngr, int chunks,
                                           int &kb0, int &kb1) {
  const int64_t tb = static_cast<int64_t>(t) * ngr;
  kb0 = static_cast<int>((u0 > tb ? u0 : tb) - tb) * chunks;
  kb1 = static_cast<int>((u1 < tb + ngr ? u1 : tb + ngr) - tb) * chunks;
}

__device__ __forceinline__ void raise_abort(Ctl *ctl, const TcParams &P) {
  *reinterpret_cast<volatile int *>(&ctl->abort_flag) = 1;
  set_status(P.w.status, SV_ERR_TIMEOUT);
  atomicExch(P.w.abort_epoch, P.epoch);
}

// Draft-logit rows streamed per warp and batch (loads in flight per lane).
constexpr int kQBatch = 8;

// (max, sum-exp) partials of q / T over the 128 entries of tile t for the
// draft rows r0, r0 + rstep, ... (warp wq of the four takes r0 = wq, rstep
// 4; in half mode the two CTAs of a pair interleave, rstep 8); a lane holds
// four consecutive entries (one 16-byte load when rows are 16-byte
// aligned), eight lanes one 32-entry subtile, so a row of the tile costs
// three shuffle levels per reduction and a batch keeps 8 x 512 bytes of
// each warp's loads in flight.
__device__ __forceinline__ void q_partials(const TcParams &P, int t, int rfirst, int rstep,
                                           int lane, float4 *qacc) {
  const int RQ = P.dims.RQ;
  const int64_t V = P.dims.V;
  const int64_t v0 = static_cast<int64_t>(t) * kTileM + lane * 4;
  const bool vec = (V & 3) == 0 && v0 < V;  // then v0 + 3 < V too
  const int sub = t * (kTileM / kSub) + (lane >> 3);
  for (int r0 = rfirst; r0 < RQ; r0 += rstep * kQBatch) {
    float4 x[kQBatch];
#pragma unroll
    for (int j = 0; j < kQBatch; ++j) {
      const int r = r0 + rstep * j;
      const float *row = P.q_logits + static_cast<int64_t>(r < RQ ? r : 0) * V;
      if (vec) {
        x[j] = __ldg(reinterpret_cast<const float4 *>(row + v0));
      } else {
        x[j].x = v0 < V ? __ldg(row + v0) : 0.0f;
        x[j].y = v0 + 1 < V ? __ldg(row + v0 + 1) : 0.0f;
        x[j].z = v0 + 2 < V ? __ldg(row + v0 + 2) : 0.0f;
        x[j].w = v0 + 3 < V ? __ldg(row + v0 + 3) : 0.0f;
      }
    }
#pragma unroll
    for (int j = 0; j < kQBatch; ++j) {
      const int r = r0 + rstep * j;
      if (r >= RQ) break;  // warp-uniform
      const float xv[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
      float a[4];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool ok = v0 + i < V;
        a[i] = ok ? xv[i] * P.inv_t : -INFINITY;
        bad |= ok && (isnan(xv[i]) || xv[i] == INFINITY);
      }
      float m = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float s = 0.0f;
      if (m > -INFINITY) {
#pragma unroll
        for (int i = 0; i < 4; ++i) s += expf(a[i] - m);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const unsigned bmask = __ballot_sync(0xffffffffu, bad);
      if ((lane & 7) == 0 && sub < P.dims.nsub) {
        const bool sub_bad = ((bmask >> (lane & ~7)) & 0xffu) != 0;
        P.w.part_q[static_cast<int64_t>(r) * P.dims.nsub + sub] =
            sub_bad ? make_float2(NAN, NAN) : make_float2(m, s);
      }
      if (qacc) {
        // this CTA's running (max, sum-exp) of the row: the tile's four
        // subtiles (one per group of eight lanes) combined, then folded
        float tm = m, ts = s;
#pragma unroll
        for (int o = 8; o < 32; o <<= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, tm, o);
          const float os = __shfl_xor_sync(0xffffffffu, ts, o);
          const float mm = fmaxf(tm, om);
          ts = mm > -INFINITY ? (tm > -INFINITY ? ts * expf(tm - mm) : 0.0f) +
                                    (om > -INFINITY ? os * expf(om - mm) : 0.0f)
                              : 0.0f;
          tm = mm;
        }
        if (lane == 0) {
          float4 a = qacc[r];
          if (bmask) {
            a.w = 1.0f;
          } else {
            float M = a.x;
            ff S{a.y, a.z};
            lse_fold(tm, ff_make(ts), M, S);
            a = make_float4(M, S.hi, S.lo, a.w);
          }
          qacc[r] = a;
        }
      }
    }
  }
}

// One epilogue warp's staging box (generic and shared-window addresses).
struct EpiBox {
  float *buf;
  uint32_t saddr;
};

// Writes logits and target partials for columns n0 .. n0+15 of a finished
// tile; this lane holds vocab entry v = vw + lane of the warp's 32 entries
// vw .. vw+31 (one subtile).  The 16 x 32 block goes through a shared-memory
// box: row i holds column n0+i, its 16-byte chunks swizzled by (i mod 8) as
// the TMA 128-byte pattern expects, so both the lanes' writes (one column
// each) and the partial pass's 16-byte reads (half a column each) are free
// of bank conflicts.  One TMA store then writes the box to the logits; the
// partials need one shuffle per reduction instead of a butterfly.
// With P.row_stats the lane pair of column c also folds the subtile's
// (max, sum-exp) into this warp's running pair of the column (accM, accS;
// accBad for NaN or +inf entries).
__device__ __forceinline__ void finish_group(const TcParams &P, const CUtensorMap *tmL,
                                             const EpiBox &bx, const float (&x)[16], int n0,
                                             int64_t vw, int sub, int lane, float &accM,
                                             ff &accS, bool &accBad) {
  const int64_t V = P.dims.V;
  const int R = P.dims.R;
  const bool greedy = P.greedy != 0;
  const int64_t v = vw + lane;
  const bool valid = v < V;
  // FP8: logit = acc * h_scale[row] * w_scale[v]
  const float ws = P.fp8 ? (valid ? __ldg(&P.w_scale[v]) : 0.0f) : 1.0f;
  float l[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int n = n0 + i;
    l[i] = P.fp8 ? __fmul_rn(__fmul_rn(x[i], __ldg(&P.h_scale[n < R ? n : 0])), ws) : x[i];
  }
  float *box = bx.buf;
  const uint32_t sbox = bx.saddr;
  // the previous group's store must have finished reading the box
  if (P.tma_logits && lane == 0) bulk_wait_read0();
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 16; ++i) box[i * 32 + (((lane >> 2) ^ (i & 7)) << 2) + (lane & 3)] = l[i];
  if (P.tma_logits) {
    fence_proxy_async_smem();
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (valid && n0 + i < R) P.w.logits[static_cast<int64_t>(n0 + i) * V + v] = l[i];
  }
  __syncwarp();
  if (P.tma_logits && lane == 0 && vw < V && n0 < R) {
    tma_store_2d(tmL, sbox, static_cast<int32_t>(vw), n0);
    bulk_commit();
  }
  // partials: lane -> column c = lane / 2, entries 16h .. 16h+15 (h = lane % 2).
  // Scalar loads: on this part 16-byte loads of this pattern measured
  // about four times slower.
  const int c = lane >> 1, h = lane & 1;
  float a[16];
  bool bad = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float q = box[c * 32 + (((4 * h + k) ^ (c & 7)) << 2) + j];
      const bool ok = vw + 16 * h + 4 * k + j < V;
      a[4 * k + j] = ok ? (greedy ? q : q * P.inv_t) : -INFINITY;
      bad |= ok && (isnan(q) || q == INFINITY);
    }
  }
  float t8[8], t4[4];
#pragma unroll
  for (int i = 0; i < 8; ++i) t8[i] = fmaxf(a[i], a[i + 8]);
#pragma unroll
  for (int i = 0; i < 4; ++i) t4[i] = fmaxf(t8[i], t8[i + 4]);
  float m = fmaxf(fmaxf(t4[0], t4[2]), fmaxf(t4[1], t4[3]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  float sum = 0.0f;
  if (!greedy) {
    // all entries -inf: every exp is 0 against any finite reference
    const float ref = m > -INFINITY ? m : 0.0f;
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = expf(a[i] - ref);
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] += e[i + 8];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] += e[i + 4];
    sum = (e[0] + e[2]) + (e[1] + e[3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  }
  const unsigned bmask = __ballot_sync(0xffffffffu, bad);
  const int n = n0 + c;
  const bool sub_bad = ((bmask >> (2 * c)) & 3u) != 0;
  // the last tile may end inside a subtile row
  if (h == 0 && n < R && sub < P.dims.nsub)
    P.w.part_p[static_cast<int64_t>(n) * P.dims.nsub + sub] =
        sub_bad ? make_float2(NAN, NAN) : make_float2(m, sum);
  if (P.row_stats && !greedy && sub < P.dims.nsub) {
    if (sub_bad) accBad = true;
    else lse_fold(m, ff_make(sum), accM, accS);
  }
}

// Split-tile hand-off, per warp (each warp owns 32 vocab rows of the tile and
// has its own counter, so no cross-warp barrier is needed): publish this
// CTA's part and learn whether the other part is already there.  Returns
// true (on every lane) if this warp must finish its rows of the tile.
__device__ __forceinline__ bool split_publish(const TcParams &P, int bidx, int quad,
                                              int lane) {
  __threadfence();
  __syncwarp();
  int flag = 0;
  if (lane == 0) flag = atomicAdd(&P.w.split_cnt[bidx * 4 + quad], 1);
  flag = __shfl_sync(0xffffffffu, flag, 0);
  if (flag != 0) __threadfence();
  return flag != 0;
}

__device__ __forceinline__ void split_reset(const TcParams &P, int bidx, int quad, int lane) {
  if (lane == 0) P.w.split_cnt[bidx * 4 + quad] = 0;
}

// Drain mode hands a split tile over in one direction only, so that the
// CTA holding the tile's first k block always finishes it (and the tiles
// each CTA finishes, and the order it finishes them in, do not depend on
// timing).  The later part (published by the next CTA at the start of its
// work) is stored, then flagged; the earlier part waits for the flag
// (bounded; in practice it has long been set) and clears it.
__device__ __forceinline__ void split_hand_over(const TcParams &P, int bidx, int quad, int lane) {
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicExch(&P.w.split_cnt[bidx * 4 + quad], 1);
}

__device__ __forceinline__ bool split_take(const TcParams &P, int bidx, int quad, int lane,
                                           const volatile int *abort) {
  int ok = 1;
  if (lane == 0) {
    const int *flag = &P.w.split_cnt[bidx * 4 + quad];
    auto load = [flag]() {
      int v;
      asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      return v;
    };
    if (load() == 0) {
      const uint64_t t0 = globaltimer();
      while (load() == 0) {
        if (*abort || globaltimer() - t0 >= P.wait_limit_ns) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    if (ok) P.w.split_cnt[bidx * 4 + quad] = 0;
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) __threadfence();
  return ok != 0;
}

template <int NCOL>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmL, const TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  // [stage ring][epilogue boxes][control block]
  const uint32_t epi_off = (base - raw) + static_cast<uint32_t>(P.stages * P.stage_bytes);
  Ctl *ctl = reinterpret_cast<Ctl *>(smem_raw + epi_off + kEpiBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int nkb = P.nkb;
  const int C = P.chunks;
  const int ngr = nkb / C;
  const int64_t U = static_cast<int64_t>(P.dims.ntile) * ngr;
  // half mode: CTAs 2p and 2p+1 take the same units, each for half of the
  // columns (its first column col0); otherwise every CTA its own units
  const int G = P.half ? gridDim.x / 2 : gridDim.x;
  const int c = P.half ? blockIdx.x / 2 : blockIdx.x;
  const int hsel = P.half ? (blockIdx.x & 1) : 0;
  const int col0 = hsel * P.npad;
  const int64_t u0 = U * c / G, u1 = U * (c + 1) / G;
  const int t_first = static_cast<int>(u0 / ngr);
  const int t_last = static_cast<int>((u1 - 1) / ngr);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int s = 0; s < drain_slots<NCOL>(); ++s) {
      mbar_init(smem_u32(&ctl->tfull[s]), 1);
      mbar_init(smem_u32(&ctl->tempty[s]), kNumEpiWarps);
    }
    mbar_init(smem_u32(&ctl->teardown), 1);
    ctl->abort_flag = 0;
    ctl->issued = 0;
    ctl->consumed = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
    if (P.tma_logits) tma_prefetch_desc(&tmL);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), P.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const volatile int *abort = &ctl->abort_flag;

  // Everything above only touched this CTA's own resources; inputs written
  // by earlier work in the stream are visible after this point.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // half mode: the partner CTA reads the same W tile at about the same
      // time, so it keeps normal priority in L2
      const uint64_t pol_w = P.half ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      const uint32_t tx = static_cast<uint32_t>(C * (kWSlabBytes + P.npad * 128));
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      for (int t = t_first; t <= t_last; ++t) {
        int kb0, kb1;
        tile_range(t, u0, u1, ngr, C, kb0, kb1);
        bool ok = true;
        for (int kb = kb0; kb < kb1; kb += C) {
          if (!mbar_wait(smem_u32(&ctl->empty[stage]), phase ^ 1u, P.wait_limit_ns, abort)) {
            raise_abort(ctl, P);
            ok = false;
            break;
          }
          const uint32_t sbase = base + static_cast<uint32_t>(stage * P.stage_bytes);
          const uint32_t full = smem_u32(&ctl->full[stage]);
          mbar_arrive_expect_tx(full, tx);
          if (C > 1) {
            // C consecutive k blocks in one 3-D box: 128 rows x (C x 128 B)
            // contiguous runs; in shared memory C [128 x 64] swizzled tiles
            tma_load_3d(sbase, &tmW, 0, t * kTileM, kb, full, pol_w);
            tma_load_3d(sbase + static_cast<uint32_t>(C * kWSlabBytes), &tmH, 0, col0, kb, full,
                        pol_h);
          } else {
            tma_load_2d(sbase, &tmW, kb * P.kbk, t * kTileM, full, pol_w);
            for (int hb = 0; hb < P.h_boxes; ++hb)
              tma_load_2d(sbase + kWSlabBytes + static_cast<uint32_t>(hb * P.h_box_rows * 128),
                          &tmH, kb * P.kbk, col0 + hb * P.h_box_rows, full, pol_h);
          }
          ++issued;
          if (++stage == P.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      ctl->issued = issued;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs the loop and waits together, so the stage/slot
    // state and the descriptors stay warp-uniform; one elected lane issues
    // the MMAs and commits.  (Issued from a single-lane branch the same
    // sequence costs several times more per k block, which made the issuer,
    // not HBM, the limit for small N.)
    int stage = 0, consumed = 0;
    uint32_t sphase = 0;
    int slot = 0;
    uint32_t tphase = 0;
    bool ok = true;
    // descriptor address fields are (addr >> 4); shared addresses stay
    // below 256 KB, so offsets add without carrying out of the field
    const uint64_t adesc0 = sw128_desc(base);
    const uint64_t bdesc0 = sw128_desc(base + static_cast<uint32_t>(C * kWSlabBytes));
    const uint32_t stage16 = static_cast<uint32_t>(P.stage_bytes >> 4);
    const uint32_t bchunk16 = static_cast<uint32_t>((P.npad * 128) >> 4);
    const int n1 = NCOL != 0 ? P.npad : (P.npad <= 256 ? P.npad : 256);
    const int n2 = P.npad > 256 ? P.npad - 256 : 16;
    const uint32_t idesc = P.fp8 ? idesc_e4m3(kTileM, n1) : idesc_bf16(kTileM, n1);
    const uint32_t idesc2 = P.fp8 ? idesc_e4m3(kTileM, n2) : idesc_bf16(kTileM, n2);
    // one 128-byte row of a stage is 4 instructions of 32 bytes: K = 16
    // bf16 or K = 32 E4M3 each
    auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
      if (P.fp8) umma_f8(d, a, b, id, acc);
      else umma_bf16(d, a, b, id, acc);
    };
    for (int t = t_first; t <= t_last && ok; ++t) {
      int kb0, kb1;
      tile_range(t, u0, u1, ngr, C, kb0, kb1);
      if constexpr (NCOL == 0) {
        // direct mode: tiles alternate between nbuf TMEM buffers of 256
        // columns; tphase bit b is buffer b's phase
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->tempty[slot]),
                                               ((tphase >> slot) & 1u) ^ 1u, P.wait_limit_ns,
                                               abort))) {
          if (lane == 0) raise_abort(ctl, P);
          break;
        }
        tc_fence_after();
      }
      uint64_t adesc = 0, bdesc = 0;
      int j = 0;  // chunk within the current stage (kb0 is a multiple of C)
      // direct mode: accumulator ds = floor(kb * nslot / nkb) of block kb and
      // the first block of the next accumulator, advanced incrementally
      int ds = 0, dnext = 0;
      if constexpr (NCOL == 0) {
        ds = (kb0 * P.nslot) / nkb;
        dnext = ((ds + 1) * nkb + P.nslot - 1) / P.nslot;
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        // drain mode: groups of kblocks_per_slot k blocks share a slot
        const int gpos = (kb - kb0) % kblocks_per_slot<NCOL>();
        const bool group_first = gpos == 0;
        const bool group_last = gpos == kblocks_per_slot<NCOL>() - 1 || kb == kb1 - 1;
        if constexpr (NCOL != 0) {
          if (group_first && slot % tempty_batch<NCOL>() == 0 &&
              !__all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&ctl->tempty[slot + tempty_batch<NCOL>() - 1]),
                                    tphase ^ 1u, P.wait_limit_ns, abort))) {
            if (lane == 0) raise_abort(ctl, P);
            ok = false;
            break;
          }
        }
        if (j == 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->full[stage]), sphase,
                                                 P.wait_limit_ns, abort))) {
            if (lane == 0) raise_abort(ctl, P);
            ok = false;
            break;
          }
          ++consumed;
          adesc = adesc0 + static_cast<uint64_t>(stage) * stage16;
          bdesc = bdesc0 + static_cast<uint64_t>(stage) * stage16;
        }
        tc_fence_after();
        if constexpr (NCOL != 0) {
          const uint32_t d = tmem + static_cast<uint32_t>(slot * NCOL);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(d, adesc + 2u * k, bdesc + 2u * k, idesc, (k > 0 || !group_first) ? 1u : 0u);
            // release the stage first: the producer's refill is on the
            // critical path, the drain of this slot is not
            if (j == C - 1) umma_commit(smem_u32(&ctl->empty[stage]));
            if (group_last) umma_commit(smem_u32(&ctl->tfull[slot]));
          }
          __syncwarp();
          if (group_last && ++slot == drain_slots<NCOL>()) {
            slot = 0;
            tphase ^= 1u;
          }
        } else {
          bool first = kb == kb0;
          if (kb == dnext) {
            ++ds;
            first = true;
            dnext = ((ds + 1) * nkb + P.nslot - 1) / P.nslot;
          }
          const uint32_t d = tmem + static_cast<uint32_t>(slot * 256 + ds * P.npad);
          // npad > 256 only with single-chunk stages
          const uint64_t bdesc2 = bdesc + ((256u * 128u) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t acc = (k > 0 || !first) ? 1u : 0u;
              mma(d, adesc + 2u * k, bdesc + 2u * k, idesc, acc);
              if (P.npad > 256) mma(d + 256u, adesc + 2u * k, bdesc2 + 2u * k, idesc2, acc);
            }
            if (j == C - 1) umma_commit(smem_u32(&ctl->empty[stage]));
          }
          __syncwarp();
        }
        adesc += kWSlabBytes >> 4;
        bdesc += bchunk16;
        if (++j == C) {
          j = 0;
          if (++stage == P.stages) {
            stage = 0;
            sphase ^= 1u;
          }
        }
      }
      if constexpr (NCOL == 0) {
        if (ok) {
          if (elect_one()) umma_commit(smem_u32(&ctl->tfull[slot]));
          __syncwarp();
          tphase ^= 1u << slot;
          if (++slot >= P.nbuf) slot = 0;
        }
      }
    }
    if (lane == 0) ctl->consumed = consumed;
    // every MMA issued by the elected lane must finish before TMEM is
    // freed; a commit tracks the MMAs of the thread that issues it
    if (elect_one()) {
      umma_commit(smem_u32(&ctl->teardown));
      const int never = 0;
      mbar_wait(smem_u32(&ctl->teardown), 0u, kCleanupLimitNs, &never);
    }
    __syncwarp();
  } else if (is_q_warp(warp)) {
    // ---------------- draft-logit partials (independent of the GEMM) -------
    if (!P.greedy && P.dims.RQ > 0) {
      const int quad = q_warp_index(warp);
      // the exact logit of every draft token (one warp each, spread over
      // the grid) and the draft logit at that token; the decision pass reads
      // them instead of recomputing.  First, so that these dependent loads
      // overlap the stream rather than trail it.
      const int K = P.dims.K;
      const int64_t n16 = P.dims.d / (P.fp8 ? 16 : 8);
      for (int idx = static_cast<int>(blockIdx.x) * kNumQWarps + quad; idx < P.dims.RQ;
           idx += static_cast<int>(gridDim.x) * kNumQWarps) {
        const int b = idx / K, i = idx - b * K;
        const int x = P.draft[idx];
        const bool valid = x >= 0 && static_cast<int64_t>(x) < P.dims.V;
        float qx = 0.0f;
        if (lane == 0 && valid && P.q_logits != nullptr)
          qx = __ldg(&P.q_logits[static_cast<int64_t>(idx) * P.dims.V + x]);
        ff l = ff_make(NAN);
        if (valid) {
          const uint4 *h = static_cast<const uint4 *>(P.H) +
                           (static_cast<int64_t>(b) * (K + 1) + i) * n16;
          const uint4 *w = static_cast<const uint4 *>(P.W) + static_cast<int64_t>(x) * n16;
          if (P.fp8) {
            const int64_t r = static_cast<int64_t>(b) * (K + 1) + i;
            l = ff_mul_f(ff_mul_f(dot_e4m3_warp(h, w, 0, n16, lane), __ldg(&P.h_scale[r])),
                         __ldg(&P.w_scale[x]));
          } else {
            l = dot_bf16_warp(h, w, 0, n16, lane);
          }
        }
        if (lane == 0) {
          P.w.draft_logit[idx] = make_float2(l.hi, l.lo);
          if (P.w.draft_q) P.w.draft_q[idx] = qx;
        }
      }
      // row statistics: this warp's draft rows (quad, quad + kNumQWarps, ...) start
      // empty in shared memory (row_stats runs in drain mode only, where
      // RQ < kQaccRows and no CTA pair splits the columns)
      const bool qstats = P.row_stats && P.q_logits != nullptr;
      float4 *qacc = qstats ? ctl->qacc : nullptr;
      if (qstats && lane == 0)
        for (int r = quad; r < P.dims.RQ; r += kNumQWarps)
          qacc[r] = make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
      __syncwarp();
      // no draft distribution (point-mass drafts): nothing to normalise
      for (int t = t_first; t <= t_last && P.q_logits != nullptr; ++t) {
        int kb0, kb1;
        tile_range(t, u0, u1, ngr, C, kb0, kb1);
        if (kb0 != 0) continue;  // the CTA holding a tile's first k block does it
        q_partials(P, t, quad + kNumQWarps * hsel, P.half ? 2 * kNumQWarps : kNumQWarps, lane,
                   qacc);
      }
      __syncwarp();
      if (qstats)
        for (int r = quad + kNumQWarps * lane; r < P.dims.RQ; r += 32 * kNumQWarps)
          P.w.rowpart[static_cast<int64_t>(P.dims.R + r) * gridDim.x + blockIdx.x] = qacc[r];
    }
  } else if (warp < 2 + kNumEpiWarps) {
    // ---------------- epilogue warps ----------------
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t box_off = epi_off + static_cast<uint32_t>(quad * kBoxFloats * 4);
    const EpiBox bx{reinterpret_cast<float *>(smem_raw + box_off), raw + box_off};
    // drain mode with row_stats: this warp's running (max, sum-exp) of each
    // column over the tiles it finishes (lane pair 2c, 2c+1 holds column c
    // of each 16-column group)
    constexpr int kGroups = NCOL != 0 ? NCOL / 16 : 1;
    float accM[kGroups];
    ff accS[kGroups];
    bool accBad[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      accM[g] = -INFINITY;
      accS[g] = ff_make(0.0f);
      accBad[g] = false;
    }
    int slot = 0;
    uint32_t tphase = 0;
    for (int t = t_first; t <= t_last; ++t) {
      int kb0, kb1;
      tile_range(t, u0, u1, ngr, C, kb0, kb1);
      const int64_t vw = static_cast<int64_t>(t) * kTileM + quad * 32;
      const int sub = t * (kTileM / kSub) + quad;
      const bool split = kb0 != 0 || kb1 != nkb;
      // split-tile partner: the CTA of the same half in the neighbouring
      // pair (or the neighbouring CTA)
      const int bidx = P.half ? (kb0 == 0 ? c : c - 1) * 2 + hsel : (kb0 == 0 ? c : c - 1);
      const int part = kb0 == 0 ? 0 : 1;
      float *mine = P.w.split_buf + (static_cast<int64_t>(bidx) * 2 + part) * (kTileM * P.npad);
      float *other =
          P.w.split_buf + (static_cast<int64_t>(bidx) * 2 + (1 - part)) * (kTileM * P.npad);

      if constexpr (NCOL != 0) {
        float acc[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) acc[n] = 0.0f;
        bool ok = true;
        for (int kb = kb0; kb < kb1; kb += kblocks_per_slot<NCOL>()) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->tfull[slot]), tphase,
                                                 P.wait_limit_ns, abort))) {
            if (lane == 0) raise_abort(ctl, P);
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t xr[NCOL / 16][16];
#pragma unroll
          for (int g = 0; g < NCOL / 16; ++g)
            tmem_ld16(tmem + lane_addr + static_cast<uint32_t>(slot * NCOL + g * 16), xr[g]);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < NCOL / 16; ++g) tmem_reg_fence(xr[g]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[slot]));
          // one k block's exact-product chunk (4 MMAs); the running sum is
          // rounded to nearest, so its errors are unbiased
#pragma unroll
          for (int n = 0; n < NCOL; ++n) acc[n] = __fadd_rn(acc[n], __uint_as_float(xr[n / 16][n % 16]));
          if (++slot == drain_slots<NCOL>()) {
            slot = 0;
            tphase ^= 1u;
          }
        }
        if (!ok) break;
        float val[NCOL];
#pragma unroll
        for (int n = 0; n < NCOL; ++n) val[n] = acc[n];
        if (split) {
          if (part == 1) {
            // the tile's later k blocks: handed to the CTA that holds its
            // first k block, which finishes the tile
#pragma unroll
            for (int n = 0; n < NCOL; ++n)
              if (n < P.npad) mine[n * kTileM + row_in_tile] = val[n];
            split_hand_over(P, bidx, quad, lane);
            continue;
          }
          if (!split_take(P, bidx, quad, lane, abort)) {
            if (lane == 0) raise_abort(ctl, P);
            break;
          }
#pragma unroll
          for (int n = 0; n < NCOL; ++n)
            if (n < P.npad) val[n] = val[n] + __ldcg(&other[n * kTileM + row_in_tile]);
        }
#pragma unroll
        for (int g = 0; g < NCOL / 16; ++g) {
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = val[g * 16 + i];
          finish_group(P, &tmL, bx, x, col0 + g * 16, vw, sub, lane, accM[g], accS[g],
                       accBad[g]);
        }
      } else {
        // direct mode: sum the tile's accumulators column group by group
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->tfull[slot]),
                                               (tphase >> slot) & 1u, P.wait_limit_ns, abort))) {
          if (lane == 0) raise_abort(ctl, P);
          break;
        }
        tc_fence_after();
        const int s_lo = (kb0 * P.nslot) / nkb;
        const int s_hi = ((kb1 - 1) * P.nslot) / nkb;
        for (int g = 0; g < P.npad / 16; ++g) {
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = 0.0f;
          // the tile's accumulators (at most four), two per round of loads
#pragma unroll
          for (int j0 = 0; j0 < 4; j0 += 2) {
            if (s_lo + j0 > s_hi) break;
            uint32_t y[2][16];
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (s_lo + j0 + j <= s_hi)
                tmem_ld16(tmem + lane_addr +
                              static_cast<uint32_t>(slot * 256 + (s_lo + j0 + j) * P.npad + g * 16),
                          y[j]);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              if (s_lo + j0 + j <= s_hi) {
                tmem_reg_fence(y[j]);
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] += __uint_as_float(y[j][i]);
              }
            }
          }
          if (split) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[(g * 16 + i) * kTileM + row_in_tile] = x[i];
          } else {
            finish_group(P, &tmL, bx, x, col0 + g * 16, vw, sub, lane, accM[0], accS[0],
                         accBad[0]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[slot]));
        tphase ^= 1u << slot;
        if (++slot >= P.nbuf) slot = 0;
        if (split) {
          if (!split_publish(P, bidx, quad, lane)) continue;
          for (int g = 0; g < P.npad / 16; ++g) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int idx = (g * 16 + i) * kTileM + row_in_tile;
              x[i] = __ldcg(&mine[idx]) + __ldcg(&other[idx]);
            }
            finish_group(P, &tmL, bx, x, col0 + g * 16, vw, sub, lane, accM[0], accS[0],
                         accBad[0]);
          }
          split_reset(P, bidx, quad, lane);
        }
      }
    }
    // the logits stores must be complete (and done reading the boxes)
    // before the kernel ends
    if (P.tma_logits && lane == 0) bulk_wait_all();
    __syncwarp();
    if constexpr (NCOL != 0) {
      if (P.row_stats && !P.greedy) {
        // the four warps' running pairs through their (now idle) staging
        // boxes; thread i of the four warps then writes column i's pair for
        // this CTA
        float4 *mine4 = reinterpret_cast<float4 *>(bx.buf);
        if ((lane & 1) == 0) {
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            mine4[g * 16 + (lane >> 1)] =
                make_float4(accM[g], accS[g].hi, accS[g].lo, accBad[g] ? 1.0f : 0.0f);
        }
        named_bar_sync(1, 32 * kNumEpiWarps);
        const int i = (warp - 2) * 32 + lane;
        if (i < NCOL && col0 + i < P.dims.R) {
          float M = -INFINITY;
          ff S = ff_make(0.0f);
          bool bad = false;
#pragma unroll
          for (int w = 0; w < kNumEpiWarps; ++w) {
            const float4 e =
                reinterpret_cast<const float4 *>(smem_raw + epi_off + w * kBoxFloats * 4)[i];
            bad |= e.w != 0.0f;
            lse_fold(e.x, ff{e.y, e.z}, M, S);
          }
          P.w.rowpart[static_cast<int64_t>(col0 + i) * gridDim.x + blockIdx.x] =
              make_float4(M, S.hi, S.lo, bad ? 1.0f : 0.0f);
        }
      }
    }
  }

  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    // only after an abort can loads still be in flight: wait for them so
    // no copy lands in shared memory after this CTA has exited
    const int never = 0;
    for (int i = ctl->consumed; i < ctl->issued; ++i)
      mbar_wait(smem_u32(&ctl->full[i % P.stages]),
                static_cast<uint32_t>((i / P.stages) & 1), kCleanupLimitNs, &never);
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, P.tmem_cols);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
TcPlan plan_tc(const Dims &dims, int num_sms, int smem_optin, int elt) {
  TcPlan pl{};
  const int npad_all = ((dims.R + 15) / 16) * 16;
  pl.ncol = npad_all <= 16 ? 16 : npad_all <= 32 ? 32 : npad_all <= 64 ? 64 : 0;
  // half mode (direct mode above SV_TC_HALF_MIN columns): the two CTAs of a
  // pair take the same tiles, each for half of the columns, so each loads
  // half of the hidden-row block into shared memory and holds two
  // half-width tiles in TMEM
  pl.half = (pl.ncol == 0 && npad_all > SV_TC_HALF_MIN && num_sms >= 2) ? 1 : 0;
  pl.npad = pl.half ? ((npad_all / 2 + 15) / 16) * 16 : npad_all;
  pl.kbk = 128 / elt;  // elements in one 128-byte row of a block
  pl.nkb = static_cast<int>((dims.d + pl.kbk - 1) / pl.kbk);
  const int ctl_bytes = static_cast<int>(sizeof(tc::Ctl)) + tc::kEpiBytes;
  const int budget = smem_optin - 1024 - ctl_bytes;
  // Stages of C consecutive k blocks, loaded as one 3-D box (longer
  // contiguous DRAM runs per W row); needs d a multiple of 64 * C and the
  // hidden slab in one box (npad <= 256).
  pl.chunks = 1;
  if (dims.d % pl.kbk == 0 && pl.npad <= 256) {
    for (int cand = SV_TC_MAX_CHUNKS; cand >= 2; cand /= 2) {
      const int sb = ((cand * (tc::kWSlabBytes + pl.npad * 128) + 1023) / 1024) * 1024;
      if (pl.nkb % cand == 0 && 2 * sb <= budget) {
        pl.chunks = cand;
        break;
      }
    }
  }
  const int max_stages = pl.chunks == 4 ? SV_TC_STAGES_C4
                         : pl.chunks == 2 ? SV_TC_STAGES_C2 : tc::kMaxStages;
  pl.stage_bytes = ((pl.chunks * (tc::kWSlabBytes + pl.npad * 128) + 1023) / 1024) * 1024;
  int stages = budget / pl.stage_bytes;
  if (stages > max_stages) stages = max_stages;
  pl.stages = stages;
  pl.smem = stages * pl.stage_bytes + ctl_bytes + 1024;
  // above half of the SM's shared memory: exactly one CTA per SM, so the
  // TMEM allocation below can never wait on another CTA
  if (pl.smem < 120 * 1024) pl.smem = 120 * 1024;
  pl.h_boxes = pl.npad <= 256 ? 1 : 2;
  pl.h_box_rows = pl.npad <= 256 ? pl.npad : pl.npad / 2;
  if (pl.ncol != 0) {
    pl.nslot = 1;
    pl.nbuf = 1;
    const int slots = pl.ncol == 16 ? tc::drain_slots<16>()
                      : pl.ncol == 32 ? tc::drain_slots<32>() : tc::drain_slots<64>();
    int cols = 32;
    while (cols < slots * pl.ncol) cols *= 2;  // TMEM allocations are powers of two
    pl.tmem_cols = static_cast<uint32_t>(cols);
  } else {
    // contiguous k ranges, one per accumulator; never more accumulators
    // than k blocks, so every accumulator of a tile range receives a block.
    // Up to 256 columns two tiles fit (the MMA fills one while the
    // epilogue drains the other).
    pl.nbuf = pl.npad <= 256 ? 2 : 1;
    int ns = (pl.nbuf == 2 ? 256 : 512) / pl.npad;
    ns = ns < 1 ? 1 : (ns > 4 ? 4 : ns);
    pl.nslot = ns < pl.nkb ? ns : pl.nkb;
    pl.tmem_cols = 512;
  }
  if (pl.half) {
    const int pairs = dims.ntile < num_sms / 2 ? dims.ntile : num_sms / 2;
    pl.grid = 2 * pairs;
  } else {
    pl.grid = dims.ntile < num_sms ? dims.ntile : num_sms;
  }
  pl.threads = tc::kThreads;
  pl.valid = stages >= 2 && npad_all <= SV_MAX_ROWS_BF16;
  return pl;
}

// Dynamic shared memory each kernel variant has been opted in to, per
// device (the attribute is a per-device setting).  Atomics: handles on
// several host threads may launch at once; two threads that both raise the
// attribute set the same value.
constexpr int kAttrDevices = 64;
static std::atomic<int> g_attr_smem[kAttrDevices][4];

cudaError_t launch_tc(const TcPlan &pl, const TcParams &P, const CUtensorMap &tmW,
                      const CUtensorMap &tmH, const CUtensorMap &tmL, cudaStream_t stream) {
  const void *fn;
  int which;
  switch (pl.ncol) {
    case 16: fn = reinterpret_cast<const void *>(&tc::lmhead_tc_kernel<16>); which = 0; break;
    case 32: fn = reinterpret_cast<const void *>(&tc::lmhead_tc_kernel<32>); which = 1; break;
    case 64: fn = reinterpret_cast<const void *>(&tc::lmhead_tc_kernel<64>); which = 2; break;
    default: fn = reinterpret_cast<const void *>(&tc::lmhead_tc_kernel<0>); which = 3; break;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::atomic<int> *done = dev < kAttrDevices ? &g_attr_smem[dev][which] : nullptr;
  if (!done || done->load(std::memory_order_acquire) < pl.smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    if (done) {
      int cur = done->load(std::memory_order_relaxed);
      while (cur < pl.smem && !done->compare_exchange_weak(cur, pl.smem)) {
      }
    }
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(pl.threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(pl.smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {const_cast<CUtensorMap *>(&tmW), const_cast<CUtensorMap *>(&tmH),
                  const_cast<CUtensorMap *>(&tmL), const_cast<TcParams *>(&P)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv
