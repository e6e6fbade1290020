// sv_tail.cu -- kernels (b) and (c) of the verify step, fused into one
// launch that follows the LM-head contraction.
//
// CTAs take tickets from a device counter, so a CTA with a lower ticket is
// known to be running before any CTA with a higher ticket starts waiting:
//
//  row CTAs (tickets 0 .. R+RQ-1), one per target row (logits / T) and per
//      draft row (q_logits / T): combine the per-32-entry softmax partials
//      into the row maximum M and sum S = sum_v exp(x_v - M); a draft-row
//      CTA also recomputes its draft token's logit with a compensated dot
//      product.  The last row CTA of a sequence becomes its decider: it
//      evaluates the K accept thresholds in parallel and walks the
//      draft left to right, x_{i+1} surviving iff u_i < p_{i+1}(x) /
//      q_{i+1}(x) ("Speculative Decoding: Two Models, One Voice", "The idea"
//      step 3; "Speculative Decoding" (library wiki), "One speculation
//      round"), writes the accepted prefix and publishes the row of the
//      final draw.  At T == 0 it runs greedy verification instead, with an
//      exact re-ranking of the near-maximal logits ("Speculative Decoding:
//      Guess Several Tokens, Check Them in One Pass", Step 2).
//  chunk CTAs (higher tickets), one per 4096-entry vocabulary chunk and
//      sequence: wait (bounded) for the decision, compute the chunk's mass
//      of max(0, p_j - q_j) (or of p_{K+1} for the bonus) with 128-bit
//      loads; the last chunk CTA of a sequence inverts the CDF: the smallest
//      v with u * S < C_v, falling back to p_j when the residual is empty
//      ("What Actually Happens During Speculative Decoding in LLMs",
//      speculative_sample_step).
//
// All arithmetic is fp32 or float-float (hi + lo pairs carried with
// error-free transforms): with the row statistics (M, S), exp(M - LSE) is
// 1 / S, and the accept threshold is p/q = exp(delta) * S_q / S_p with
// delta = (l / T - M_p) - (ql / T - M_q), evaluated as expf of delta's head
// times (1 + its tail).  No transcendental function needs more than fp32.
#include <cuda_bf16.h>

#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {

// ---------------------------------------------------------------------------
// Block-level helpers (kTailThreads threads; block_sum_ff and block_max_f
// live in sv_internal.cuh)
// ---------------------------------------------------------------------------
// Exclusive prefix sum over the block, in thread order (float-float).
__device__ __forceinline__ ff block_excl_scan_ff(ff x, ff *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ff inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff y = ff_shfl_up(inc, o);
    if (lane >= o) inc = ff_add(y, inc);
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    ff t = lane < kTailWarps ? s_warp[lane] : ff_make(0.0f);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff y = ff_shfl_up(t, o);
      if (lane >= o) t = ff_add(y, t);
    }
    if (lane < kTailWarps) s_warp[lane] = t;
  }
  __syncthreads();
  const ff before = warp > 0 ? s_warp[warp - 1] : ff_make(0.0f);
  return ff_add(before, ff_add(inc, ff_neg(x)));
}

// Bounded wait until *flag == value (one thread).
__device__ __forceinline__ bool wait_flag(const unsigned *flag, unsigned value,
                                          uint64_t limit_ns) {
  const volatile unsigned *f = flag;
  if (*f == value) return true;
  const uint64_t t0 = globaltimer();
  while (*f != value) {
    if (globaltimer() - t0 >= limit_ns) return false;
    __nanosleep(32);
  }
  return true;
}

__device__ __forceinline__ ff ld_ff(const float2 *p) {
  const float2 v = __ldcg(p);
  return ff{v.x, v.y};
}
__device__ __forceinline__ void st_ff(float2 *p, ff v) { *p = make_float2(v.hi, v.lo); }

// ---------------------------------------------------------------------------
// Dot products and the greedy argmax
// ---------------------------------------------------------------------------

// Part `part` of `nparts` (contiguous ranges of 16-byte vectors) of the dot
// product of hidden row `hrow` with W row `wrow`, by one warp with 16-byte
// loads (rows are 16-byte aligned: d is a multiple of 8 for bf16, of 4 for
// fp32, and the base pointers are 16-byte aligned).  The result is a
// float-float accurate to about 2^-40 of the row's sum of |h * w|; every
// lane returns the same value, and the parts sum to the whole in a fixed
// order.
__device__ ff dot_warp(const TailParams &P, int64_t hrow, int64_t wrow, int lane, int part = 0,
                       int nparts = 1) {
  const int64_t d = P.dims.d;
  float s = 0.0f, c = 0.0f;
  constexpr int kBatch = 4;
  if (P.dtype == SV_FP8) {
    // FP8 LM head: the exact dot of the E4M3 values times both scales
    const uint4 *h = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.H) + hrow * d);
    const uint4 *w = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.W) + wrow * d);
    const int64_t n = d / 16;
    const ff raw = dot_e4m3_warp(h, w, n * part / nparts, n * (part + 1) / nparts, lane);
    return ff_mul_f(ff_mul_f(raw, __ldg(&P.h_scale[hrow])), __ldg(&P.w_scale[wrow]));
  } else if (P.dtype == SV_BF16) {
    const uint4 *h =
        reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(P.H) + hrow * d);
    const uint4 *w =
        reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(P.W) + wrow * d);
    const int64_t n = d / 8;
    return dot_bf16_warp(h, w, n * part / nparts, n * (part + 1) / nparts, lane);
  } else {
    const float4 *h = reinterpret_cast<const float4 *>(static_cast<const float *>(P.H) + hrow * d);
    const float4 *w = reinterpret_cast<const float4 *>(static_cast<const float *>(P.W) + wrow * d);
    const int64_t n = d / 4;
    const int64_t lo = n * part / nparts, hi = n * (part + 1) / nparts;
    for (int64_t k0 = lo; k0 < hi; k0 += 32 * kBatch) {
      float4 hv[kBatch], wv[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int64_t k = k0 + j * 32 + lane;
        hv[j] = k < hi ? __ldg(&h[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
        wv[j] = k < hi ? __ldg(&w[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        acc_product(hv[j].x, wv[j].x, s, c);
        acc_product(hv[j].y, wv[j].y, s, c);
        acc_product(hv[j].z, wv[j].z, s, c);
        acc_product(hv[j].w, wv[j].w, s, c);
      }
    }
  }
  // renormalise this lane's pair, then sum the lanes
  const float hi = __fadd_rn(s, c);
  return warp_sum_ff(ff{hi, __fsub_rn(c, __fsub_rn(hi, s))});
}

// Greedy argmax of target row r with ties to the smallest id.  Only entries
// whose fp32 logit is within eps of the row maximum can be the argmax (the
// fp32 logits are far more accurate than eps); the row CTA listed the
// subtiles holding such entries, and those entries are re-ranked here with
// the exact dot product.  If the list overflowed, every subtile is scanned.
__device__ __forceinline__ float greedy_eps(float M) { return 1e-3f + 1e-5f * fabsf(M); }

__device__ int exact_argmax(const TailParams &P, int64_t r, float M, int lane) {
  const int nsub = P.dims.nsub;
  const int64_t V = P.dims.V;
  const float2 *part = P.w.part_p + r * nsub;
  const float thr = M - greedy_eps(M);
  const int *cand = P.w.cand + r * (1 + kMaxCand);
  const int ncand = __ldcg(&cand[0]);
  const bool listed = ncand <= kMaxCand;
  const int n = listed ? ncand : nsub;
  ff best = ff_make(-INFINITY);
  int best_v = 0x7fffffff;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    int sub = -1;
    if (i < n) sub = listed ? __ldcg(&cand[1 + i]) : i;
    const bool ok = sub >= 0 && (listed || __ldcg(&part[sub].x) >= thr);
    unsigned subs = __ballot_sync(0xffffffffu, ok);
    while (subs) {
      const int src = __ffs(subs) - 1;
      subs &= subs - 1;
      const int sc = __shfl_sync(0xffffffffu, sub, src);
      const int64_t v = static_cast<int64_t>(sc) * kSub + lane;
      unsigned hit =
          __ballot_sync(0xffffffffu, v < V && __ldcg(&P.w.logits[r * V + v]) >= thr);
      while (hit) {
        const int64_t vv = static_cast<int64_t>(sc) * kSub + __ffs(hit) - 1;
        hit &= hit - 1;
        const ff e = dot_warp(P, r, vv, lane);
        const bool same = e.hi == best.hi && e.lo == best.lo;
        if (ff_lt(best, e) || (same && vv < best_v)) {
          best = e;
          best_v = static_cast<int>(vv);
        }
      }
    }
  }
  return best_v == 0x7fffffff ? -1 : best_v;
}

// ---------------------------------------------------------------------------
// Draw weights
// ---------------------------------------------------------------------------

// Weight of vocabulary entry v in the final draw: max(0, p - q) for a
// residual, p for a bonus; for a point-mass draft's residual, p with the
// proposed token's entry removed (max(0, p - 1) = 0 there).
// p(v) = exp(l / T - LSE) is evaluated as exp(l * inv_t - M) * (1 / S) with M
// the row maximum, so the fp32 argument stays small near the mass; the
// explicit _rn operations keep the value bit-identical wherever it is
// recomputed.
__device__ __forceinline__ float draw_weight(const SeqState &st, int64_t v, float l, float ql,
                                             float inv_t) {
  // truncated sampling: entries below a row's cut have no mass (the cut is
  // -inf for an untruncated row)
  const float p = l >= st.p_tau ? __fmul_rn(expf(fmaf(l, inv_t, -st.p_max)), st.p_corr) : 0.0f;
  if (st.mode == kModeResidual) {
    const float q =
        ql >= st.q_tau ? __fmul_rn(expf(fmaf(ql, inv_t, -st.q_max)), st.q_corr) : 0.0f;
    return fmaxf(__fsub_rn(p, q), 0.0f);
  }
  if (st.mode == kModeResidualPoint && v == st.q_row) return 0.0f;
  return p;
}

// The kChunkPerThread consecutive weights of this thread in chunk `chunk`,
// and their sum (in index order).
__device__ __forceinline__ float chunk_weights(const TailParams &P, const SeqState &st,
                                               int chunk, float (&r)[kChunkPerThread]) {
  const int64_t V = P.dims.V;
  const int64_t v0 = static_cast<int64_t>(chunk) * kChunk + threadIdx.x * kChunkPerThread;
  const float *lrow = P.w.logits + static_cast<int64_t>(st.p_row) * V;
  const bool resid = st.mode == kModeResidual;
  const float *qrow = resid ? P.q_logits + static_cast<int64_t>(st.q_row) * V : nullptr;
  float l[kChunkPerThread], q[kChunkPerThread];
  if ((V & 3) == 0 && v0 + kChunkPerThread <= V) {
    const float4 *l4 = reinterpret_cast<const float4 *>(lrow + v0);
#pragma unroll
    for (int j = 0; j < kChunkPerThread / 4; ++j) {
      const float4 a = __ldcg(&l4[j]);
      l[4 * j] = a.x; l[4 * j + 1] = a.y; l[4 * j + 2] = a.z; l[4 * j + 3] = a.w;
    }
    if (resid) {
      const float4 *q4 = reinterpret_cast<const float4 *>(qrow + v0);
#pragma unroll
      for (int j = 0; j < kChunkPerThread / 4; ++j) {
        const float4 a = q4[j];
        q[4 * j] = a.x; q[4 * j + 1] = a.y; q[4 * j + 2] = a.z; q[4 * j + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kChunkPerThread; ++j) q[j] = 0.0f;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kChunkPerThread; ++j) {
      const bool in = v0 + j < V;
      l[j] = in ? __ldcg(&lrow[v0 + j]) : 0.0f;
      q[j] = (in && resid) ? qrow[v0 + j] : 0.0f;
    }
  }
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) {
    r[j] = v0 + j < V ? draw_weight(st, v0 + j, l[j], q[j], P.inv_t) : 0.0f;
    sum = __fadd_rn(sum, r[j]);
  }
  return sum;
}

// ---------------------------------------------------------------------------
// The accept threshold p / q from row statistics (see the file comment).
// lp = l / T - M_p and lq = ql / T - M_q as float-floats, ratio = S_q / S_p.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float accept_threshold(ff lp, ff lq, float ratio) {
  if (lq.hi == -INFINITY) return lp.hi == -INFINITY ? 0.0f : INFINITY;  // q(x) == 0
  const ff delta = ff_add(lp, ff_neg(lq));
  if (!(delta.hi < 80.0f)) return INFINITY;  // far above 1: accepted for any u
  if (delta.hi < -120.0f) return 0.0f;       // below every uniform on the 2^-24 grid
  return __fmul_rn(__fmul_rn(expf(delta.hi), __fadd_rn(1.0f, delta.lo)), ratio);
}

// ---------------------------------------------------------------------------
// Decider (one CTA, the last row CTA of sequence b)
// ---------------------------------------------------------------------------
// Per-sequence finalisation.  The decision (row phase) and the last chunk
// CTA of the residual-mass phase both arrive on seq_final[b]; the second to
// arrive finalises the sequence.  A chunk CTA whose wait for the decision
// ran out contributed no mass, so it sets the poison bit and the sequence
// is reported as -1 instead of drawing from an incomplete distribution.
constexpr int kArrivalMask = 0xffff;
constexpr int kPoisoned = 1 << 16;
enum : int { kFinNone = 0, kFinSelect = 1, kFinPoison = 2 };

// thread 0 only
__device__ __forceinline__ int arrive_final(const TailParams &P, int b) {
  const int prev = atomicAdd(&P.w.seq_final[b], 1);
  if ((prev & kArrivalMask) != 1) return kFinNone;
  P.w.seq_final[b] = 0;  // both arrived: rewind for the next launch
  __threadfence();
  return (prev & kPoisoned) ? kFinPoison : kFinSelect;
}

// Row statistics of sequence b from the contraction's per-CTA pairs (fast
// mode): target rows i = 0..K and, with draft logits, draft rows 0..K-1.
// Warps 2.. take the rows (warps 0 and 1 load the decision's other inputs
// meanwhile); a warp folds the grid_parts pairs of its row (up to eight per
// lane, loaded at once) and then across lanes.  The results go to shared
// memory and to row_m / row_s (which spec_verify_debug_lse reads).  A NaN
// or +inf entry anywhere in a row makes its maximum NaN.
constexpr int kMaxParts = 256;
__device__ void fast_row_stats(const TailParams &P, int b, float *s_lp_m, ff *s_lp_s,
                               float *s_lq_m, ff *s_lq_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = P.dims.K, R = P.dims.R, G = P.grid_parts;
  const int nstat = P.q_logits ? 2 * K + 1 : K + 1;
  constexpr int kStatWarps = kTailWarps - 2;
  for (int j = warp - 2; j >= 0 && j < nstat; j += kStatWarps) {
    const int64_t row = j <= K ? static_cast<int64_t>(b) * (K + 1) + j
                               : static_cast<int64_t>(R) + static_cast<int64_t>(b) * K + (j - K - 1);
    const float4 *src = P.w.rowpart + row * G;
    float4 e[kMaxParts / 32];
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k) {
      const int c = lane + 32 * k;
      e[k] = c < G ? __ldcg(&src[c]) : make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
    }
    float M = -INFINITY;
    ff S = ff_make(0.0f);
    bool bad = false;
#pragma unroll
    for (int k = 0; k < kMaxParts / 32; ++k) {
      bad |= e[k].w != 0.0f;
      lse_fold(e[k].x, ff{e[k].y, e[k].z}, M, S);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, M, o);
      const ff os = ff_shfl_xor(S, o);
      lse_fold(om, os, M, S);
    }
    if (__any_sync(0xffffffffu, bad)) M = NAN;
    if (lane == 0) {
      if (j <= K) {
        s_lp_m[j] = M;
        s_lp_s[j] = S;
      } else {
        s_lq_m[j - K - 1] = M;
        s_lq_s[j - K - 1] = S;
      }
      P.w.row_m[row] = M;
      st_ff(&P.w.row_s[row], S);
    }
  }
  if (!P.q_logits && warp == 1) {
    // drafts proposed with certainty: the draft rows are neutral (M = 0, S = 1)
    for (int i = lane; i < K; i += 32) {
      const int64_t row = static_cast<int64_t>(R) + static_cast<int64_t>(b) * K + i;
      s_lq_m[i] = 0.0f;
      s_lq_s[i] = ff_make(1.0f);
      P.w.row_m[row] = 0.0f;
      st_ff(&P.w.row_s[row], ff_make(1.0f));
    }
  }
}

// Returns (to every thread of the block) what this CTA must finalise.
// With `local` (cooperative selection: every chunk CTA of the sequence
// takes the same decision from the same inputs) the decision goes to that
// shared-memory state instead of being published, and the accepted prefix
// and count are written only if `emit` (by one of the CTAs).
// kCoop compiles the cooperative path alone (sampling, no truncation, no
// tree, row statistics from the contraction's pairs).
template <bool kCoop>
__device__ int decide(const TailParams &P, int b, SeqState *local = nullptr, bool emit = true) {
  const bool greedy = !kCoop && P.greedy;
  const int32_t *parents = kCoop ? nullptr : P.parents;
  const int p_cut = kCoop ? 0 : P.p_cut, q_cut = kCoop ? 0 : P.q_cut;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = P.dims.K, rows = K + 1;
  const int64_t V = P.dims.V;
  const int R = P.dims.R;
  const int64_t out0 = static_cast<int64_t>(b) * rows;
  __shared__ ff s_l[SV_MAX_K];           // draft-token logits
  __shared__ int s_acc[SV_MAX_K];        // 1 accept, 0 reject, -1 non-finite
  __shared__ float s_lp_m[SV_MAX_K + 1], s_lq_m[SV_MAX_K];    // row maxima
  __shared__ ff s_lp_s[SV_MAX_K + 1], s_lq_s[SV_MAX_K];       // row sums
  __shared__ float s_ql[SV_MAX_K], s_u[SV_MAX_K + 1];
  __shared__ int s_x[SV_MAX_K], s_arg[SV_MAX_K + 1];
  __shared__ float s_tp[SV_MAX_K + 1], s_tq[SV_MAX_K], s_lbuf[SV_MAX_K];  // cuts, L[x]
  __shared__ int s_err, s_fin, s_kb;
  // no draft distribution: the draft was proposed with certainty (q is a
  // point mass at each proposed token) and a -1 ends it early (not for a
  // tree, whose nodes all carry tokens)
  const bool point = P.q_logits == nullptr && parents == nullptr;
  __shared__ int s_par[SV_MAX_K];               // tree: node parents
  __shared__ int s_depth[SV_MAX_K + 1];         // tree: depth of root / nodes
  __shared__ unsigned char s_match[SV_MAX_K + 1];

  // fast mode: this CTA computes the row statistics itself (warps 2..)
  const bool fast = kCoop || P.fast != 0;
  if (threadIdx.x == 0) s_err = 0;
  __syncthreads();
  // everything the walk needs, loaded in parallel
  if (threadIdx.x < rows) {
    const int i = threadIdx.x;
    s_tp[i] = p_cut ? __ldcg(&P.w.row_tau[out0 + i]) : -INFINITY;
    if (!fast) {
      s_lp_m[i] = __ldcg(&P.w.row_m[out0 + i]);
      s_lp_s[i] = ld_ff(&P.w.row_s[out0 + i]);
    }
    if (!greedy) s_u[i] = P.u[out0 + i];
    if (!fast) {
      const bool fin = isfinite(s_lp_m[i]) &&
                       (greedy || (s_lp_s[i].hi > 0.0f && s_lp_s[i].hi < INFINITY));
      if (!fin) atomicCAS(&s_err, 0, SV_ERR_NONFINITE);
    }
  }
  if (threadIdx.x >= 32 && threadIdx.x < 32 + K) {
    const int i = threadIdx.x - 32;
    const int x = P.draft[static_cast<int64_t>(b) * K + i];
    // fast mode: the draft logit at the token and the token's exact logit
    // do not depend on x; load them together with it
    float ql_fast = 0.0f;
    ff l_fast = ff_make(0.0f);
    if (fast && !greedy) {
      ql_fast = point ? 0.0f : __ldcg(&P.w.draft_q[static_cast<int64_t>(b) * K + i]);
      l_fast = ld_ff(&P.w.draft_logit[static_cast<int64_t>(b) * K + i]);
    }
    s_x[i] = x;
    if (parents) {
      // a parent must come before its child
      const int pa = parents[static_cast<int64_t>(b) * K + i];
      s_par[i] = pa;
      if (pa < -1 || pa >= i) atomicExch(&s_err, SV_ERR_TOKEN);
    }
    if (point && x == -1) {
      // end of a short draft (checked below)
    } else if (x < 0 || static_cast<int64_t>(x) >= V) {
      atomicExch(&s_err, SV_ERR_TOKEN);
    } else if (!greedy) {
      // a point-mass draft row holds M = 0, S = 1 and q_logits(x) counts
      // as 0, so the threshold below is p(x) / 1
      const int64_t rq = static_cast<int64_t>(R) + static_cast<int64_t>(b) * K + i;
      if (!fast) {
        s_lq_m[i] = __ldcg(&P.w.row_m[rq]);
        s_lq_s[i] = ld_ff(&P.w.row_s[rq]);
      }
      // fast mode: the contraction also left q_logits at the draft token
      s_ql[i] = point ? 0.0f : fast ? ql_fast : P.q_logits[(static_cast<int64_t>(b) * K + i) * V + x];
      // truncated sampling: membership of x is decided on the same fp32
      // values the cut was found on
      s_tq[i] = q_cut ? __ldcg(&P.w.row_tau[rq]) : -INFINITY;
      s_lbuf[i] = p_cut ? __ldcg(&P.w.logits[(out0 + i) * V + x]) : 0.0f;
      s_l[i] = fast ? l_fast : ld_ff(&P.w.draft_logit[static_cast<int64_t>(b) * K + i]);
      if (!fast) {
        const bool fin = isfinite(s_lq_m[i]) && s_lq_s[i].hi > 0.0f && s_lq_s[i].hi < INFINITY;
        if (!fin) atomicCAS(&s_err, 0, SV_ERR_NONFINITE);
      }
    }
  }
  if (threadIdx.x == 64 &&
      *reinterpret_cast<volatile unsigned *>(P.w.abort_epoch) == P.epoch) {
    // a contraction that gave up in this run leaves the partials undefined
    atomicExch(&s_err, SV_ERR_TIMEOUT);
  }
  if (fast) fast_row_stats(P, b, s_lp_m, s_lp_s, s_lq_m, s_lq_s);
  __syncthreads();
  if (fast) {
    // the finiteness checks of the row statistics just computed
    if (threadIdx.x < rows) {
      const int i = threadIdx.x;
      const bool fin = isfinite(s_lp_m[i]) && s_lp_s[i].hi > 0.0f && s_lp_s[i].hi < INFINITY;
      if (!fin) atomicCAS(&s_err, 0, SV_ERR_NONFINITE);
    }
    if (threadIdx.x >= 32 && threadIdx.x < 32 + K) {
      const int i = threadIdx.x - 32;
      const int x = s_x[i];
      if (x >= 0 && static_cast<int64_t>(x) < V) {
        const bool fin = isfinite(s_lq_m[i]) && s_lq_s[i].hi > 0.0f && s_lq_s[i].hi < INFINITY;
        if (!fin) atomicCAS(&s_err, 0, SV_ERR_NONFINITE);
      }
    }
  }
  if (threadIdx.x == 0) {
    // proposed tokens of this sequence: K, or the position of the first -1
    // of a point-mass draft, after which every entry must be -1 too
    int kb = K;
    if (point)
      for (int i = 0; i < K && kb == K; ++i)
        if (s_x[i] == -1) kb = i;
    for (int i = kb; i < K; ++i)
      if (s_x[i] != -1) atomicExch(&s_err, SV_ERR_TOKEN);
    s_kb = kb;
  }
  __syncthreads();
  const int kb = s_kb;
  if (s_err == SV_ERR_TIMEOUT && b == 0) {
    // the aborted contraction may have left split-tile counters half-used
    for (int i = threadIdx.x; i < P.split_cnt_n; i += kTailThreads) P.w.split_cnt[i] = 0;
  }
  if (s_err == 0) {
    if (!greedy) {
      // accept thresholds of the proposed positions, one thread each
      if (threadIdx.x < kb) {
        const int i = threadIdx.x;
        const float T = static_cast<float>(P.T);
        const ff l = s_l[i];
        const ff lp = ff_add(ff_div_f(l, T), ff_make(-s_lp_m[i]));
        const ff lq = ff_add(ff_div_f(ff_make(s_ql[i]), T), ff_make(-s_lq_m[i]));
        const float ratio = ff_to_f(ff_div(s_lq_s[i], s_lp_s[i]));
        // outside the truncated target: p(x) = 0, rejected; outside the
        // truncated draft only: q(x) = 0 < p(x), accepted (R2)
        const bool keep_p = !p_cut || s_lbuf[i] >= s_tp[i];
        const bool keep_q = !q_cut || s_ql[i] >= s_tq[i];
        const float thr =
            keep_p ? (keep_q ? accept_threshold(lp, lq, ratio) : INFINITY) : 0.0f;
        s_acc[i] = isfinite(l.hi) ? (s_u[i] < thr ? 1 : 0) : -1;
      }
    } else {
      for (int i = warp; i <= kb; i += kTailWarps) {
        const int a = exact_argmax(P, out0 + i, s_lp_m[i], lane);
        if (lane == 0) s_arg[i] = a;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int err = s_err;
    SeqState st = {};
    st.mode = kModeSkip;
    if (err == 0 && !greedy) {
      int n = kb, mode = kModeP;
      for (int i = 0; i < kb; ++i) {
        if (s_acc[i] < 0) {
          err = SV_ERR_NONFINITE;
          break;
        }
        if (s_acc[i]) {
          if (emit) P.out_tokens[out0 + i] = s_x[i];
        } else {
          n = i;
          mode = point ? kModeResidualPoint : kModeResidual;
          break;
        }
      }
      if (err == 0) {
        if (emit) {
          for (int i = n + 1; i < rows; ++i) P.out_tokens[out0 + i] = -1;
          P.out_n[b] = n;
        }
        st.mode = mode;
        st.n_acc = n;
        st.p_row = static_cast<int>(out0 + n);
        st.p_max = s_lp_m[n];
        st.p_corr = __fdiv_rn(1.0f, ff_to_f(s_lp_s[n]));
        st.p_tau = s_tp[n];
        st.q_tau = -INFINITY;
        if (mode == kModeResidual) {
          st.q_row = b * K + n;
          st.q_max = s_lq_m[n];
          st.q_corr = __fdiv_rn(1.0f, ff_to_f(s_lq_s[n]));
          st.q_tau = s_tq[n];
        } else if (mode == kModeResidualPoint) {
          st.q_row = s_x[n];  // the token whose entry the residual drops
        }
        st.u_final = s_u[K];
      }
    } else if (err == 0) {
      bool ok = true;
      for (int i = 0; i <= kb; ++i) ok = ok && s_arg[i] >= 0;
      if (!ok) {
        err = SV_ERR_NONFINITE;
      } else if (parents) {
        // greedy tree verification: one pass over the nodes (parents come
        // first); row 0 is the root, row 1 + j node j
        s_depth[0] = 0;
        s_match[0] = 1;
        int best = 0;
        for (int j = 0; j < K; ++j) {
          const int pr = s_par[j] + 1;
          s_depth[1 + j] = s_depth[pr] + 1;
          s_match[1 + j] = (s_match[pr] && s_x[j] == s_arg[pr]) ? 1 : 0;
          if (s_match[1 + j] && s_depth[1 + j] > s_depth[best]) best = 1 + j;
        }
        const int n = s_depth[best];
        int r = best;
        for (int i = n - 1; i >= 0; --i) {
          const int node = r - 1;
          P.out_tokens[out0 + i] = s_x[node];
          if (P.out_nodes) P.out_nodes[static_cast<int64_t>(b) * K + i] = node;
          r = s_par[node] + 1;
        }
        P.out_tokens[out0 + n] = s_arg[best];
        for (int i = n + 1; i < rows; ++i) P.out_tokens[out0 + i] = -1;
        if (P.out_nodes)
          for (int i = n; i < K; ++i) P.out_nodes[static_cast<int64_t>(b) * K + i] = -1;
        P.out_n[b] = n;
      } else {
        int n = kb;
        for (int i = 0; i < kb; ++i) {
          if (s_x[i] == s_arg[i]) {
            P.out_tokens[out0 + i] = s_x[i];
          } else {
            P.out_tokens[out0 + i] = s_arg[i];
            n = i;
            break;
          }
        }
        if (n == kb) P.out_tokens[out0 + kb] = s_arg[kb];
        for (int i = n + 1; i < rows; ++i) P.out_tokens[out0 + i] = -1;
        P.out_n[b] = n;
      }
    }
    if (err != 0) {
      st.mode = kModeSkip;
      if (emit) {
        if (err != SV_ERR_TIMEOUT) set_status(P.w.status, err);
        for (int i = 0; i < rows; ++i) P.out_tokens[out0 + i] = -1;
        if (P.out_nodes)
          for (int i = 0; i < K; ++i) P.out_nodes[static_cast<int64_t>(b) * K + i] = -1;
        P.out_n[b] = -1;
      }
    }
    s_fin = kFinNone;
    if (local) {
      *local = st;
    } else {
      P.w.seq[b] = st;
      __threadfence();
      *reinterpret_cast<volatile unsigned *>(&P.w.seq_flag[b]) = P.epoch;
      if (!greedy) {
        __threadfence();
        s_fin = arrive_final(P, b);
      }
    }
  }
  __syncthreads();
  return s_fin;
}

// ---------------------------------------------------------------------------
// Selection (one CTA, the last chunk CTA of sequence b)
// ---------------------------------------------------------------------------
// Warp 0: the total mass S of the chunk masses and the chunk holding
// u * S (a scan of the masses in chunk order), each mass loaded once when
// there are at most 32 chunks.  Leaves S, the chunk, the mass before it and
// the target u * S in shared memory.
__device__ __forceinline__ void locate_chunk(const float2 *mass, int nchunk, float u, int lane,
                                             ff &s_S, ff &s_base, ff &s_target, int &s_chunk,
                                             const ff *held = nullptr) {
  // held: this lane's mass (chunk `lane`), already loaded, when nchunk <= 32
  const bool one = nchunk <= 32;
  const ff m0 = (one && lane < nchunk) ? (held ? *held : ld_ff(&mass[lane])) : ff_make(0.0f);
  ff S = m0;
  if (!one)
    for (int c = lane + 32; c < nchunk; c += 32) S = ff_add(S, ld_ff(&mass[c]));
  if (!one && lane < nchunk) S = ff_add(ld_ff(&mass[lane]), S);
  S = warp_sum_ff(S);
  const ff target = ff_mul_f(S, u);
  ff carry = ff_make(0.0f), base = ff_make(0.0f), base_last = ff_make(0.0f);
  int chunk = -1, last = -1;
  if (S.hi > 0.0f) {
    for (int c0 = 0; c0 < nchunk && chunk < 0; c0 += 32) {
      const int c = c0 + lane;
      const ff m = one ? m0 : (c < nchunk ? ld_ff(&mass[c]) : ff_make(0.0f));
      ff inc = m;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const ff y = ff_shfl_up(inc, o);
        if (lane >= o) inc = ff_add(y, inc);
      }
      const ff incl = ff_add(carry, inc);
      const ff excl = ff_add(incl, ff_neg(m));
      const unsigned hit = __ballot_sync(0xffffffffu, c < nchunk && ff_lt(target, incl));
      const unsigned pos = __ballot_sync(0xffffffffu, c < nchunk && m.hi > 0.0f);
      if (pos) {
        const int lp = 31 - __clz(pos);
        last = c0 + lp;
        base_last = ff_shfl(excl, lp);
      }
      if (hit) {
        const int lh = __ffs(hit) - 1;
        chunk = c0 + lh;
        base = ff_shfl(excl, lh);
      }
      carry = ff_shfl(incl, 31);
    }
  }
  if (lane == 0) {
    if (chunk < 0) {  // rounding pushed the target past the end
      chunk = last;
      base = base_last;
    }
    s_S = S;
    s_chunk = chunk;
    s_base = base;
    s_target = target;
  }
}

// Chunk masses not yet published hold all-ones bits (a NaN pair, which no
// mass can be); every launch leaves them so.  A mass is published, and
// polled, as one 64-bit access, so a reader sees either the sentinel or the
// whole pair.
constexpr unsigned long long kMassUnset = ~0ull;

__device__ __forceinline__ void publish_mass(float2 *slot, ff m) {
  const unsigned long long bits =
      (static_cast<unsigned long long>(__float_as_uint(m.lo)) << 32) | __float_as_uint(m.hi);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(slot), "l"(bits) : "memory");
}

__device__ __forceinline__ unsigned long long peek_mass(const float2 *slot) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(slot) : "memory");
  return v;
}

__device__ __forceinline__ ff mass_of(unsigned long long bits) {
  return ff{__uint_as_float(static_cast<unsigned>(bits)), __uint_as_float(static_cast<unsigned>(bits >> 32))};
}

// Rewinds sequence b's masses to the sentinel (one thread; after everything
// that reads them in this launch).
__device__ __forceinline__ void unset_masses(const TailParams &P, int b) {
  unsigned long long *m = reinterpret_cast<unsigned long long *>(
      P.w.chunk_mass + static_cast<int64_t>(b) * P.dims.nchunk);
  for (int c = 0; c < P.dims.nchunk; ++c) m[c] = kMassUnset;
}

// The inverse CDF inside the chunk that holds the target: a block scan of
// this thread's weights r (the chunk's entries threadIdx.x * 8 .. + 7, sum
// tsum) on top of `base`, the mass before the chunk; thread 0 writes the
// smallest v with target < C_v (or, if rounding left none, the largest v of
// the chunk with positive weight) to *out.
__device__ void scan_chunk(const float (&r)[kChunkPerThread], float tsum, int chunk, ff base,
                           ff target, int32_t *out, ff *s_warp) {
  __shared__ int s_found, s_last;
  if (threadIdx.x == 0) {
    s_found = 0x7fffffff;
    s_last = -1;
  }
  ff run = ff_add(base, block_excl_scan_ff(ff_make(tsum), s_warp));
  const int64_t v0 = static_cast<int64_t>(chunk) * kChunk + threadIdx.x * kChunkPerThread;
  int found = 0x7fffffff, last = -1;
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) {
    run = ff_add(run, ff_make(r[j]));
    if (r[j] > 0.0f) {
      last = static_cast<int>(v0 + j);
      if (found == 0x7fffffff && ff_lt(target, run)) found = static_cast<int>(v0 + j);
    }
  }
  if (found != 0x7fffffff) atomicMin(&s_found, found);
  if (last >= 0) atomicMax(&s_last, last);
  __syncthreads();
  if (threadIdx.x == 0) *out = s_found != 0x7fffffff ? s_found : s_last;
}

// The final draw of sequence b by one CTA.  With masses_ready the chunk
// masses of st's weights are in `mass`; otherwise (or when the residual
// turns out empty: p_j == q_j on the row) the CTA computes the masses of
// p_j itself into `mass` and draws from p_j.
__device__ void select_token(const TailParams &P, int b, SeqState st, float2 *mass,
                             bool masses_ready) {
  __shared__ ff s_warp[kTailWarps];
  __shared__ ff s_S, s_base, s_target;
  __shared__ int s_chunk;
  const int lane = threadIdx.x & 31;
  const int nchunk = P.dims.nchunk;
  bool recompute = !masses_ready;
  if (masses_ready) {
    if (threadIdx.x < 32)
      locate_chunk(mass, nchunk, st.u_final, lane, s_S, s_base, s_target, s_chunk);
    __syncthreads();
    recompute = !(s_S.hi > 0.0f) && (st.mode == kModeResidual || st.mode == kModeResidualPoint);
  }
  if (recompute) {
    // p_j == q_j on this row: draw from p_j instead
    st.mode = kModeP;
    for (int c = 0; c < nchunk; ++c) {
      float r[kChunkPerThread];
      const ff m = block_sum_ff(ff_make(chunk_weights(P, st, c, r)), s_warp);
      if (threadIdx.x == 0) st_ff(&mass[c], m);
    }
    __syncthreads();
    if (threadIdx.x < 32)
      locate_chunk(mass, nchunk, st.u_final, lane, s_S, s_base, s_target, s_chunk);
    __syncthreads();
  }
  const int64_t rows = P.dims.K + 1;
  int32_t *out = P.out_tokens + static_cast<int64_t>(b) * rows + st.n_acc;
  if (!(s_S.hi > 0.0f)) {
    if (threadIdx.x == 0) {
      set_status(P.w.status, SV_ERR_NONFINITE);
      *out = -1;
      P.out_n[b] = -1;
    }
    return;
  }
  const int chunk = s_chunk;
  float r[kChunkPerThread];
  const float tsum = chunk_weights(P, st, chunk, r);
  scan_chunk(r, tsum, chunk, s_base, s_target, out, s_warp);
}

// Bounded wait (one thread) until *cnt >= target, with acquire ordering.
__device__ __forceinline__ bool wait_count(const int *cnt, int target, uint64_t limit_ns) {
  auto load = [cnt]() {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = globaltimer();
  while (load() < target) {
    if (globaltimer() - t0 >= limit_ns) return false;
    __nanosleep(20);
  }
  return true;
}

// Cooperative selection (the whole tail grid resident at once): every chunk
// CTA of sequence b publishes its mass (one 64-bit store over the unset
// sentinel); warp 0 of every CTA polls the sequence's masses, one slot per
// lane, with relaxed loads (a warp's slots share two cache lines) until
// none is unset (bounded), and locates the chunk holding u * S from the
// values it polled; the CTA that computed that chunk scans the weights it
// still holds.  A CTA whose wait ran out reports SV_ERR_TIMEOUT and marks
// the sequence; the last CTA past the selection withdraws a marked
// sequence (outputs -1) and rewinds its counter and masses.
__device__ void coop_select(const TailParams &P, int b, int c, const SeqState &st,
                            const float (&r)[kChunkPerThread], float tsum, ff mass) {
  __shared__ ff s_warp[kTailWarps];
  __shared__ ff s_S, s_base, s_target;
  __shared__ int s_chunk, s_all;
  const int lane = threadIdx.x & 31;
  const int nchunk = P.dims.nchunk;
  float2 *masses = P.w.chunk_mass + static_cast<int64_t>(b) * nchunk;
  const int64_t rows = P.dims.K + 1;
  if (threadIdx.x == 0) publish_mass(&masses[c], mass);
  if (threadIdx.x < 32) {
    bool all = true;
    ff held = ff_make(0.0f);
    for (int c0 = lane; c0 < nchunk && all; c0 += 32) {
      unsigned long long v = peek_mass(&masses[c0]);
      if (v == kMassUnset) {
        const uint64_t t0 = globaltimer();
        while ((v = peek_mass(&masses[c0])) == kMassUnset) {
          if (globaltimer() - t0 >= P.wait_limit_ns) {
            all = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (c0 == lane) held = mass_of(v);
    }
    all = __all_sync(0xffffffffu, all);
    if (all && st.mode != kModeSkip)
      locate_chunk(masses, nchunk, st.u_final, lane, s_S, s_base, s_target, s_chunk,
                   nchunk <= 32 ? &held : nullptr);
    if (lane == 0) s_all = all ? 1 : 0;
  }
  __syncthreads();
  if (s_all && st.mode != kModeSkip) {
    if (!(s_S.hi > 0.0f)) {
      // an empty residual (or no mass at all): the first chunk CTA draws
      // alone, with masses of its own in the second half of chunk_mass
      if (c == 0)
        select_token(P, b, st,
                     P.w.chunk_mass + static_cast<int64_t>(P.dims.B + b) * nchunk, false);
    } else if (s_chunk == c) {
      scan_chunk(r, tsum, c, s_base, s_target, P.out_tokens + b * rows + st.n_acc, s_warp);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!s_all) {
      set_status(P.w.status, SV_ERR_TIMEOUT);
      atomicOr(&P.w.seq_final[b], kPoisoned);
    }
    __threadfence();
    if (atomicAdd(&P.w.chunk_done[b], 1) == nchunk - 1) {
      __threadfence();
      if (*reinterpret_cast<volatile int *>(&P.w.seq_final[b]) & kPoisoned) {
        for (int i = 0; i < rows; ++i) P.out_tokens[static_cast<int64_t>(b) * rows + i] = -1;
        P.out_n[b] = -1;
      }
      unset_masses(P, b);
      P.w.chunk_done[b] = 0;
      P.w.seq_final[b] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// The fused tail kernel
// ---------------------------------------------------------------------------
// Carries out what arrive_final decided (block-wide).  `known` is the
// sequence's published state when the caller already holds it.
__device__ void finalize_sequence(const TailParams &P, int b, int fin,
                                  const SeqState *known = nullptr) {
  if (fin == kFinPoison) {
    if (threadIdx.x == 0) {
      const int rows = P.dims.K + 1;
      for (int i = 0; i < rows; ++i) P.out_tokens[static_cast<int64_t>(b) * rows + i] = -1;
      P.out_n[b] = -1;
      unset_masses(P, b);
    }
  } else if (fin == kFinSelect) {
    SeqState st;
    if (known) {
      st = *known;
    } else {
      const int *src = reinterpret_cast<const int *>(&P.w.seq[b]);
      int *dst = reinterpret_cast<int *>(&st);
#pragma unroll
      for (int i = 0; i < static_cast<int>(sizeof(SeqState) / 4); ++i) dst[i] = __ldcg(&src[i]);
    }
    if (st.mode != kModeSkip)
      select_token(P, b, st, P.w.chunk_mass + static_cast<int64_t>(b) * P.dims.nchunk, true);
    __syncthreads();
    if (threadIdx.x == 0) unset_masses(P, b);
  }
}

// two CTAs per SM (64 registers), so twice as many run at once when a
// round has many rows
__global__ void __launch_bounds__(kTailThreads, 2) tail_kernel(const TailParams P) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ unsigned s_ticket;
  __shared__ float s_wf[kTailWarps];
  __shared__ ff s_wff[kTailWarps];
  __shared__ int s_last;
  const int K = P.dims.K;
  const int R = P.dims.R;
  // fast mode: one decision CTA per sequence; otherwise one CTA per row
  const int nrow = P.fast ? P.dims.B : P.greedy ? R : R + P.dims.RQ;
  if (threadIdx.x == 0) s_ticket = atomicAdd(P.w.ticket, 1u);
  __syncthreads();
  const int t = static_cast<int>(s_ticket);
  if (P.stall && t == 0 && threadIdx.x == 0) {
    // test of the timeout path: a wait for a flag that nothing sets runs
    // out; the run reports it and sequence 0 is withdrawn
    if (!wait_flag(reinterpret_cast<const unsigned *>(P.w.never), 1u, P.wait_limit_ns)) {
      set_status(P.w.status, SV_ERR_TIMEOUT);
      atomicOr(&P.w.seq_final[0], kPoisoned);
      __threadfence();
    }
  }

  if (t < nrow && P.fast) {
    finalize_sequence(P, t, decide<false>(P, t));
  } else if (t < nrow) {
    // ---- row statistics ----
    const bool qrow = t >= R;
    const int b = qrow ? (t - R) / (K > 0 ? K : 1) : t / (K + 1);
    const float2 *part = qrow ? P.w.part_q + static_cast<int64_t>(t - R) * P.dims.nsub
                              : P.w.part_p + static_cast<int64_t>(t) * P.dims.nsub;
    // one pass, 8 loads in flight per thread: running (max, sum) with
    // rescaling whenever the running maximum grows.  A point-mass draft
    // row has no partials: it is published as M = 0, S = 1.
    const bool neutral = qrow && P.q_logits == nullptr;
    // a truncated row's (M, S) were published by the truncation kernel
    const bool given = !P.greedy && (qrow ? P.q_cut : P.p_cut);
    float m = -INFINITY, acc = 0.0f;
    int bad = 0;
    for (int s0 = threadIdx.x; s0 < P.dims.nsub && !neutral && !given;
         s0 += kTailThreads * 8) {
      float2 pm[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int s = s0 + j * kTailThreads;
        pm[j] = s < P.dims.nsub ? __ldcg(&part[s]) : make_float2(-INFINITY, 0.0f);
      }
      float mn = m;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        bad |= (isnan(pm[j].x) || pm[j].x == INFINITY) ? 1 : 0;
        mn = fmaxf(mn, pm[j].x);
      }
      if (!P.greedy && mn > -INFINITY) {
        acc = m > -INFINITY ? acc * expf(m - mn) : 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (pm[j].x > -INFINITY) acc += pm[j].y * expf(pm[j].x - mn);
      }
      m = mn;
    }
    bad = __syncthreads_or(bad);
    float M = block_max_f(m, s_wf);
    ff S = ff_make(0.0f);
    if (!P.greedy && !bad) {
      const float mine = m > -INFINITY ? acc * expf(m - M) : 0.0f;
      S = block_sum_ff(ff_make(mine), s_wff);
    }
    if (neutral) {
      M = 0.0f;
      S = ff_make(1.0f);
    }
    if (given) {
      M = __ldcg(&P.w.row_m[t]);
      S = ld_ff(&P.w.row_s[t]);
    }
    if (bad) M = NAN;
    if (P.greedy && !bad) {
      // list the subtiles that may hold the argmax (see exact_argmax)
      __shared__ int s_nc;
      __shared__ int s_cand[kMaxCand];
      if (threadIdx.x == 0) s_nc = 0;
      __syncthreads();
      const float thr = M - greedy_eps(M);
      for (int s0 = threadIdx.x; s0 < P.dims.nsub; s0 += kTailThreads * 8) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int s = s0 + j * kTailThreads;
          x[j] = s < P.dims.nsub ? __ldcg(&part[s].x) : -INFINITY;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (x[j] >= thr) {
            const int k = atomicAdd(&s_nc, 1);
            if (k < kMaxCand) s_cand[k] = s0 + j * kTailThreads;
          }
      }
      __syncthreads();
      int *cand = P.w.cand + static_cast<int64_t>(t) * (1 + kMaxCand);
      const int nc = s_nc;
      for (int k = threadIdx.x; k < nc && k < kMaxCand; k += kTailThreads) cand[1 + k] = s_cand[k];
      if (threadIdx.x == 0) cand[0] = nc;
    }
    if (qrow && !P.greedy && !P.draft_logits_ready) {
      // the exact logit of this position's draft token, split over the
      // CTA's warps (fixed order), so the decider only reads it (the
      // tensor-core contraction computes these itself)
      const int i = (t - R) - b * K;
      const int x = P.draft[static_cast<int64_t>(b) * K + i];
      if (x >= 0 && static_cast<int64_t>(x) < P.dims.V) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const ff part = dot_warp(P, static_cast<int64_t>(b) * (K + 1) + i, x, lane, warp,
                                 kTailWarps);
        if (lane == 0) s_wff[warp] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
          ff l = s_wff[0];
          for (int w2 = 1; w2 < kTailWarps; ++w2) l = ff_add(l, s_wff[w2]);
          st_ff(&P.w.draft_logit[t - R], l);
        }
      }
    }
    if (threadIdx.x == 0) {
      P.w.row_m[t] = M;
      st_ff(&P.w.row_s[t], S);
      __threadfence();
      const int need = P.greedy ? K + 1 : 2 * K + 1;
      s_last = atomicAdd(&P.w.row_count[b], 1) == need - 1;
      if (s_last) {
        P.w.row_count[b] = 0;
        __threadfence();
      }
    }
    __syncthreads();
    if (s_last) finalize_sequence(P, b, decide<false>(P, b));
  } else {
    // ---- residual chunk ----
    const int idx = t - nrow;
    const int b = idx / P.dims.nchunk, c = idx % P.dims.nchunk;
    __shared__ int s_seen, s_fin;
    if (threadIdx.x == 0) {
      if (!wait_flag(&P.w.seq_flag[b], P.epoch, P.wait_limit_ns))
        set_status(P.w.status, SV_ERR_TIMEOUT);
      // one read of the flag decides for the whole CTA
      s_seen = *reinterpret_cast<const volatile unsigned *>(&P.w.seq_flag[b]) == P.epoch;
      __threadfence();
    }
    __syncthreads();
    SeqState st;
    {
      const int *src = reinterpret_cast<const int *>(&P.w.seq[b]);
      int *dst = reinterpret_cast<int *>(&st);
#pragma unroll
      for (int i = 0; i < static_cast<int>(sizeof(SeqState) / 4); ++i) dst[i] = __ldcg(&src[i]);
    }
    if (!s_seen) st.mode = kModeSkip;
    float m = 0.0f;
    if (st.mode != kModeSkip) {
      float r[kChunkPerThread];
      m = chunk_weights(P, st, c, r);
    }
    const ff mass = block_sum_ff(ff_make(m), s_wff);
    if (threadIdx.x == 0) {
      st_ff(&P.w.chunk_mass[static_cast<int64_t>(b) * P.dims.nchunk + c], mass);
      if (!s_seen) atomicOr(&P.w.seq_final[b], kPoisoned);
      __threadfence();
      s_fin = kFinNone;
      if (atomicAdd(&P.w.chunk_count[b], 1) == P.dims.nchunk - 1) {
        P.w.chunk_count[b] = 0;
        __threadfence();
        s_fin = arrive_final(P, b);
      }
    }
    __syncthreads();
    // a chunk CTA that saw the decision holds its state; one that timed out
    // set the poison bit, so the selection never runs on its copy
    finalize_sequence(P, b, s_fin, &st);
  }

  // the last CTA to finish rewinds the ticket counter for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(P.w.finished, 1u) == gridDim.x - 1) {
      *P.w.ticket = 0;
      *P.w.finished = 0;
    }
  }
}

// 1-D bulk copy (TMA) of `bytes` from global to this CTA's shared memory,
// completing on the mbarrier; both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// The weights of chunk c from the rows staged in shared memory (stage row
// j <= K: target row j of the sequence; K+1+j: draft row j); the same
// arithmetic as chunk_weights.
__device__ __forceinline__ float staged_weights(const TailParams &P, const SeqState &st, int b,
                                                int c, const float *stage,
                                                float (&r)[kChunkPerThread]) {
  const int K = P.dims.K;
  const int64_t V = P.dims.V;
  const int i0 = threadIdx.x * kChunkPerThread;
  const int64_t v0 = static_cast<int64_t>(c) * kChunk + i0;
  const float *ls = stage + static_cast<int64_t>(st.p_row - b * (K + 1)) * kChunk + i0;
  const bool resid = st.mode == kModeResidual;
  const float *qs =
      resid ? stage + static_cast<int64_t>(K + 1 + st.q_row - b * K) * kChunk + i0 : nullptr;
  float l[kChunkPerThread], q[kChunkPerThread];
#pragma unroll
  for (int j = 0; j < kChunkPerThread; j += 4) {
    const bool in = v0 + j < V;  // V % 4 == 0: a group of four is all in or all out
    const float4 a = in ? *reinterpret_cast<const float4 *>(ls + j) : make_float4(0, 0, 0, 0);
    const float4 e = (in && resid) ? *reinterpret_cast<const float4 *>(qs + j) : make_float4(0, 0, 0, 0);
    l[j] = a.x; l[j + 1] = a.y; l[j + 2] = a.z; l[j + 3] = a.w;
    q[j] = e.x; q[j + 1] = e.y; q[j + 2] = e.z; q[j + 3] = e.w;
  }
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) {
    r[j] = v0 + j < V ? draw_weight(st, v0 + j, l[j], q[j], P.inv_t) : 0.0f;
    sum = __fadd_rn(sum, r[j]);
  }
  return sum;
}

// The cooperative tail, when the whole grid is resident at once: CTA
// b * nchunk + c is chunk c of sequence b.  With P.stage_rows it first
// copies its chunk of every row the final draw may use (the K+1 target
// rows, then the K draft rows) into shared memory, one bulk copy per row,
// which lands while it takes the sequence's decision itself (as every chunk
// CTA of the sequence does, from the same inputs; the first writes the
// accepted prefix).  Then it computes its chunk's mass and runs the
// cooperative selection.  No CTA waits for another except in that
// selection.
__global__ void __launch_bounds__(kTailThreads, 2) tail_coop_kernel(const TailParams P) {
  extern __shared__ __align__(1024) unsigned char stage_raw[];
  __shared__ ff s_wff[kTailWarps];
  __shared__ SeqState s_st;
  __shared__ __align__(8) uint64_t s_stage_bar;
  __shared__ int s_staged;
  pdl_wait();
  pdl_launch_dependents();
  const int nchunk = P.dims.nchunk;
  const int b = static_cast<int>(blockIdx.x) / nchunk, c = static_cast<int>(blockIdx.x) % nchunk;
  const uint32_t bar = smem_u32(&s_stage_bar);
  if (P.stage_rows && threadIdx.x == 0) {
    const int K = P.dims.K;
    const int64_t V = P.dims.V;
    const int64_t v0 = static_cast<int64_t>(c) * kChunk;
    const uint32_t bytes = static_cast<uint32_t>((V - v0 < kChunk ? V - v0 : kChunk) * 4);
    mbar_init(bar, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(P.stage_rows));
    const uint32_t dst0 = smem_u32(stage_raw);
    for (int j = 0; j < P.stage_rows; ++j) {
      const float *row = j <= K ? P.w.logits + (static_cast<int64_t>(b) * (K + 1) + j) * V
                                : P.q_logits + (static_cast<int64_t>(b) * K + (j - K - 1)) * V;
      bulk_load(dst0 + static_cast<uint32_t>(j) * kChunk * 4, row + v0, bytes, bar);
    }
  }
  if (P.stall && blockIdx.x == 0 && threadIdx.x == 0) {
    // test of the timeout path (see tail_kernel)
    if (!wait_flag(reinterpret_cast<const unsigned *>(P.w.never), 1u, P.wait_limit_ns)) {
      set_status(P.w.status, SV_ERR_TIMEOUT);
      atomicOr(&P.w.seq_final[0], kPoisoned);
      __threadfence();
    }
  }
  decide<true>(P, b, &s_st, c == 0);
  if (P.stage_rows && threadIdx.x == 0) {
    // the copies must have landed before the rows are read, and before the
    // CTA may exit
    const int never = 0;
    s_staged = mbar_wait(bar, 0u, P.wait_limit_ns, &never) ? 1 : 0;
  }
  __syncthreads();
  SeqState st = s_st;
  if (P.stage_rows && !s_staged) {
    if (threadIdx.x == 0) {
      set_status(P.w.status, SV_ERR_TIMEOUT);
      atomicOr(&P.w.seq_final[b], kPoisoned);
    }
    st.mode = kModeSkip;
  }
  float r[kChunkPerThread];
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) r[j] = 0.0f;
  float m = 0.0f;
  if (st.mode != kModeSkip)
    m = P.stage_rows ? staged_weights(P, st, b, c, reinterpret_cast<const float *>(stage_raw), r)
                     : chunk_weights(P, st, c, r);
  const ff mass = block_sum_ff(ff_make(m), s_wff);
  coop_select(P, b, c, st, r, m, mass);
}

int tail_resident_ctas(int num_sms, int stage_bytes) {
  if (stage_bytes > 0 &&
      cudaFuncSetAttribute(tail_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           stage_bytes) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tail_coop_kernel, kTailThreads,
                                                    stage_bytes) != cudaSuccess)
    return 0;
  return per_sm * num_sms;
}

int tail_stage_bytes(const Dims &d, bool with_q) {
  const int rows = d.K + 1 + (with_q ? d.K : 0);
  const int64_t bytes = static_cast<int64_t>(rows) * kChunk * 4;
  return (d.V % 4 == 0 && bytes <= kStageMaxBytes) ? static_cast<int>(bytes) : 0;
}

cudaError_t launch_tail(const TailParams &P, cudaStream_t stream) {
  void *args[] = {const_cast<TailParams *>(&P)};
  if (P.coop) {
    const size_t smem = static_cast<size_t>(P.stage_rows) * kChunk * 4;
    // the opt-in above 48 KB is per device; idempotent and cheap
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(
          tail_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_pdl(reinterpret_cast<const void *>(&tail_coop_kernel),
                      dim3(P.dims.B * P.dims.nchunk), dim3(kTailThreads), smem, stream, args);
  }
  const int nrow = P.fast ? P.dims.B : P.greedy ? P.dims.R : P.dims.R + P.dims.RQ;
  const int nchunk_ctas = P.greedy ? 0 : P.dims.B * P.dims.nchunk;
  return launch_pdl(reinterpret_cast<const void *>(&tail_kernel), dim3(nrow + nchunk_ctas),
                    dim3(kTailThreads), 0, stream, args);
}

// ---------------------------------------------------------------------------
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, void **args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv
