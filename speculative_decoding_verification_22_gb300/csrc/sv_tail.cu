// sv_tail.cu -- kernels (b) and (c) of the verify step.
//
// (b1) decide_kernel, one CTA per sequence: combines the per-subtile
//      softmax partials into fp64 log-sum-exp normalisers of logits / T and
//      q_logits / T, recomputes the K draft-token logits with a compensated
//      dot product, and walks the draft left to right: x_{i+1} survives iff
//      u_i < p_{i+1}(x) / q_{i+1}(x) ("Speculative Decoding: Two Models, One
//      Voice", "The idea" step 3; "Speculative Decoding" (library wiki),
//      "One speculation round").  It writes the accepted prefix and hands
//      the row of the final draw to the next passes.  At T == 0 it performs
//      greedy verification instead ("Speculative Decoding: Guess Several
//      Tokens, Check Them in One Pass", Step 2) with an exact re-ranking of
//      the near-maximal logits, and writes every output itself.
// (b2) residual_kernel, vocab-parallel: per 2048-entry chunk, the mass of
//      max(0, p_j - q_j) (or of p_{K+1} for the bonus) with 128-bit loads.
// (c)  select_kernel, one CTA per sequence: locates u * S in the chunk
//      prefix sums, rescans that chunk and emits the smallest v with
//      u * S < C_v (inverse CDF in token-id order); an empty residual falls
//      back to p_j ("What Actually Happens During Speculative Decoding in
//      LLMs", speculative_sample_step).
#include <cuda_bf16.h>

#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {

// ---------------------------------------------------------------------------
// Helpers
// ---------------------------------------------------------------------------

// Dot product of hidden row `hrow` with W row `wrow` by one warp.  Products
// are formed without rounding error (bf16 x bf16 is exact in fp32; fp32 x
// fp32 via an FMA error term) and summed with TwoSum error tracking, so the
// result is accurate to a few fp64 ulps of the logit.  Every lane returns
// the same value.
__device__ double dot_warp(const TailParams &P, int64_t hrow, int64_t wrow, int lane) {
  const int64_t d = P.dims.d;
  float s = 0.0f, c = 0.0f;
  if (P.dtype == SV_BF16) {
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(P.H) + hrow * d;
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(P.W) + wrow * d;
#pragma unroll 8
    for (int64_t k = lane; k < d; k += 32) {
      const float p = __fmul_rn(__bfloat162float(h[k]), __bfloat162float(w[k]));
      float t, e;
      two_sum(s, p, t, e);
      s = t;
      c += e;
    }
  } else {
    const float *h = static_cast<const float *>(P.H) + hrow * d;
    const float *w = static_cast<const float *>(P.W) + wrow * d;
#pragma unroll 8
    for (int64_t k = lane; k < d; k += 32) {
      const float a = h[k], b = w[k];
      const float p = __fmul_rn(a, b);
      const float pe = fmaf(a, b, -p);
      float t, e;
      two_sum(s, p, t, e);
      s = t;
      c += e + pe;
    }
  }
  return warp_sum_d(static_cast<double>(s) + static_cast<double>(c));
}

// Greedy argmax of target row r with ties to the smallest id.  Only entries
// whose fp32 logit is within eps of the row maximum can be the argmax (the
// fp32 logits are far more accurate than eps); those are re-ranked with the
// exact dot product in increasing id order.  Returns -1 if the row is not
// finite.
__device__ int exact_argmax(const TailParams &P, int64_t r, int lane) {
  const int nsub = P.dims.nsub;
  const int64_t V = P.dims.V;
  const float2 *part = P.w.part_p + r * nsub;
  float M = -INFINITY;
  for (int s = lane; s < nsub; s += 32) M = fmaxf(M, part[s].x);
  M = warp_max(M);
  if (!isfinite(M)) return -1;
  const float thr = M - (1e-3f + 1e-5f * fabsf(M));
  double best = -INFINITY;
  int best_v = -1;
  for (int s0 = 0; s0 < nsub; s0 += 32) {
    const int s = s0 + lane;
    unsigned cand = __ballot_sync(0xffffffffu, s < nsub && part[s].x >= thr);
    while (cand) {
      const int sc = s0 + __ffs(cand) - 1;
      cand &= cand - 1;
      const int64_t v = static_cast<int64_t>(sc) * kSub + lane;
      unsigned hit = __ballot_sync(0xffffffffu, v < V && P.w.logits[r * V + v] >= thr);
      while (hit) {
        const int64_t vv = static_cast<int64_t>(sc) * kSub + __ffs(hit) - 1;
        hit &= hit - 1;
        const double e = dot_warp(P, r, vv, lane);
        if (e > best) {
          best = e;
          best_v = static_cast<int>(vv);
        }
      }
    }
  }
  return best_v;
}

__device__ __forceinline__ double block_sum_d(double x, double *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  x = warp_sum_d(x);
  __syncthreads();
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  double t = 0.0;
  if (warp == 0) {
    t = lane < (blockDim.x >> 5) ? s_warp[lane] : 0.0;
    t = warp_sum_d(t);
    if (lane == 0) s_warp[0] = t;
  }
  __syncthreads();
  return s_warp[0];
}

// Exclusive prefix sum over the block (fixed order).
__device__ __forceinline__ double block_excl_scan_d(double x, double *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    double t = lane < (blockDim.x >> 5) ? s_warp[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < (blockDim.x >> 5)) s_warp[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const double before = warp > 0 ? s_warp[warp - 1] : 0.0;
  return before + inc - x;
}

// Weight of vocabulary entry v in the final draw: max(0, p - q) for a
// residual, p for a bonus.  p(v) = exp(l / T - LSE) is evaluated as
// exp(l * inv_t - M) * exp(M - LSE) with M the row maximum, so the fp32
// argument stays small near the mass; the explicit _rn operations keep the
// value bit-identical wherever it is recomputed.
__device__ __forceinline__ float draw_weight(const SeqState &st, float l, float ql,
                                             float inv_t) {
  const float p = __fmul_rn(expf(fmaf(l, inv_t, -st.p_max)), st.p_corr);
  if (st.mode != kModeResidual) return p;
  const float q = __fmul_rn(expf(fmaf(ql, inv_t, -st.q_max)), st.q_corr);
  return fmaxf(__fsub_rn(p, q), 0.0f);
}

// The 8 consecutive weights of this thread in chunk `chunk`, and their sum.
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
    const float4 a = l4[0], b = l4[1];
    l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
    l[4] = b.x; l[5] = b.y; l[6] = b.z; l[7] = b.w;
    if (resid) {
      const float4 *q4 = reinterpret_cast<const float4 *>(qrow + v0);
      const float4 c = q4[0], e = q4[1];
      q[0] = c.x; q[1] = c.y; q[2] = c.z; q[3] = c.w;
      q[4] = e.x; q[5] = e.y; q[6] = e.z; q[7] = e.w;
    } else {
#pragma unroll
      for (int j = 0; j < kChunkPerThread; ++j) q[j] = 0.0f;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kChunkPerThread; ++j) {
      const bool in = v0 + j < V;
      l[j] = in ? lrow[v0 + j] : 0.0f;
      q[j] = (in && resid) ? qrow[v0 + j] : 0.0f;
    }
  }
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) {
    r[j] = v0 + j < V ? draw_weight(st, l[j], q[j], P.inv_t) : 0.0f;
    sum += r[j];
  }
  return sum;
}

// ---------------------------------------------------------------------------
// (b1) decision pass
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTailThreads) decide_kernel(const TailParams P) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int K = P.dims.K, rows = K + 1;
  const int64_t V = P.dims.V;
  const int nsub = P.dims.nsub;
  const int64_t out0 = static_cast<int64_t>(b) * rows;
  __shared__ double s_lse[2 * SV_MAX_K + 1];
  __shared__ float s_max[2 * SV_MAX_K + 1];
  __shared__ double s_lx[SV_MAX_K];
  __shared__ int s_arg[SV_MAX_K + 1];
  __shared__ int s_err;

  if (threadIdx.x == 0) {
    // a contraction that gave up in this run leaves the partials undefined
    s_err = *reinterpret_cast<volatile unsigned *>(P.w.abort_epoch) == P.epoch ? SV_ERR_TIMEOUT
                                                                               : 0;
  }
  __syncthreads();
  if (s_err == SV_ERR_TIMEOUT && b == 0) {
    // the aborted contraction may have left split-tile counters half-used
    for (int i = threadIdx.x; i < P.split_cnt_n; i += blockDim.x) P.w.split_cnt[i] = 0;
  }
  if (threadIdx.x < K) {
    const int x = P.draft[static_cast<int64_t>(b) * K + threadIdx.x];
    if (x < 0 || static_cast<int64_t>(x) >= V) atomicCAS(&s_err, 0, SV_ERR_TOKEN);
  }
  __syncthreads();

  if (s_err == 0) {
    if (!P.greedy) {
      const int nrow = 2 * K + 1;
      for (int r = warp; r < nrow; r += nwarps) {
        const float2 *part =
            r < rows ? P.w.part_p + (out0 + r) * nsub
                     : P.w.part_q + (static_cast<int64_t>(b) * K + (r - rows)) * nsub;
        float M = -INFINITY;
        for (int s = lane; s < nsub; s += 32) M = fmaxf(M, part[s].x);
        M = warp_max(M);
        double S = 0.0;
        for (int s = lane; s < nsub; s += 32) {
          const float2 pm = part[s];
          S += static_cast<double>(pm.y * expf(pm.x - M));
        }
        S = warp_sum_d(S);
        if (lane == 0) {
          s_max[r] = M;
          s_lse[r] = static_cast<double>(M) + log(S);
          const int64_t dst = r < rows ? out0 + r
                                       : static_cast<int64_t>(P.dims.R) +
                                             static_cast<int64_t>(b) * K + (r - rows);
          P.w.lse[dst] = s_lse[r];
        }
      }
      for (int i = warp; i < K; i += nwarps) {
        const int x = P.draft[static_cast<int64_t>(b) * K + i];
        const double l = dot_warp(P, out0 + i, x, lane);
        if (lane == 0) s_lx[i] = l;
      }
    } else {
      for (int i = warp; i < rows; i += nwarps) {
        const int a = exact_argmax(P, out0 + i, lane);
        if (lane == 0) s_arg[i] = a;
      }
    }
  }
  __syncthreads();

  if (threadIdx.x != 0) return;
  int err = s_err;
  SeqState st = {};
  st.mode = kModeSkip;
  if (err == 0 && !P.greedy) {
    bool finite = true;
    for (int r = 0; r < 2 * K + 1; ++r) finite = finite && isfinite(s_lse[r]);
    for (int i = 0; i < K; ++i) finite = finite && isfinite(s_lx[i]);
    if (!finite) {
      err = SV_ERR_NONFINITE;
    } else {
      int n = K, mode = kModeP;
      for (int i = 0; i < K; ++i) {
        const int x = P.draft[static_cast<int64_t>(b) * K + i];
        const double p = exp(s_lx[i] / P.T - s_lse[i]);
        const double ql = static_cast<double>(
            P.q_logits[(static_cast<int64_t>(b) * K + i) * V + x]);
        const double q = exp(ql / P.T - s_lse[rows + i]);
        const double u = static_cast<double>(P.u[out0 + i]);
        const bool accept = q > 0.0 ? (u < p / q) : (p > 0.0);
        if (accept) {
          P.out_tokens[out0 + i] = x;
        } else {
          n = i;
          mode = kModeResidual;
          break;
        }
      }
      for (int i = n + 1; i < rows; ++i) P.out_tokens[out0 + i] = -1;
      P.out_n[b] = n;
      st.mode = mode;
      st.n_acc = n;
      st.p_row = static_cast<int>(out0 + n);
      st.p_max = s_max[n];
      st.p_corr = static_cast<float>(exp(static_cast<double>(s_max[n]) - s_lse[n]));
      if (mode == kModeResidual) {
        st.q_row = b * K + n;
        st.q_max = s_max[rows + n];
        st.q_corr = static_cast<float>(exp(static_cast<double>(s_max[rows + n]) - s_lse[rows + n]));
      }
      st.u_final = P.u[out0 + K];
    }
  } else if (err == 0) {
    bool ok = true;
    for (int i = 0; i < rows; ++i) ok = ok && s_arg[i] >= 0;
    if (!ok) {
      err = SV_ERR_NONFINITE;
    } else {
      int n = K;
      for (int i = 0; i < K; ++i) {
        const int x = P.draft[static_cast<int64_t>(b) * K + i];
        if (x == s_arg[i]) {
          P.out_tokens[out0 + i] = x;
        } else {
          P.out_tokens[out0 + i] = s_arg[i];
          n = i;
          break;
        }
      }
      if (n == K) P.out_tokens[out0 + K] = s_arg[K];
      for (int i = n + 1; i < rows; ++i) P.out_tokens[out0 + i] = -1;
      P.out_n[b] = n;
    }
  }
  if (err != 0) {
    if (err != SV_ERR_TIMEOUT) set_status(P.w.status, err);
    for (int i = 0; i < rows; ++i) P.out_tokens[out0 + i] = -1;
    P.out_n[b] = -1;
  }
  P.w.seq[b] = st;
}

// ---------------------------------------------------------------------------
// (b2) residual masses
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTailThreads) residual_kernel(const TailParams P) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ double s_warp[kTailThreads / 32];
  const int c = blockIdx.x, b = blockIdx.y;
  const SeqState st = P.w.seq[b];
  double t = 0.0;
  if (st.mode != kModeSkip) {
    float r[kChunkPerThread];
    t = static_cast<double>(chunk_weights(P, st, c, r));
  }
  const double m = block_sum_d(t, s_warp);
  if (threadIdx.x == 0) P.w.chunk_mass[static_cast<int64_t>(b) * P.dims.nchunk + c] = m;
}

// ---------------------------------------------------------------------------
// (c) selection
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTailThreads) select_kernel(const TailParams P) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ double s_warp[kTailThreads / 32];
  __shared__ double s_total, s_base, s_target;
  __shared__ int s_chunk;
  __shared__ int s_found, s_last;
  const int b = blockIdx.x;
  SeqState st = P.w.seq[b];
  if (st.mode == kModeSkip) return;
  const int nchunk = P.dims.nchunk;
  double *mass = P.w.chunk_mass + static_cast<int64_t>(b) * nchunk;

  if (threadIdx.x == 0) {
    double S = 0.0;
    for (int c = 0; c < nchunk; ++c) S += mass[c];
    s_total = S;
  }
  __syncthreads();
  if (!(s_total > 0.0) && st.mode == kModeResidual) {
    // p_j == q_j on this row: draw from p_j instead
    st.mode = kModeP;
    for (int c = 0; c < nchunk; ++c) {
      float r[kChunkPerThread];
      const double m = block_sum_d(static_cast<double>(chunk_weights(P, st, c, r)), s_warp);
      if (threadIdx.x == 0) mass[c] = m;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      double S = 0.0;
      for (int c = 0; c < nchunk; ++c) S += mass[c];
      s_total = S;
    }
    __syncthreads();
  }
  const int64_t rows = P.dims.K + 1;
  int32_t *out = P.out_tokens + static_cast<int64_t>(b) * rows + st.n_acc;
  if (!(s_total > 0.0)) {
    if (threadIdx.x == 0) {
      set_status(P.w.status, SV_ERR_NONFINITE);
      *out = -1;
      P.out_n[b] = -1;
    }
    return;
  }
  if (threadIdx.x == 0) {
    const double target = static_cast<double>(st.u_final) * s_total;
    double acc = 0.0;
    int chunk = -1, last = -1;
    double acc_last = 0.0;
    for (int c = 0; c < nchunk; ++c) {
      const double m = mass[c];
      if (m > 0.0) {
        last = c;
        acc_last = acc;
      }
      if (target < acc + m) {
        chunk = c;
        break;
      }
      acc += m;
    }
    if (chunk < 0) {  // rounding pushed the target past the end
      chunk = last;
      acc = acc_last;
    }
    s_chunk = chunk;
    s_base = acc;
    s_target = target;
    s_found = 0x7fffffff;
    s_last = -1;
  }
  __syncthreads();
  const int chunk = s_chunk;
  float r[kChunkPerThread];
  const float tsum = chunk_weights(P, st, chunk, r);
  double run = s_base + block_excl_scan_d(static_cast<double>(tsum), s_warp);
  const int64_t v0 = static_cast<int64_t>(chunk) * kChunk + threadIdx.x * kChunkPerThread;
  int found = 0x7fffffff, last = -1;
#pragma unroll
  for (int j = 0; j < kChunkPerThread; ++j) {
    run += static_cast<double>(r[j]);
    if (r[j] > 0.0f) {
      last = static_cast<int>(v0 + j);
      if (found == 0x7fffffff && s_target < run) found = static_cast<int>(v0 + j);
    }
  }
  if (found != 0x7fffffff) atomicMin(&s_found, found);
  if (last >= 0) atomicMax(&s_last, last);
  __syncthreads();
  if (threadIdx.x == 0) *out = s_found != 0x7fffffff ? s_found : s_last;
}

// ---------------------------------------------------------------------------
// Launchers
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

cudaError_t launch_decide(const TailParams &P, cudaStream_t stream) {
  void *args[] = {const_cast<TailParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&decide_kernel), dim3(P.dims.B),
                    dim3(kTailThreads), 0, stream, args);
}

cudaError_t launch_residual(const TailParams &P, cudaStream_t stream) {
  void *args[] = {const_cast<TailParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&residual_kernel),
                    dim3(P.dims.nchunk, P.dims.B), dim3(kTailThreads), 0, stream, args);
}

cudaError_t launch_select(const TailParams &P, cudaStream_t stream) {
  void *args[] = {const_cast<TailParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&select_kernel), dim3(P.dims.B),
                    dim3(kTailThreads), 0, stream, args);
}

}  // namespace sv
