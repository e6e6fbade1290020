// sv_trunc.cu -- truncated sampling: the cut of every truncated row.
//
// "Speculative Decoding: Two Models, One Voice" (three remarks) and
// "Speculative Decoding: The Algebra and the Proof" ("Where it breaks"):
// the rule stays exact when p and q are the distributions after
// temperature, top-k and top-p.  Both cuts are by value (ties kept): top-k
// keeps every logit at or above the k-th largest, top-p (applied to the
// top-k distribution) every logit at or above the one at which the
// cumulative mass, in descending order, reaches top_p.
//
// One CTA per truncated row.  Logits are mapped to order-preserving 32-bit
// keys; a cut is found by a three-pass radix select (11, 11 and 10 bits from
// the top), each pass one read of the row from L2 building a 2048-bin
// histogram in shared memory: counts for top-k, masses exp(x / T - M) for
// top-p (restricted to the top-k set; the first top-p pass also sums that
// set's mass, the base of the top_p fraction).  Masses are accumulated in
// 64-bit fixed point (2^-40 units; every mass is at most ~1 since M is the
// row maximum), so the sums are exact integers, independent of the order
// of the atomics, and the cut is reproducible.  The crossing bin is the
// highest bin whose suffix sum reaches what remains of the target.  A last
// pass sums the kept mass S in a fixed order; M comes from the
// contraction's per-subtile partials.  The tail reads (M, S, cut) instead
// of reducing the partials.
#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {
namespace {

constexpr int kTruncThreads = kTailThreads;  // the block helpers assume it
constexpr int kBins = 2048;                  // 11-bit digits
constexpr float kMassScale = 1099511627776.0f;  // 2^40: fixed-point unit of a mass

__device__ __forceinline__ unsigned long long fixed_mass(float w) {
  return __float2ull_rn(w * kMassScale);
}

__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ int digit_shift(int pass) { return pass == 0 ? 21 : pass == 1 ? 10 : 0; }
__device__ __forceinline__ uint32_t digit_mask(int pass) { return pass == 2 ? 0x3ffu : 0x7ffu; }

// Applies f(value) to every entry of a row (16-byte loads where aligned).
template <typename F>
__device__ __forceinline__ void for_each_entry(const float *row, int64_t V, F f) {
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    for (int64_t i = threadIdx.x; i < V / 4; i += kTruncThreads) {
      const float4 a = __ldcg(&r4[i]);
      f(a.x);
      f(a.y);
      f(a.z);
      f(a.w);
    }
  } else {
    for (int64_t i = threadIdx.x; i < V; i += kTruncThreads) f(__ldcg(&row[i]));
  }
}

// Inclusive suffix sum over the block's threads (thread t: threads t..last).
template <typename T>
__device__ __forceinline__ T block_suffix_incl(T x, T *s_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  __syncthreads();
  if (lane == 0) s_warp[warp] = x;
  __syncthreads();
  T later = T(0);
  for (int w = kTailWarps - 1; w > warp; --w) later += s_warp[w];
  return x + later;
}

// The highest bin c of hist[0..nb) whose suffix sum (bins c..nb-1) reaches
// r; *above receives the suffix sum of the bins above c.  Where rounding
// leaves every suffix short of r, the lowest non-empty bin is taken.
// Thread t owns bins [t * per, (t + 1) * per).  Block-wide.
template <typename T>
__device__ void find_cut_bin(const T *hist, const int *cnt, int nb, T r, int *s_bin, T *s_above,
                             T *s_warp, T *s_incl, int *s_owner) {
  const int per = nb / kTruncThreads;
  const int b0 = threadIdx.x * per;
  T mine = T(0);
  bool nonempty = false;
  for (int j = 0; j < per; ++j) {
    mine += hist[b0 + j];
    nonempty = nonempty || cnt[b0 + j] > 0;
  }
  if (threadIdx.x == 0) *s_owner = -1;
  const T incl = block_suffix_incl(mine, s_warp);
  s_incl[threadIdx.x] = incl;
  __syncthreads();
  if (incl >= r) atomicMax(s_owner, static_cast<int>(threadIdx.x));
  __syncthreads();
  if (*s_owner < 0) {
    // nothing reaches r: the owner of the lowest non-empty bin
    if (threadIdx.x == 0) *s_owner = kTruncThreads;
    __syncthreads();
    if (nonempty) atomicMin(s_owner, static_cast<int>(threadIdx.x));
    __syncthreads();
    if (*s_owner == kTruncThreads) {  // empty histogram (not reached for valid rows)
      if (threadIdx.x == 0) {
        *s_bin = 0;
        *s_above = T(0);
      }
      __syncthreads();
      return;
    }
  }
  if (static_cast<int>(threadIdx.x) == *s_owner) {
    T acc = threadIdx.x + 1 < kTruncThreads ? s_incl[threadIdx.x + 1] : T(0);
    int c = -1, low = -1;
    T above = acc, above_low = acc;
    for (int j = per - 1; j >= 0; --j) {
      const T next = acc + hist[b0 + j];
      if (cnt[b0 + j] > 0) {
        low = b0 + j;
        above_low = acc;
      }
      if (next >= r && cnt[b0 + j] > 0) {
        c = b0 + j;
        above = acc;
        break;
      }
      acc = next;
    }
    if (c < 0) {
      c = low;
      above = above_low;
    }
    *s_bin = c < 0 ? 0 : c;
    *s_above = above;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTruncThreads) trunc_kernel(const TruncParams P) {
  pdl_wait();
  pdl_launch_dependents();
  using u64 = unsigned long long;
  __shared__ int s_cnt[kBins];
  __shared__ u64 s_mass[kBins];
  __shared__ int s_warp_i[kTailWarps];
  __shared__ u64 s_warp_u[kTailWarps];
  __shared__ float s_warp_f[kTailWarps];
  __shared__ ff s_wff[kTailWarps];
  __shared__ int s_incl_i[kTruncThreads];
  __shared__ u64 s_incl_u[kTruncThreads];
  __shared__ int s_owner, s_bin, s_above_i;
  __shared__ u64 s_above_u;

  const int R = P.dims.R;
  const int64_t V = P.dims.V;
  const int n_target = P.p_cut ? R : 0;
  const int t = blockIdx.x;
  const int row = t < n_target ? t : R + (t - n_target);
  const bool qrow = row >= R;
  const float *x = qrow ? P.q_logits + static_cast<int64_t>(row - R) * V
                        : P.w.logits + static_cast<int64_t>(row) * V;
  const float2 *part = qrow ? P.w.part_q + static_cast<int64_t>(row - R) * P.dims.nsub
                            : P.w.part_p + static_cast<int64_t>(row) * P.dims.nsub;
  const int top_k = qrow ? P.q_top_k : P.p_top_k;
  const float top_p = qrow ? P.q_top_p : P.p_top_p;
  const float inv_t = P.inv_t;

  // row maximum of x / T from the contraction's partials
  float m = -INFINITY;
  int bad = 0;
  for (int s = threadIdx.x; s < P.dims.nsub; s += kTruncThreads) {
    const float2 pm = __ldcg(&part[s]);
    bad |= (isnan(pm.x) || pm.x == INFINITY) ? 1 : 0;
    m = fmaxf(m, pm.x);
  }
  bad = __syncthreads_or(bad);
  const float M = block_max_f(m, s_warp_f);
  if (bad || !(M > -INFINITY)) {
    if (threadIdx.x == 0) {
      P.w.row_m[row] = bad ? NAN : M;
      st_ff_raw(&P.w.row_s[row], ff_make(0.0f));
      P.w.row_tau[row] = -INFINITY;
    }
    return;
  }

  // top-k: the k-th largest key
  uint32_t tau = 0;  // below every key: nothing cut
  if (top_k > 0 && static_cast<int64_t>(top_k) < V) {
    uint32_t prefix = 0, pmask = 0;
    int kr = top_k;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = digit_shift(pass);
      const uint32_t dm = digit_mask(pass);
      for (int i = threadIdx.x; i < kBins; i += kTruncThreads) s_cnt[i] = 0;
      __syncthreads();
      for_each_entry(x, V, [&](float v) {
        const uint32_t key = float_key(v);
        if ((key & pmask) == prefix) atomicAdd(&s_cnt[(key >> shift) & dm], 1);
      });
      __syncthreads();
      find_cut_bin<int>(s_cnt, s_cnt, static_cast<int>(dm) + 1, kr, &s_bin, &s_above_i,
                        s_warp_i, s_incl_i, &s_owner);
      prefix |= static_cast<uint32_t>(s_bin) << shift;
      pmask |= dm << shift;
      kr -= s_above_i;
      __syncthreads();
    }
    tau = prefix;
  }

  // top-p over the top-k set: the key at which the descending cumulative
  // mass reaches top_p of that set's mass
  if (top_p < 1.0f) {
    const uint32_t tau_k = tau;
    uint32_t prefix = 0, pmask = 0;
    u64 r = 0;
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = digit_shift(pass);
      const uint32_t dm = digit_mask(pass);
      for (int i = threadIdx.x; i < kBins; i += kTruncThreads) {
        s_cnt[i] = 0;
        s_mass[i] = 0;
      }
      __syncthreads();
      u64 mine = 0;
      for_each_entry(x, V, [&](float v) {
        const uint32_t key = float_key(v);
        if (key >= tau_k && (key & pmask) == prefix) {
          const u64 w = fixed_mass(expf(fmaf(v, inv_t, -M)));
          const uint32_t dg = (key >> shift) & dm;
          atomicAdd(&s_mass[dg], w);
          atomicAdd(&s_cnt[dg], 1);
          mine += w;
        }
      });
      if (pass == 0) {
        // the top-k set's mass (exact), and the smallest integer mass that
        // reaches top_p of it
        const u64 total = block_suffix_incl(mine, s_warp_u);
        if (threadIdx.x == 0) s_above_u = total;
        __syncthreads();
        r = static_cast<u64>(ceil(static_cast<double>(top_p) * static_cast<double>(s_above_u)));
      }
      __syncthreads();
      find_cut_bin<u64>(s_mass, s_cnt, static_cast<int>(dm) + 1, r, &s_bin, &s_above_u,
                        s_warp_u, s_incl_u, &s_owner);
      prefix |= static_cast<uint32_t>(s_bin) << shift;
      pmask |= dm << shift;
      r = r > s_above_u ? r - s_above_u : 0;
      __syncthreads();
    }
    tau = prefix > tau ? prefix : tau;
  }

  // the kept mass, in a fixed order
  float ssum = 0.0f;
  for_each_entry(x, V, [&](float v) {
    if (float_key(v) >= tau) ssum = __fadd_rn(ssum, expf(fmaf(v, inv_t, -M)));
  });
  const ff S = block_sum_ff(ff_make(ssum), s_wff);
  if (threadIdx.x == 0) {
    P.w.row_m[row] = M;
    st_ff_raw(&P.w.row_s[row], S);
    P.w.row_tau[row] = tau == 0 ? -INFINITY : key_float(tau);
  }
}

}  // namespace

cudaError_t launch_trunc(const TruncParams &P, cudaStream_t stream) {
  const int rows = (P.p_cut ? P.dims.R : 0) + (P.q_cut ? P.dims.RQ : 0);
  if (rows == 0) return cudaSuccess;
  void *args[] = {const_cast<TruncParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&trunc_kernel), dim3(rows),
                    dim3(kTruncThreads), 0, stream, args);
}

}  // namespace sv
