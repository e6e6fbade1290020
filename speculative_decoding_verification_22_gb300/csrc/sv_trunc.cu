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
// One CTA per truncated row; logits are compared as order-preserving 32-bit
// keys, masses are exp(x / T - M) with M the row maximum (from the
// contraction's per-32-entry partials).
//
// Fast path (1 <= top_k <= kFastK): the contraction's per-subtile maxima
// bound the cut.  If t0 is the k-th largest subtile maximum, k entries are
// >= t0, so every entry of the top-k set (ties included) is >= t0 and lies in
// a subtile whose maximum is >= t0.  The CTA stages the subtile maxima in
// shared memory, selects t0, gathers the entries >= t0 of those subtiles
// (about k * 32) and finishes in shared memory: a radix select for the
// k-th largest, then, for top-p, a rank of every kept entry (at most
// kFastKept) and a scan of their masses in descending order.  No pass over
// the whole row.
//
// General path (larger k, or top-p alone): a three-pass radix select over
// the whole row (11, 11 and 10 bits from the top; counts for top-k, masses
// for top-p restricted to the top-k set; eight 16-byte loads in flight per
// thread), then one pass that sums the kept mass in a fixed order.
//
// The decision kernel reads (M, S, cut) instead of reducing the partials.
#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {
namespace {

constexpr int kTruncThreads = kTailThreads;  // the block helpers assume it
constexpr int kBins = 2048;                  // 11-bit digits
constexpr int kLoadsInFlight = 8;            // 16-byte loads per thread per batch
constexpr int kFastK = 256;                  // largest top_k of the fast path
constexpr int kMaxSub = 4096;                // subtile maxima staged (V <= 131072)
constexpr int kCandCap = 2048;               // gathered candidate entries
constexpr int kFastKept = kTruncThreads;     // kept entries ranked for top-p
// Fixed-point unit of the general path's bin masses: a weight exp(x/T - M)
// <= 1 is added as round(w * 2^e), e = min(44, 62 - ceil(log2 V)), so a
// row's total stays below 2^63 and each weight carries an absolute error
// of at most 2^-(e+1) (2^-45 up to V = 2^18).
__device__ __forceinline__ float mass_unit(int64_t V) {
  int bits = 0;
  while ((int64_t(1) << bits) < V) ++bits;
  const int e = 62 - bits < 44 ? 62 - bits : 44;
  return __int_as_float((127 + e) << 23);  // 2^e, exactly
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

// Applies f(value) to every entry of a row, kLoadsInFlight 16-byte loads in
// flight per thread where the row is 16-byte aligned.
template <typename F>
__device__ __forceinline__ void for_each_entry(const float *row, int64_t V, F f) {
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const int64_t n4 = V / 4;
    for (int64_t base = threadIdx.x; base < n4; base += kTruncThreads * kLoadsInFlight) {
      float4 a[kLoadsInFlight];
#pragma unroll
      for (int j = 0; j < kLoadsInFlight; ++j) {
        const int64_t i = base + static_cast<int64_t>(j) * kTruncThreads;
        a[j] = i < n4 ? __ldcg(&r4[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kLoadsInFlight; ++j) {
        if (base + static_cast<int64_t>(j) * kTruncThreads < n4) {
          f(a[j].x);
          f(a[j].y);
          f(a[j].z);
          f(a[j].w);
        }
      }
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

// Shared memory of one CTA (about 40 KB).  The general path's mass
// histogram and the fast path's buffers are never live together.
struct TruncSmem {
  int cnt[kBins];
  int incl_i[kTruncThreads];
  float incl_f[kTruncThreads];
  int warp_i[kTailWarps];
  float warp_f[kTailWarps];
  ff warp_ff[kTailWarps];
  int owner, bin, n, overflow;
  union {
    struct {  // general path: bin masses in fixed point, then as floats
      unsigned long long mass_fx[kBins];
      float mass[kBins];
    } g;
    struct {
      float sub_max[kMaxSub];  // subtile maxima
      float cand[kCandCap];    // candidate entries
      float kept_w[kFastKept];
      uint32_t kept_key[kFastKept];
    } f;
  } u;
};

// The highest bin c of hist[0..nb) whose suffix sum (bins c..nb-1) reaches
// r (the lowest non-empty bin if none does); *above_out receives the suffix
// sum of the bins above c.  Thread t owns bins [t * per, (t + 1) * per).
// Block-wide; the result is in sm.bin.
template <typename T>
__device__ void find_cut_bin(TruncSmem &sm, const T *hist, int nb, T r, T *incl_buf, T *warp_buf,
                             T &above_out) {
  __shared__ T s_above;
  const int per = nb / kTruncThreads;
  const int b0 = threadIdx.x * per;
  T mine = T(0);
  bool nonempty = false;
  for (int j = 0; j < per; ++j) {
    mine += hist[b0 + j];
    nonempty = nonempty || sm.cnt[b0 + j] > 0;
  }
  if (threadIdx.x == 0) sm.owner = -1;
  const T incl = block_suffix_incl(mine, warp_buf);
  incl_buf[threadIdx.x] = incl;
  __syncthreads();
  if (incl >= r) atomicMax(&sm.owner, static_cast<int>(threadIdx.x));
  __syncthreads();
  if (sm.owner < 0) {
    // nothing reaches r: the owner of the lowest non-empty bin
    if (threadIdx.x == 0) sm.owner = kTruncThreads;
    __syncthreads();
    if (nonempty) atomicMin(&sm.owner, static_cast<int>(threadIdx.x));
    __syncthreads();
    if (sm.owner == kTruncThreads) {  // empty histogram (not reached for valid rows)
      if (threadIdx.x == 0) {
        sm.bin = 0;
        s_above = T(0);
      }
      __syncthreads();
      above_out = s_above;
      return;
    }
  }
  if (static_cast<int>(threadIdx.x) == sm.owner) {
    T acc = threadIdx.x + 1 < kTruncThreads ? incl_buf[threadIdx.x + 1] : T(0);
    int c = -1, low = -1;
    T above = acc, above_low = acc;
    for (int j = per - 1; j >= 0; --j) {
      const T next = acc + hist[b0 + j];
      if (sm.cnt[b0 + j] > 0) {
        low = b0 + j;
        above_low = acc;
      }
      if (next >= r && sm.cnt[b0 + j] > 0) {
        c = b0 + j;
        above = acc;
        break;
      }
      acc = next;
    }
    sm.bin = c < 0 ? low : c;
    s_above = c < 0 ? above_low : above;
  }
  __syncthreads();
  above_out = s_above;
  __syncthreads();
}

// The k-th largest key among n values in shared memory (radix select).
__device__ uint32_t kth_largest_smem(TruncSmem &sm, const float *vals, int n, int k) {
  uint32_t prefix = 0, pmask = 0;
  int kr = k;
  for (int p = 0; p < 3; ++p) {
    const int shift = digit_shift(p);
    const uint32_t dm = digit_mask(p);
    for (int i = threadIdx.x; i < kBins; i += kTruncThreads) sm.cnt[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kTruncThreads) {
      const uint32_t key = float_key(vals[i]);
      if ((key & pmask) == prefix) atomicAdd(&sm.cnt[(key >> shift) & dm], 1);
    }
    __syncthreads();
    int above = 0;
    find_cut_bin<int>(sm, sm.cnt, static_cast<int>(dm) + 1, kr, sm.incl_i, sm.warp_i, above);
    kr -= above;
    prefix |= static_cast<uint32_t>(sm.bin) << shift;
    pmask |= dm << shift;
    __syncthreads();
  }
  return prefix;
}

// At most 72 registers per thread (36,864 for a 512-thread CTA).
__global__ void __maxnreg__(72) trunc_kernel(const TruncParams P) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TruncSmem &sm = *reinterpret_cast<TruncSmem *>(smem_raw);

  const int R = P.dims.R;
  const int64_t V = P.dims.V;
  const int nsub = P.dims.nsub;
  const int n_target = P.p_cut ? R : 0;
  const int t = blockIdx.x;
  const int row = t < n_target ? t : R + (t - n_target);
  const bool qrow = row >= R;
  const float *x = qrow ? P.q_logits + static_cast<int64_t>(row - R) * V
                        : P.w.logits + static_cast<int64_t>(row) * V;
  const float2 *part = qrow ? P.w.part_q + static_cast<int64_t>(row - R) * nsub
                            : P.w.part_p + static_cast<int64_t>(row) * nsub;
  const int top_k = qrow ? P.q_top_k : P.p_top_k;
  const float top_p = qrow ? P.q_top_p : P.p_top_p;
  const float inv_t = P.inv_t;
  // the subtile bound needs k subtile maxima
  const bool fast = top_k >= 1 && top_k <= kFastK && static_cast<int64_t>(top_k) < V &&
                    top_k <= nsub && nsub <= kMaxSub;

  // row maximum of x / T from the contraction's partials (staged, fast path)
  float m = -INFINITY;
  int bad = 0;
  for (int s = threadIdx.x; s < nsub; s += kTruncThreads) {
    const float2 pm = __ldcg(&part[s]);
    bad |= (isnan(pm.x) || pm.x == INFINITY) ? 1 : 0;
    m = fmaxf(m, pm.x);
    if (fast) sm.u.f.sub_max[s] = pm.x;
  }
  bad = __syncthreads_or(bad);
  const float M = block_max_f(m, sm.warp_f);
  if (bad || !(M > -INFINITY)) {
    if (threadIdx.x == 0) {
      P.w.row_m[row] = bad ? NAN : M;
      st_ff_raw(&P.w.row_s[row], ff_make(0.0f));
      P.w.row_tau[row] = -INFINITY;
    }
    return;
  }

  uint32_t tau = 0;  // below every key: nothing cut
  bool done = false;
  ff S = ff_make(0.0f);

  if (fast) {
    // t0: the k-th largest subtile maximum (of x * inv_t, as the partials)
    const float t0 = key_float(kth_largest_smem(sm, sm.u.f.sub_max, nsub, top_k));
    // gather the entries >= t0 of the subtiles whose maximum reaches t0:
    // list those subtiles (in the candidate buffer, as ints), then load
    // their entries with every thread at once
    if (threadIdx.x == 0) {
      sm.n = 0;
      sm.overflow = 0;
    }
    __syncthreads();
    int *list = reinterpret_cast<int *>(sm.u.f.cand);
    constexpr int kListCap = kCandCap / 2;  // the list sits in the first half
    for (int s = threadIdx.x; s < nsub; s += kTruncThreads) {
      if (sm.u.f.sub_max[s] >= t0) {
        const int slot = atomicAdd(&sm.overflow, 1);
        if (slot < kListCap) list[slot] = s;
      }
    }
    __syncthreads();
    const int nlist = sm.overflow;
    if (nlist <= kListCap) {
      // entries in list order; the values go to the second half
      float *vals = sm.u.f.cand + kListCap;
      const int total = nlist * kSub;
      for (int e = threadIdx.x; e < total; e += kTruncThreads) {
        const int64_t v = static_cast<int64_t>(list[e / kSub]) * kSub + (e % kSub);
        const float val = v < V ? __ldcg(&x[v]) : -INFINITY;
        if (v < V && val * inv_t >= t0) {
          const int slot = atomicAdd(&sm.n, 1);
          if (slot < kCandCap - kListCap) vals[slot] = val;
        }
      }
      __syncthreads();
      // move the values to the front of the buffer
      const int nv = sm.n < kCandCap - kListCap ? sm.n : 0;
      float tmp[(kCandCap - kListCap) / kTruncThreads];
#pragma unroll
      for (int j = 0; j < (kCandCap - kListCap) / kTruncThreads; ++j) {
        const int i = threadIdx.x + j * kTruncThreads;
        tmp[j] = i < nv ? vals[i] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < (kCandCap - kListCap) / kTruncThreads; ++j) {
        const int i = threadIdx.x + j * kTruncThreads;
        if (i < nv) sm.u.f.cand[i] = tmp[j];
      }
      if (threadIdx.x == 0 && sm.n > kCandCap - kListCap) sm.n = kCandCap + 1;
    } else if (threadIdx.x == 0) {
      sm.n = kCandCap + 1;  // too many subtiles: general path
    }
    __syncthreads();
    const int n = sm.n;
    if (n <= kCandCap) {
      // the exact k-th largest entry among the candidates
      tau = kth_largest_smem(sm, sm.u.f.cand, n, top_k);
      if (top_p >= 1.0f) {
        // the kept mass in 64-bit fixed point (2^-40 units): exact, so
        // independent of the order the candidates were gathered in
        unsigned long long mine = 0;
        for (int i = threadIdx.x; i < n; i += kTruncThreads) {
          const float v = sm.u.f.cand[i];
          if (float_key(v) >= tau)
            mine += __float2ull_rn(expf(fmaf(v, inv_t, -M)) * 1099511627776.0f);
        }
        __shared__ unsigned long long s_wu[kTailWarps];
        const unsigned long long tot = block_suffix_incl(mine, s_wu);
        __shared__ unsigned long long s_tot;
        if (threadIdx.x == 0) s_tot = tot;
        __syncthreads();
        const unsigned long long kept = s_tot;
        const float hi = __ull2float_rn(kept);
        const float lo = __ll2float_rn(static_cast<long long>(kept - __float2ull_rn(hi)));
        S = ff{hi * (1.0f / 1099511627776.0f), lo * (1.0f / 1099511627776.0f)};
        done = true;
      } else {
        // compact the kept set, rank it by key (ties by position), scan its
        // masses in descending order
        if (threadIdx.x == 0) sm.n = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kTruncThreads) {
          const float v = sm.u.f.cand[i];
          const uint32_t key = float_key(v);
          if (key >= tau) {
            const int slot = atomicAdd(&sm.n, 1);
            if (slot < kFastKept) {
              sm.u.f.kept_key[slot] = key;
              sm.u.f.kept_w[slot] = v;  // value for now
            }
          }
        }
        __syncthreads();
        const int nk = sm.n;
        if (nk <= kFastKept) {
          // rank of entry i: keys above it, and equal keys stored before it
          const int i = threadIdx.x;
          uint32_t key = 0;
          float v = 0.0f;
          int rank = -1;
          if (i < nk) {
            key = sm.u.f.kept_key[i];
            v = sm.u.f.kept_w[i];
            rank = 0;
            for (int j = 0; j < nk; ++j) {
              const uint32_t kj = sm.u.f.kept_key[j];
              rank += (kj > key || (kj == key && j < i)) ? 1 : 0;
            }
          }
          __syncthreads();
          if (i < nk) {
            sm.u.f.kept_key[rank] = key;
            sm.u.f.kept_w[rank] = expf(fmaf(v, inv_t, -M));
          }
          __syncthreads();
          // inclusive prefix sums of the masses in rank order (thread = rank)
          const float w = i < nk ? sm.u.f.kept_w[i] : 0.0f;
          float inc = w;
          const int lane2 = threadIdx.x & 31, warp2 = threadIdx.x >> 5;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane2 >= o) inc += y;
          }
          if (lane2 == 31) sm.warp_f[warp2] = inc;
          __syncthreads();
          float before = 0.0f;
          for (int w2 = 0; w2 < warp2; ++w2) before += sm.warp_f[w2];
          const float cum = before + inc;
          sm.incl_f[threadIdx.x] = cum;
          __syncthreads();
          const float total = sm.incl_f[nk - 1];
          const float target = top_p * total;
          // the first rank whose cumulative mass reaches the target
          if (threadIdx.x == 0) sm.owner = nk - 1;
          __syncthreads();
          if (i < nk && cum >= target) atomicMin(&sm.owner, i);
          __syncthreads();
          const uint32_t tp = sm.u.f.kept_key[sm.owner];
          // ties at the cut are kept: the last rank with that key
          if (threadIdx.x == 0) sm.bin = sm.owner;
          __syncthreads();
          if (i < nk && sm.u.f.kept_key[i] == tp) atomicMax(&sm.bin, i);
          __syncthreads();
          tau = tp;
          const float s_kept = sm.incl_f[sm.bin];
          S = ff_make(s_kept);
          done = true;
        }
      }
    }
    __syncthreads();
  }

  if (!done) {
    // general path: radix select over the whole row
    tau = 0;
    if (top_k > 0 && static_cast<int64_t>(top_k) < V) {
      uint32_t prefix = 0, pmask = 0;
      int kr = top_k;
      for (int p = 0; p < 3; ++p) {
        const int shift = digit_shift(p);
        const uint32_t dm = digit_mask(p);
        for (int i = threadIdx.x; i < kBins; i += kTruncThreads) sm.cnt[i] = 0;
        __syncthreads();
        for_each_entry(x, V, [&](float v) {
          const uint32_t key = float_key(v);
          if ((key & pmask) == prefix) atomicAdd(&sm.cnt[(key >> shift) & dm], 1);
        });
        __syncthreads();
        int above = 0;
        find_cut_bin<int>(sm, sm.cnt, static_cast<int>(dm) + 1, kr, sm.incl_i, sm.warp_i, above);
        kr -= above;
        prefix |= static_cast<uint32_t>(sm.bin) << shift;
        pmask |= dm << shift;
        __syncthreads();
      }
      tau = prefix;
    }
    if (top_p < 1.0f) {
      const uint32_t floor = tau;
      uint32_t prefix = 0, pmask = 0;
      float r = 0.0f;
      for (int p = 0; p < 3; ++p) {
        const int shift = digit_shift(p);
        const uint32_t dm = digit_mask(p);
        const float unit = mass_unit(V);
        for (int i = threadIdx.x; i < kBins; i += kTruncThreads) {
          sm.cnt[i] = 0;
          sm.u.g.mass_fx[i] = 0ull;
        }
        __syncthreads();
        float mine = 0.0f;
        for_each_entry(x, V, [&](float v) {
          const uint32_t key = float_key(v);
          if (key >= floor && (key & pmask) == prefix) {
            const float w = expf(fmaf(v, inv_t, -M));
            const uint32_t dg = (key >> shift) & dm;
            // integer adds commute: the bin masses, and so the cut, do not
            // depend on the order the threads add in
            atomicAdd(&sm.u.g.mass_fx[dg], __float2ull_rn(w * unit));
            atomicAdd(&sm.cnt[dg], 1);
            mine = __fadd_rn(mine, w);
          }
        });
        if (p == 0) r = ff_to_f(ff_mul_f(block_sum_ff(ff_make(mine), sm.warp_ff), top_p));
        __syncthreads();
        for (int i = threadIdx.x; i < kBins; i += kTruncThreads)
          sm.u.g.mass[i] = __ull2float_rn(sm.u.g.mass_fx[i]) / unit;
        __syncthreads();
        float above = 0.0f;
        find_cut_bin<float>(sm, sm.u.g.mass, static_cast<int>(dm) + 1, r, sm.incl_f, sm.warp_f,
                            above);
        r -= above;
        prefix |= static_cast<uint32_t>(sm.bin) << shift;
        pmask |= dm << shift;
        __syncthreads();
      }
      tau = prefix > tau ? prefix : tau;
    }
    // the kept mass, in a fixed order
    float mine = 0.0f;
    for_each_entry(x, V, [&](float v) {
      if (float_key(v) >= tau) mine = __fadd_rn(mine, expf(fmaf(v, inv_t, -M)));
    });
    S = block_sum_ff(ff_make(mine), sm.warp_ff);
  }

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
  const size_t smem = sizeof(TruncSmem);
  cudaError_t e = cudaFuncSetAttribute(trunc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  void *args[] = {const_cast<TruncParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&trunc_kernel), dim3(rows),
                    dim3(kTruncThreads), smem, stream, args);
}

}  // namespace sv
