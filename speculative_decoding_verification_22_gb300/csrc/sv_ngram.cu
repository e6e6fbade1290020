// sv_ngram.cu -- prompt-lookup drafting on the GPU ("Speculative Decoding:
// Guess Several Tokens, Check Them in One Pass", "Drafts without a model";
// "Speculative Decoding: Two Models, One Voice", "No model at all").
//
// One CTA per sequence.  For n = n_max down to n_min the CTA stages the last
// n context tokens in shared memory and scans candidate starts j from the
// end of the context backwards, one block-sized slab at a time, each thread
// comparing one start; the first slab with a match holds the latest
// occurrence (the largest matching j, by an atomicMax), so the scan stops
// there.  The work is proportional to the distance from the end to the
// latest occurrence, at most n_max * length token comparisons per n.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace sv {
namespace {

constexpr int kNgramThreads = 256;

__global__ void __launch_bounds__(kNgramThreads)
    ngram_draft_kernel(const int32_t *__restrict__ tokens, int64_t ld,
                       const int32_t *__restrict__ lengths, int K, int n_min, int n_max,
                       int32_t *__restrict__ out_draft, int32_t *__restrict__ out_len) {
  __shared__ int32_t s_pat[SV_NGRAM_MAX];
  __shared__ int s_best, s_n;
  const int b = blockIdx.x;
  const int32_t *t = tokens + static_cast<int64_t>(b) * ld;
  int64_t len = lengths[b];
  if (len < 0 || len > ld) len = 0;
  if (threadIdx.x == 0) {
    s_best = -1;
    s_n = 0;
  }
  for (int n = n_max; n >= n_min; --n) {
    if (static_cast<int64_t>(n) >= len) continue;  // needs n + 1 tokens at least
    __syncthreads();
    if (threadIdx.x < n) s_pat[threadIdx.x] = t[len - n + threadIdx.x];
    __syncthreads();
    // starts j in [0, len - n - 1], latest first
    for (int64_t top = len - n - 1; top >= 0; top -= kNgramThreads) {
      const int64_t j = top - threadIdx.x;
      bool match = j >= 0;
      for (int k = 0; k < n && match; ++k) match = t[j + k] == s_pat[k];
      if (match) atomicMax(&s_best, static_cast<int>(j));
      if (__syncthreads_or(match)) break;
    }
    if (s_best >= 0) {
      if (threadIdx.x == 0) s_n = n;
      break;
    }
  }
  __syncthreads();
  const int j = s_best, n = s_n;
  const int64_t avail = j >= 0 ? len - (j + n) : 0;
  const int m = static_cast<int>(avail < K ? avail : K);
  for (int k = threadIdx.x; k < K; k += kNgramThreads)
    out_draft[static_cast<int64_t>(b) * K + k] = k < m ? t[j + n + k] : -1;
  if (threadIdx.x == 0) out_len[b] = m;
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace sv

extern "C" int spec_ngram_draft(const int32_t *tokens, int64_t ld, const int32_t *lengths,
                                int32_t B, int32_t K, int32_t n_min, int32_t n_max,
                                int32_t *out_draft, int32_t *out_len, void *stream) {
  if (!tokens || !lengths || !out_draft || !out_len) return SV_ERR_ARG;
  if (B < 1 || ld < 1 || K < 1 || K > SV_MAX_K || n_min < 1 || n_max < n_min ||
      n_max > SV_NGRAM_MAX || ld > (static_cast<int64_t>(1) << 31) - 1)
    return SV_ERR_ARG;
  if (!sv::aligned4(tokens) || !sv::aligned4(lengths) || !sv::aligned4(out_draft) ||
      !sv::aligned4(out_len))
    return SV_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SV_ERR_CUDA;
  if (major != 10 || minor != 3) return SV_ERR_ARCH;
  sv::ngram_draft_kernel<<<B, sv::kNgramThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      tokens, ld, lengths, K, n_min, n_max, out_draft, out_len);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
