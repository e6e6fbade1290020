// sv_ngram.cu -- prompt-lookup drafting on the GPU ("Speculative Decoding:
// Guess Several Tokens, Check Them in One Pass", "Drafts without a model";
// "Speculative Decoding: Two Models, One Voice", "No model at all").
//
// One CTA per sequence, one pass.  An occurrence of the last n tokens that
// ends at position e (e <= len - 2, so at least one token follows it) is a
// position whose n tokens up to e equal the context's last n tokens, i.e.
// the common suffix of t[0..e] and t[0..len-1] has length >= n.  Each thread
// takes end positions e, counts that common suffix (up to n_max, comparing
// against the context's suffix staged in shared memory) and, for every n it
// reaches, raises the latest end seen for n with a shared-memory atomicMax.
// The longest n with an occurrence wins; its latest occurrence starts at
// e - n + 1 and the draft is the tokens after e.  The context is staged in
// shared memory when it fits (one coalesced load), else read from global
// memory.  Work: O(length * common-suffix length), one barrier.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"

namespace sv {
namespace {

constexpr int kNgramThreads = 256;
constexpr int64_t kNgramSmemTokens = 48 * 1024;  // 192 KB of context in shared memory

__global__ void __launch_bounds__(kNgramThreads)
    ngram_draft_kernel(const int32_t *__restrict__ tokens, int64_t ld,
                       const int32_t *__restrict__ lengths, int K, int n_min, int n_max,
                       int staged, int32_t *__restrict__ out_draft,
                       int32_t *__restrict__ out_len) {
  extern __shared__ int32_t s_ctx[];
  __shared__ int32_t s_suf[SV_NGRAM_MAX];  // s_suf[k] = t[len - 1 - k]
  __shared__ int s_end[SV_NGRAM_MAX + 1];  // latest end position per n
  // the context may be written by earlier work in the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int32_t *t = tokens + static_cast<int64_t>(b) * ld;
  int64_t len = lengths[b];
  if (len < 0 || len > ld) len = 0;
  if (threadIdx.x <= SV_NGRAM_MAX) s_end[threadIdx.x] = -1;
  if (threadIdx.x < n_max && threadIdx.x < len) s_suf[threadIdx.x] = t[len - 1 - threadIdx.x];
  if (staged)
    for (int64_t i = threadIdx.x; i < len; i += kNgramThreads) s_ctx[i] = t[i];
  __syncthreads();
  const int32_t *ctx = staged ? s_ctx : t;
  for (int64_t e = threadIdx.x; e + 1 < len; e += kNgramThreads) {
    int c = 0;
    while (c < n_max && c <= e && ctx[e - c] == s_suf[c]) ++c;
    for (int n = n_min; n <= c; ++n) atomicMax(&s_end[n], static_cast<int>(e));
  }
  __syncthreads();
  int n = n_max;
  while (n >= n_min && s_end[n] < 0) --n;
  const int64_t e = n >= n_min ? s_end[n] : -1;
  const int64_t avail = e >= 0 ? len - 1 - e : 0;
  const int m = static_cast<int>(avail < K ? avail : K);
  for (int k = threadIdx.x; k < K; k += kNgramThreads)
    out_draft[static_cast<int64_t>(b) * K + k] = k < m ? ctx[e + 1 + k] : -1;
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
  const int staged = ld <= sv::kNgramSmemTokens ? 1 : 0;
  const size_t smem = staged ? static_cast<size_t>(ld) * sizeof(int32_t) : 0;
  // above the default 48 KB the kernel must opt in (per device)
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(sv::ngram_draft_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B));
  cfg.blockDim = dim3(sv::kNgramThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sv::ngram_draft_kernel, tokens, ld, lengths,
                                           static_cast<int>(K), static_cast<int>(n_min),
                                           static_cast<int>(n_max), staged, out_draft, out_len);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
