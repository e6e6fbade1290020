// sv_lmhead_simt.cu -- kernel (a) of the verify step, fp32 path: the LM-head
// contraction on CUDA cores for small vocabularies and fp32 weights.
//
// Same outputs as the tensor-core path (fp32 logits, per-32-entry softmax
// partials of logits / T and of q_logits / T), so the decision, residual and
// selection passes are shared.  A product of two fp32 values is exact in
// fp64, so each logit is accumulated in fp64 and rounded to fp32 once.
// One warp covers one row and one 32-entry vocabulary subtile; rows past
// R are the draft rows, whose partials are taken straight from q_logits.
#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace sv {

constexpr int kSimtWarps = 8;

__global__ void __launch_bounds__(kSimtWarps * 32) lmhead_simt_kernel(const SimtParams P) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y * kSimtWarps + warp;
  const int sub = blockIdx.x;
  const int64_t V = P.dims.V, d = P.dims.d;
  const int64_t v = static_cast<int64_t>(sub) * kSub + lane;
  const bool valid = v < V;
  if (row < P.dims.R) {
    double acc = 0.0;
    if (valid) {
      const float *h = P.H + static_cast<int64_t>(row) * d;
      const float *w = P.W + v * d;
      for (int64_t k = 0; k < d; ++k) acc += static_cast<double>(h[k]) * static_cast<double>(w[k]);
    }
    const float l = static_cast<float>(acc);
    if (valid) P.w.logits[static_cast<int64_t>(row) * V + v] = l;
    const float2 pm = subtile_partial(l, valid, P.inv_t, P.greedy != 0);
    if (lane == 0) P.w.part_p[static_cast<int64_t>(row) * P.dims.nsub + sub] = pm;
  } else if (!P.greedy && P.q_logits != nullptr && row - P.dims.R < P.dims.RQ) {
    const int rq = row - P.dims.R;
    const float x = valid ? P.q_logits[static_cast<int64_t>(rq) * V + v] : 0.0f;
    const float2 pm = subtile_partial(x, valid, P.inv_t, false);
    if (lane == 0) P.w.part_q[static_cast<int64_t>(rq) * P.dims.nsub + sub] = pm;
  }
}

cudaError_t launch_simt(const SimtParams &P, cudaStream_t stream) {
  const int rows = P.dims.R + ((P.greedy || P.q_logits == nullptr) ? 0 : P.dims.RQ);
  dim3 grid(P.dims.nsub, (rows + kSimtWarps - 1) / kSimtWarps);
  void *args[] = {const_cast<SimtParams *>(&P)};
  return launch_pdl(reinterpret_cast<const void *>(&lmhead_simt_kernel), grid,
                    dim3(kSimtWarps * 32), 0, stream, args);
}

}  // namespace sv
