// sv_kernels.h -- launch interfaces of the kernels of the verify step
// (host side of the library; see sv_api.cu for the C ABI).
#pragma once

#include "sv_internal.cuh"

namespace sv {

// ---- (a) LM-head contraction, bf16 tensor-core path -----------------------
struct TcParams {
  Dims dims;
  Work w;
  const float *q_logits;   // [RQ, V]
  float inv_t;             // 1/T (T > 0); unused for greedy
  int greedy;              // T == 0
  int npad;                // MMA N = R rounded up to 16
  int nkb;                 // k blocks (128 bytes of a row) per tile
  int kbk;                 // elements per k block: 64 (bf16) or 128 (FP8 E4M3)
  int fp8;                 // FP8 E4M3 operands (kind::f8f6f4) and scales
  const float *h_scale;    // FP8: [R] hidden-row scales
  const float *w_scale;    // FP8: [V] vocabulary-row scales
  int chunks;              // k blocks per stage (one 3-D TMA box when > 1)
  int stages;              // shared-memory ring depth
  int stage_bytes;         // W slab + H slab, multiple of 1024
  int h_boxes;             // TMA boxes per H slab (1 or 2)
  int h_box_rows;          // rows per H box
  int nslot;               // direct mode: TMEM accumulators per tile
  int nbuf;                // direct mode: tiles in TMEM at once (1 or 2)
  int tma_logits;          // logits written by TMA stores (needs V % 4 == 0)
  int half;                // CTAs 2p, 2p+1 share tiles, npad columns each
  uint32_t tmem_cols;      // TMEM columns allocated per CTA
  uint64_t wait_limit_ns;  // bound of every device-side wait
  unsigned epoch;          // run counter (stamps an abort)
  int row_stats;           // drain mode, T > 0: write w.rowpart (per-CTA row pairs)
  const void *H;           // [R, d] bf16 / FP8 hidden states (draft-token logits)
  const void *W;           // [V, d] bf16 / FP8 LM head
  const int32_t *draft;    // [B, K]
};

struct TcPlan {
  int npad, ncol, nkb, kbk, chunks, stage_bytes, stages, smem, h_boxes, h_box_rows, nslot, nbuf;
  int half;  // npad is then the columns of one CTA of a pair (half of all)
  uint32_t tmem_cols;
  int grid, threads;
  bool valid;
};

// elt: bytes per element of hidden and W (2: bf16, 1: FP8 E4M3)
TcPlan plan_tc(const Dims &dims, int num_sms, int smem_optin, int elt);
cudaError_t launch_tc(const TcPlan &pl, const TcParams &P, const CUtensorMap &tmW,
                      const CUtensorMap &tmH, const CUtensorMap &tmL, cudaStream_t stream);

// ---- (a) LM-head contraction, fp32 SIMT path -----------------------------
struct SimtParams {
  Dims dims;
  Work w;
  const float *H;          // [R, d]
  const float *W;          // [V, d]
  const float *q_logits;   // [RQ, V]
  float inv_t;
  int greedy;
};
cudaError_t launch_simt(const SimtParams &P, cudaStream_t stream);

// ---- (b) decision/residual and (c) selection, one fused launch -----------
struct TailParams {
  Dims dims;
  Work w;
  const void *H;           // [R, d] bf16 or fp32
  const void *W;           // [V, d] bf16 or fp32
  int dtype;               // SV_BF16 / SV_FP32
  const int32_t *draft;    // [B, K]
  const float *q_logits;   // [RQ, V]
  const float *u;          // [B, K+1]
  double T;
  float inv_t;
  int greedy;
  int32_t *out_tokens;     // [B, K+1]
  int32_t *out_n;          // [B]
  unsigned epoch;          // run counter
  uint64_t wait_limit_ns;  // bound of the wait for a sequence's decision
  int split_cnt_n;         // entries of w.split_cnt
  int draft_logits_ready;  // w.draft_logit was written by the contraction
  int fast;                // one decision CTA per sequence from w.rowpart and
                           // w.draft_q (the contraction ran with row_stats)
  int grid_parts;          // contraction CTAs: pairs per row in w.rowpart
  int stall;               // tests: CTA 0 first waits for w.never (bounded)
  int coop;                // cooperative selection: the whole tail grid fits
                           // on the GPU at once (see tail_resident_ctas)
  int stage_rows;          // cooperative: rows of each chunk staged in shared
                           // memory by bulk copies (0: read from L2)
  int p_cut, q_cut;        // truncated target / draft rows: (M, S, cut) are given
  const int32_t *parents;  // greedy tree verification: [B, K] node parents (else null)
  const float *h_scale;    // FP8 (dtype SV_FP8): [R] hidden-row scales
  const float *w_scale;    // FP8: [V] vocabulary-row scales
  int32_t *out_nodes;      // tree: [B, K] accepted path's nodes (may be null)
};
cudaError_t launch_tail(const TailParams &P, cudaStream_t stream);
// CTAs of the cooperative tail kernel that fit on the GPU at once with
// stage_bytes of dynamic shared memory each (0 if unknown).
int tail_resident_ctas(int num_sms, int stage_bytes);
// Shared memory that staging a chunk of the final draw's candidate rows
// takes (K+1 target rows, and the K draft rows if with_q), or 0 when it is
// not used (V not a multiple of 4, or above kStageMaxBytes).
constexpr int kStageMaxBytes = 200 * 1024;
int tail_stage_bytes(const Dims &d, bool with_q);

// ---- truncated sampling: (M, S, cut) of every truncated row --------------
struct TruncParams {
  Dims dims;
  Work w;
  const float *q_logits;   // [RQ, V]
  float inv_t;
  int p_cut, q_cut;        // which side is truncated
  int p_top_k, q_top_k;    // 0: no top-k
  float p_top_p, q_top_p;  // 1: no top-p
};
cudaError_t launch_trunc(const TruncParams &P, cudaStream_t stream);

// cudaLaunchKernelEx with programmatic stream serialisation (PDL).
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, void **args);

}  // namespace sv
