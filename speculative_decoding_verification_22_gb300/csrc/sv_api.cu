// sv_api.cu -- the C ABI declared in include/spec_verify.h: handle
// lifetime, argument checks, workspace, TMA descriptors and the launch
// sequence of one verify-and-sample step.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace {

constexpr int kTimingRing = 256;

// cuTensorMapEncodeTiled from the driver, looked up once per process (a
// function-local static: its initialisation is thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct spec_verify {
  sv_config_t cfg{};
  int device = 0;
  int num_sms = 0;
  int smem_optin = 0;
  int tail_resident = 0;         // cooperative tail CTAs that fit on the GPU at once
  int stage_bytes = 0;           // shared memory of the staged cooperative tail (0: none)
  int tail_resident_staged = 0;  // the same with stage_bytes of shared memory each
  cudaStream_t stream = nullptr;
  sv::Dims dims{};
  sv::Work w{};
  sv::TcPlan plan{};
  unsigned epoch = 0;
  uint64_t wait_limit_ns = 1000000000ull;
  // staging for spec_verify_run_host
  void *st_hidden = nullptr;
  int32_t *st_draft = nullptr;
  float *st_q = nullptr;
  float *st_u = nullptr;
  int32_t *st_tokens = nullptr;
  int32_t *st_n = nullptr;
  // double-buffered host rounds (spec_verify_submit_host), set up on first use
  struct Slot {
    void *hidden = nullptr;
    int32_t *draft = nullptr, *tokens = nullptr, *n = nullptr;
    float *q = nullptr, *u = nullptr;
    int *status_host = nullptr;  // pinned: the status word after the round
    cudaEvent_t copied = nullptr, kernels = nullptr, done = nullptr;
    bool busy = false;
  } slot[2];
  cudaStream_t h2d = nullptr, d2h = nullptr;
  bool pipe_ready = false;
  // TMA descriptors, re-encoded when the tensor moves
  CUtensorMap tmW{}, tmH{};
  const void *tmW_ptr = nullptr, *tmH_ptr = nullptr;
  // TMA store map of the logits scratch (fixed for the handle's life)
  CUtensorMap tmL{};
  bool tma_logits = false;
  // kernel timing
  bool timing = false;
  bool debug_stall = false;
  std::vector<cudaEvent_t> ev0, ev1;
  int64_t timed = 0, folded = 0;
  double timed_ms = 0.0;
};

namespace {

size_t esize(int dtype) { return dtype == SV_BF16 ? 2 : dtype == SV_FP8 ? 1 : 4; }

void free_all(spec_verify *h) {
  void *ptrs[] = {h->w.logits,    h->w.part_p,      h->w.part_q,    h->w.row_m,
                  h->w.row_s,     h->w.seq,         h->w.chunk_mass, h->w.split_buf,
                  h->w.split_cnt, h->w.status,      h->w.abort_epoch, h->w.ticket,
                  h->w.finished,  h->w.row_count,   h->w.chunk_count, h->w.seq_flag,
                  h->w.seq_final,
                  h->w.cand,      h->w.draft_logit, h->w.row_tau,   h->w.rowpart,
                  h->w.draft_q,   h->w.chunk_done,  h->w.never,
                  h->st_hidden,   h->st_draft,      h->st_q,        h->st_u,
                  h->st_tokens,   h->st_n};
  for (void *p : ptrs)
    if (p) cudaFree(p);
  for (cudaEvent_t e : h->ev0) cudaEventDestroy(e);
  for (cudaEvent_t e : h->ev1) cudaEventDestroy(e);
  for (auto &sl : h->slot) {
    void *dp[] = {sl.hidden, sl.draft, sl.tokens, sl.n, sl.q, sl.u};
    for (void *p : dp)
      if (p) cudaFree(p);
    if (sl.status_host) cudaFreeHost(sl.status_host);
    cudaEvent_t ev[] = {sl.copied, sl.kernels, sl.done};
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  }
  if (h->h2d) cudaStreamDestroy(h->h2d);
  if (h->d2h) cudaStreamDestroy(h->d2h);
}

template <typename T>
bool dalloc(T **p, size_t count) {
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void **>(p), count * sizeof(T)) == cudaSuccess;
}

// TMA map of a row-major [outer, inner] matrix of bf16 (elt 2) or FP8 E4M3
// bytes (elt 1).  A block is one 128-byte row piece: kbk = 128 / elt
// elements.  chunks == 1: 2-D, box {kbk, box_rows}.  chunks > 1: 3-D view
// {kbk, outer, inner / kbk} (the k-chunk dimension has a 128-byte stride),
// box {kbk, box_rows, chunks}, so one copy brings `chunks` consecutive k
// blocks of box_rows rows.
int encode_w(CUtensorMap *map, const void *base, int64_t inner, int64_t outer,
             uint32_t box_rows, int chunks, int elt = 2) {
  auto fn = encode_fn();
  if (!fn) return SV_ERR_CUDA;
  const CUtensorMapDataType type =
      elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint32_t kbk = static_cast<cuuint32_t>(128 / elt);
  CUresult r;
  if (chunks > 1) {
    cuuint64_t dims[3] = {kbk, static_cast<cuuint64_t>(outer),
                          static_cast<cuuint64_t>(inner / kbk)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * elt, 128};
    cuuint32_t box[3] = {kbk, box_rows, static_cast<cuuint32_t>(chunks)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, type, 3, const_cast<void *>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * elt};
    cuuint32_t box[2] = {kbk, box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? SV_OK : SV_ERR_CUDA;
}

// TMA store map of the fp32 logits scratch [R, V]: box of 16 rows x 32
// entries (128 bytes, the 128-byte swizzle span).  Rows must be a multiple
// of 16 bytes apart, so V % 4 == 0.
int encode_logits(CUtensorMap *map, float *base, int64_t V, int64_t R) {
  auto fn = encode_fn();
  if (!fn) return SV_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(R)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 4};
  cuuint32_t box[2] = {32, 16};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SV_OK : SV_ERR_CUDA;
}

// Folds finished timing pairs into the running total (blocking on them).
void fold_timing(spec_verify *h, int64_t upto) {
  for (; h->folded < upto; ++h->folded) {
    const int i = static_cast<int>(h->folded % kTimingRing);
    float ms = 0.0f;
    cudaEventSynchronize(h->ev1[i]);
    if (cudaEventElapsedTime(&ms, h->ev0[i], h->ev1[i]) == cudaSuccess) h->timed_ms += ms;
  }
}

}  // namespace

extern "C" {

int spec_verify_plan(const sv_config_t *cfg, int32_t num_sms, int32_t smem_optin,
                     sv_plan_t *out) {
  if (!cfg || !out || num_sms < 1) return SV_ERR_ARG;
  if (cfg->dtype != SV_BF16 && cfg->dtype != SV_FP8) return SV_ERR_ARG;
  // the shape checks of spec_verify_create
  if (cfg->V < 1 || cfg->V > INT32_MAX || cfg->d < 1 || cfg->d > (1 << 20) || cfg->B < 1 ||
      cfg->B > SV_MAX_B || cfg->K < 0 || cfg->K > SV_MAX_K)
    return SV_ERR_SHAPE;
  if (cfg->d % (cfg->dtype == SV_BF16 ? 8 : 16) != 0) return SV_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(cfg->B) * (cfg->K + 1);
  if (R > SV_MAX_ROWS_BF16 || R * cfg->V > (int64_t(1) << 40)) return SV_ERR_SHAPE;
  sv::Dims D{};
  D.V = cfg->V;
  D.d = cfg->d;
  D.B = cfg->B;
  D.K = cfg->K;
  D.R = static_cast<int>(R);
  D.RQ = cfg->B * cfg->K;
  D.nsub = static_cast<int>((cfg->V + sv::kSub - 1) / sv::kSub);
  D.ntile = static_cast<int>((cfg->V + sv::kTileM - 1) / sv::kTileM);
  D.nchunk = static_cast<int>((cfg->V + sv::kChunk - 1) / sv::kChunk);
  const sv::TcPlan pl = sv::plan_tc(D, num_sms, smem_optin, static_cast<int>(esize(cfg->dtype)));
  if (!pl.valid || pl.smem > smem_optin) return SV_ERR_SHAPE;
  sv_plan_t o{};
  o.npad = pl.npad;
  o.drain_cols = pl.ncol;
  o.half = pl.half;
  o.kblock_elems = pl.kbk;
  o.kblocks = pl.nkb;
  o.chunks = pl.chunks;
  o.stages = pl.stages;
  o.stage_bytes = pl.stage_bytes;
  o.smem_bytes = pl.smem;
  o.grid = pl.grid;
  o.tmem_cols = static_cast<int32_t>(pl.tmem_cols);
  o.tmem_buffers = pl.ncol != 0 ? 1 : pl.nbuf;
  // drain mode: a ring of slots filling the allocation (powers of two)
  o.tmem_slots = pl.ncol != 0 ? static_cast<int32_t>(pl.tmem_cols) / pl.ncol : pl.nslot;
  *out = o;
  return SV_OK;
}

const char *spec_verify_strerror(int code) {
  switch (code) {
    case SV_OK: return "ok";
    case SV_ERR_ARG: return "invalid argument";
    case SV_ERR_ALIGN: return "pointer not 16-byte aligned";
    case SV_ERR_SHAPE: return "shape outside supported limits";
    case SV_ERR_CUDA: return "CUDA call failed";
    case SV_ERR_ARCH: return "device is not compute capability 10.3 (sm_103a)";
    case SV_ERR_TIMEOUT: return "a device-side wait ran out";
    case SV_ERR_TOKEN: return "draft token outside [0, V)";
    case SV_ERR_NONFINITE: return "non-finite logits or draft logits";
    default: return "unknown error";
  }
}

int spec_verify_create(const sv_config_t *cfg, spec_verify_t **out) {
  if (!out) return SV_ERR_ARG;
  *out = nullptr;
  if (!cfg) return SV_ERR_ARG;
  if (cfg->dtype != SV_BF16 && cfg->dtype != SV_FP32 && cfg->dtype != SV_FP8) return SV_ERR_ARG;
  if (cfg->V < 1 || cfg->V > INT32_MAX || cfg->d < 1 || cfg->d > (1 << 20) || cfg->B < 1 ||
      cfg->B > SV_MAX_B || cfg->K < 0 || cfg->K > SV_MAX_K)
    return SV_ERR_SHAPE;
  // rows of 16-byte multiples (TMA and 16-byte loads)
  if (cfg->d % (cfg->dtype == SV_BF16 ? 8 : cfg->dtype == SV_FP8 ? 16 : 4) != 0)
    return SV_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(cfg->B) * (cfg->K + 1);
  if (cfg->dtype != SV_FP32 && R > SV_MAX_ROWS_BF16) return SV_ERR_SHAPE;
  if (R * cfg->V > (int64_t(1) << 40)) return SV_ERR_SHAPE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return SV_ERR_ARCH;

  spec_verify *h = new (std::nothrow) spec_verify();
  if (!h) return SV_ERR_CUDA;
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->smem_optin = static_cast<int>(prop.sharedMemPerBlockOptin);
  h->tail_resident = sv::tail_resident_ctas(h->num_sms, 0);
  h->stream = static_cast<cudaStream_t>(cfg->stream);

  sv::Dims &D = h->dims;
  D.V = cfg->V;
  D.d = cfg->d;
  D.B = cfg->B;
  D.K = cfg->K;
  D.R = static_cast<int>(R);
  D.RQ = cfg->B * cfg->K;
  D.nsub = static_cast<int>((cfg->V + sv::kSub - 1) / sv::kSub);
  D.ntile = static_cast<int>((cfg->V + sv::kTileM - 1) / sv::kTileM);
  D.nchunk = static_cast<int>((cfg->V + sv::kChunk - 1) / sv::kChunk);

  size_t split_floats = 1;
  if (cfg->dtype != SV_FP32) {
    h->plan = sv::plan_tc(D, h->num_sms, h->smem_optin, static_cast<int>(esize(cfg->dtype)));
    if (!h->plan.valid) {
      delete h;
      return SV_ERR_SHAPE;
    }
    split_floats = static_cast<size_t>(h->plan.grid) * 2 * sv::kTileM * h->plan.npad;
    h->stage_bytes = sv::tail_stage_bytes(D, true);
    h->tail_resident_staged =
        h->stage_bytes > 0 ? sv::tail_resident_ctas(h->num_sms, h->stage_bytes) : 0;
  }
  const size_t es = esize(cfg->dtype);
  bool ok = dalloc(&h->w.logits, static_cast<size_t>(R) * D.V) &&
            dalloc(&h->w.part_p, static_cast<size_t>(R) * D.nsub) &&
            dalloc(&h->w.part_q, static_cast<size_t>(D.RQ) * D.nsub) &&
            dalloc(&h->w.row_m, static_cast<size_t>(R + D.RQ)) &&
            dalloc(&h->w.row_s, static_cast<size_t>(R + D.RQ)) && dalloc(&h->w.seq, D.B) &&
            dalloc(&h->w.ticket, 1) && dalloc(&h->w.finished, 1) &&
            dalloc(&h->w.row_count, D.B) && dalloc(&h->w.chunk_count, D.B) &&
            dalloc(&h->w.seq_flag, D.B) &&
            dalloc(&h->w.seq_final, D.B) &&
            dalloc(&h->w.cand, static_cast<size_t>(R) * (1 + sv::kMaxCand)) &&
            dalloc(&h->w.row_tau, static_cast<size_t>(R + D.RQ)) &&
            dalloc(&h->w.draft_logit, static_cast<size_t>(D.RQ)) &&
            dalloc(&h->w.draft_q, static_cast<size_t>(D.RQ)) &&
            dalloc(&h->w.chunk_done, D.B) && dalloc(&h->w.never, 1) &&
            (cfg->dtype == SV_FP32 || h->plan.ncol == 0 ||
             dalloc(&h->w.rowpart, static_cast<size_t>(R + D.RQ) * h->plan.grid)) &&
            dalloc(&h->w.chunk_mass, 2 * static_cast<size_t>(D.B) * D.nchunk) &&
            dalloc(&h->w.split_buf, split_floats) &&
            dalloc(&h->w.split_cnt, static_cast<size_t>(h->num_sms) * 4) &&
            dalloc(&h->w.status, 1) && dalloc(&h->w.abort_epoch, 1) &&
            dalloc(reinterpret_cast<uint8_t **>(&h->st_hidden), static_cast<size_t>(R) * D.d * es) &&
            dalloc(&h->st_draft, static_cast<size_t>(D.RQ)) &&
            dalloc(&h->st_q, static_cast<size_t>(D.RQ) * D.V) && dalloc(&h->st_u, R) &&
            dalloc(&h->st_tokens, R) && dalloc(&h->st_n, D.B);
  if (ok)
    ok = cudaMemset(h->w.split_cnt, 0, sizeof(int) * h->num_sms * 4) == cudaSuccess &&
         cudaMemset(h->w.status, 0, sizeof(int)) == cudaSuccess &&
         cudaMemset(h->w.abort_epoch, 0, sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(h->w.row_m, 0, sizeof(float) * (R + D.RQ)) == cudaSuccess &&
         cudaMemset(h->w.row_s, 0, sizeof(float2) * (R + D.RQ)) == cudaSuccess &&
         cudaMemset(h->w.ticket, 0, sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(h->w.finished, 0, sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(h->w.row_count, 0, sizeof(int) * D.B) == cudaSuccess &&
         cudaMemset(h->w.chunk_count, 0, sizeof(int) * D.B) == cudaSuccess &&
         cudaMemset(h->w.chunk_done, 0, sizeof(int) * D.B) == cudaSuccess &&
         cudaMemset(h->w.never, 0, sizeof(int)) == cudaSuccess &&
         // chunk masses start unset (all-ones bits); every launch leaves them so
         cudaMemset(h->w.chunk_mass, 0xFF, 2 * sizeof(float2) * D.B * D.nchunk) == cudaSuccess &&

         cudaMemset(h->w.seq_flag, 0, sizeof(unsigned) * D.B) == cudaSuccess &&
         cudaMemset(h->w.seq_final, 0, sizeof(int) * D.B) == cudaSuccess &&
         cudaDeviceSynchronize() == cudaSuccess;
  if (ok && cfg->dtype != SV_FP32 && cfg->V % 4 == 0) {
    ok = encode_logits(&h->tmL, h->w.logits, D.V, R) == SV_OK;
    h->tma_logits = ok;
  }
  if (!ok) {
    free_all(h);
    delete h;
    return SV_ERR_CUDA;
  }
  *out = h;
  return SV_OK;
}

void spec_verify_destroy(spec_verify_t *h) {
  if (!h) return;
  cudaStreamSynchronize(h->stream);
  free_all(h);
  delete h;
}

int spec_verify_set_stream(spec_verify_t *h, void *stream) {
  if (!h) return SV_ERR_ARG;
  h->stream = static_cast<cudaStream_t>(stream);
  return SV_OK;
}

int spec_verify_set_wait_limit(spec_verify_t *h, uint64_t limit_ns) {
  if (!h) return SV_ERR_ARG;
  h->wait_limit_ns = limit_ns;
  return SV_OK;
}

int spec_verify_launches_per_run(spec_verify_t *h, float temperature) {
  if (!h) return SV_ERR_ARG;
  (void)temperature;
  return 2;
}

namespace {

// Variants of one run: truncated sampling (which rows are cut, and how) and
// greedy tree verification.
struct TruncSpec {
  int p_cut = 0, q_cut = 0;
  int p_top_k = 0, q_top_k = 0;
  float p_top_p = 1.0f, q_top_p = 1.0f;
  const int32_t *parents = nullptr;
  int32_t *out_nodes = nullptr;
  const float *h_scale = nullptr;  // FP8 handles: hidden-row and vocabulary-row scales
  const float *w_scale = nullptr;
};

int run_impl(spec_verify_t *h, const void *hidden, const void *W_lm,
             const int32_t *draft_tokens, const float *q_logits, const float *uniforms,
             float temperature, int32_t *out_tokens, int32_t *out_n_accepted,
             const TruncSpec &tr);

}  // namespace

int spec_verify_run(spec_verify_t *h, const void *hidden, const void *W_lm,
                    const int32_t *draft_tokens, const float *q_logits, const float *uniforms,
                    float temperature, int32_t *out_tokens, int32_t *out_n_accepted) {
  if (h && h->cfg.dtype == SV_FP8) return SV_ERR_ARG;  // needs the scales: run_fp8
  return run_impl(h, hidden, W_lm, draft_tokens, q_logits, uniforms, temperature, out_tokens,
                  out_n_accepted, TruncSpec{});
}

int spec_verify_run_fp8(spec_verify_t *h, const void *hidden8, const float *hidden_scale,
                        const void *W8, const float *w_scale, const int32_t *draft_tokens,
                        const float *q_logits, const float *uniforms, float temperature,
                        int32_t *out_tokens, int32_t *out_n_accepted) {
  if (!h || h->cfg.dtype != SV_FP8 || !hidden_scale || !w_scale) return SV_ERR_ARG;
  if (!aligned16(hidden_scale) || !aligned16(w_scale)) return SV_ERR_ALIGN;
  TruncSpec tr;
  tr.h_scale = hidden_scale;
  tr.w_scale = w_scale;
  return run_impl(h, hidden8, W8, draft_tokens, q_logits, uniforms, temperature, out_tokens,
                  out_n_accepted, tr);
}

int spec_verify_run_truncated(spec_verify_t *h, const void *hidden, const void *W_lm,
                              const int32_t *draft_tokens, const float *q_logits,
                              const float *uniforms, float temperature, int32_t target_top_k,
                              float target_top_p, int32_t draft_top_k, float draft_top_p,
                              int32_t *out_tokens, int32_t *out_n_accepted) {
  if (!h) return SV_ERR_ARG;
  if (target_top_k < 0 || draft_top_k < 0 || !(target_top_p > 0.0f) || !(target_top_p <= 1.0f) ||
      !(draft_top_p > 0.0f) || !(draft_top_p <= 1.0f))
    return SV_ERR_ARG;
  const sv::Dims &D = h->dims;
  TruncSpec tr;
  const bool sampling = temperature > 0.0f;  // greedy keeps the argmax, which no cut removes
  tr.p_top_k = target_top_k;
  tr.p_top_p = target_top_p;
  tr.q_top_k = draft_top_k;
  tr.q_top_p = draft_top_p;
  tr.p_cut = sampling && ((target_top_k > 0 && target_top_k < D.V) || target_top_p < 1.0f);
  tr.q_cut = sampling && q_logits != nullptr && D.K > 0 &&
             ((draft_top_k > 0 && draft_top_k < D.V) || draft_top_p < 1.0f);
  return run_impl(h, hidden, W_lm, draft_tokens, q_logits, uniforms, temperature, out_tokens,
                  out_n_accepted, tr);
}

int spec_verify_tree_greedy(spec_verify_t *h, const void *hidden, const void *W_lm,
                            const int32_t *tree_tokens, const int32_t *tree_parents,
                            int32_t *out_tokens, int32_t *out_nodes, int32_t *out_n) {
  if (!h) return SV_ERR_ARG;
  if (h->dims.K > 0 && (!tree_tokens || !tree_parents)) return SV_ERR_ARG;
  if ((tree_parents && !aligned16(tree_parents)) || (out_nodes && !aligned16(out_nodes)))
    return SV_ERR_ALIGN;
  TruncSpec tr;
  tr.parents = h->dims.K > 0 ? tree_parents : nullptr;
  tr.out_nodes = out_nodes;
  return run_impl(h, hidden, W_lm, tree_tokens, nullptr, nullptr, 0.0f, out_tokens, out_n, tr);
}

namespace {

int run_impl(spec_verify_t *h, const void *hidden, const void *W_lm,
             const int32_t *draft_tokens, const float *q_logits, const float *uniforms,
             float temperature, int32_t *out_tokens, int32_t *out_n_accepted,
             const TruncSpec &tr) {
  if (!h || !hidden || !W_lm || !out_tokens || !out_n_accepted) return SV_ERR_ARG;
  if (h->cfg.dtype == SV_FP8 && (!tr.h_scale || !tr.w_scale)) return SV_ERR_ARG;
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return SV_ERR_ARG;
  const sv::Dims &D = h->dims;
  const bool greedy = temperature == 0.0f;
  if (D.K > 0 && !draft_tokens) return SV_ERR_ARG;
  // q_logits == NULL: point-mass drafts (q = the proposed token with
  // certainty); a -1 draft token then ends that sequence's draft
  if (!greedy && !uniforms) return SV_ERR_ARG;
  const void *ptrs[] = {hidden, W_lm, draft_tokens, q_logits, uniforms, out_tokens,
                        out_n_accepted};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SV_ERR_ALIGN;

  cudaStream_t st = h->stream;
  const unsigned epoch = ++h->epoch;
  // Fast tail: the contraction (drain mode) leaves per-CTA row statistics
  // and the draft logits at the draft tokens, and one CTA per sequence
  // decides from them.  Truncated rows, greedy and tree verification keep
  // the per-row path.
  const bool fast = h->w.rowpart != nullptr && !greedy && !tr.p_cut && !tr.q_cut &&
                    !tr.parents && h->plan.grid <= 256;
  const float inv_t = greedy ? 1.0f : static_cast<float>(1.0 / static_cast<double>(temperature));
  cudaError_t e = cudaSuccess;

  int ti = -1;
  if (h->timing) {
    if (h->timed >= kTimingRing) fold_timing(h, h->timed - kTimingRing + 1);
    ti = static_cast<int>(h->timed % kTimingRing);
    if (cudaEventRecord(h->ev0[ti], st) != cudaSuccess) return SV_ERR_CUDA;
  }

  if (h->cfg.dtype != SV_FP32) {
    const sv::TcPlan &pl = h->plan;
    const int elt = static_cast<int>(esize(h->cfg.dtype));
    if (h->tmW_ptr != W_lm) {
      if (encode_w(&h->tmW, W_lm, D.d, D.V, sv::kTileM, pl.chunks, elt) != SV_OK)
        return SV_ERR_CUDA;
      h->tmW_ptr = W_lm;
    }
    if (h->tmH_ptr != hidden) {
      if (encode_w(&h->tmH, hidden, D.d, D.R, static_cast<uint32_t>(pl.h_box_rows), pl.chunks,
                   elt) != SV_OK)
        return SV_ERR_CUDA;
      h->tmH_ptr = hidden;
    }
    sv::TcParams P{};
    P.dims = D;
    P.w = h->w;
    P.q_logits = q_logits;
    P.inv_t = inv_t;
    P.greedy = greedy ? 1 : 0;
    P.npad = pl.npad;
    P.nkb = pl.nkb;
    P.kbk = pl.kbk;
    P.fp8 = h->cfg.dtype == SV_FP8 ? 1 : 0;
    P.h_scale = tr.h_scale;
    P.w_scale = tr.w_scale;
    P.chunks = pl.chunks;
    P.stages = pl.stages;
    P.stage_bytes = pl.stage_bytes;
    P.h_boxes = pl.h_boxes;
    P.h_box_rows = pl.h_box_rows;
    P.nslot = pl.nslot;
    P.nbuf = pl.nbuf;
    P.half = pl.half;
    P.tma_logits = h->tma_logits ? 1 : 0;
    P.tmem_cols = pl.tmem_cols;
    P.wait_limit_ns = h->wait_limit_ns;
    P.epoch = epoch;
    P.row_stats = fast ? 1 : 0;
    P.H = hidden;
    P.W = W_lm;
    P.draft = draft_tokens;
    e = sv::launch_tc(pl, P, h->tmW, h->tmH, h->tmL, st);
  } else {
    sv::SimtParams P{};
    P.dims = D;
    P.w = h->w;
    P.H = static_cast<const float *>(hidden);
    P.W = static_cast<const float *>(W_lm);
    P.q_logits = q_logits;
    P.inv_t = inv_t;
    P.greedy = greedy ? 1 : 0;
    e = sv::launch_simt(P, st);
  }
  if (e != cudaSuccess) return SV_ERR_CUDA;
  if (ti >= 0) {
    if (cudaEventRecord(h->ev1[ti], st) != cudaSuccess) return SV_ERR_CUDA;
    ++h->timed;
  }

  sv::TailParams T{};
  T.dims = D;
  T.w = h->w;
  T.H = hidden;
  T.W = W_lm;
  T.dtype = h->cfg.dtype;
  T.draft = draft_tokens;
  T.q_logits = q_logits;
  T.u = uniforms;
  T.T = static_cast<double>(temperature);
  T.inv_t = inv_t;
  T.greedy = greedy ? 1 : 0;
  T.out_tokens = out_tokens;
  T.out_n = out_n_accepted;
  T.epoch = epoch;
  T.wait_limit_ns = h->wait_limit_ns;
  T.split_cnt_n = h->num_sms * 4;
  T.draft_logits_ready = h->cfg.dtype != SV_FP32 ? 1 : 0;
  T.fast = fast ? 1 : 0;
  T.stall = h->debug_stall ? 1 : 0;
  T.grid_parts = h->plan.grid;
  // every chunk CTA of a sequence waits for the others' masses: only when
  // the whole tail grid (nchunk chunk CTAs per sequence) is resident at
  // once; staged (candidate rows in shared memory) if that still holds with
  // the staging's shared memory
  const int64_t tail_ctas = static_cast<int64_t>(D.B) * D.nchunk;
  T.coop = 0;
  T.stage_rows = 0;
  if (fast && h->stage_bytes > 0 && tail_ctas <= h->tail_resident_staged) {
    T.coop = 1;
    T.stage_rows = D.K + 1 + (q_logits ? D.K : 0);
  } else if (fast && tail_ctas <= h->tail_resident) {
    T.coop = 1;
  }
  T.h_scale = tr.h_scale;
  T.w_scale = tr.w_scale;
  T.p_cut = tr.p_cut;
  T.q_cut = tr.q_cut;
  T.parents = tr.parents;
  T.out_nodes = tr.out_nodes;
  if (tr.p_cut || tr.q_cut) {
    sv::TruncParams TP{};
    TP.dims = D;
    TP.w = h->w;
    TP.q_logits = q_logits;
    TP.inv_t = inv_t;
    TP.p_cut = tr.p_cut;
    TP.q_cut = tr.q_cut;
    TP.p_top_k = tr.p_top_k;
    TP.q_top_k = tr.q_top_k;
    TP.p_top_p = tr.p_top_p;
    TP.q_top_p = tr.q_top_p;
    if (sv::launch_trunc(TP, st) != cudaSuccess) return SV_ERR_CUDA;
  }
  if (sv::launch_tail(T, st) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace

int spec_verify_status(spec_verify_t *h) {
  if (!h) return SV_ERR_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return SV_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, h->w.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  if (code != 0) {
    // after a contraction gave up, split-tile counters may be half-used
    if (cudaMemset(h->w.status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(h->w.split_cnt, 0, sizeof(int) * h->num_sms * 4) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return SV_ERR_CUDA;
  }
  return code;
}

int spec_verify_run_host(spec_verify_t *h, const void *hidden_host, const void *W_lm,
                         const int32_t *draft_tokens_host, const float *q_logits_host,
                         const float *uniforms_host, float temperature,
                         int32_t *out_tokens_host, int32_t *out_n_accepted_host) {
  if (!h || !hidden_host || !W_lm || !out_tokens_host || !out_n_accepted_host)
    return SV_ERR_ARG;
  if (h->cfg.dtype == SV_FP8) return SV_ERR_ARG;  // no host path for the FP8 scales
  const sv::Dims &D = h->dims;
  const bool greedy = temperature == 0.0f;
  if (D.K > 0 && !draft_tokens_host) return SV_ERR_ARG;
  if (!greedy && !uniforms_host) return SV_ERR_ARG;
  cudaStream_t st = h->stream;
  const size_t es = esize(h->cfg.dtype);
  if (cudaMemcpyAsync(h->st_hidden, hidden_host, static_cast<size_t>(D.R) * D.d * es,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (D.K > 0 && cudaMemcpyAsync(h->st_draft, draft_tokens_host, sizeof(int32_t) * D.RQ,
                                 cudaMemcpyHostToDevice, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (!greedy) {
    if (D.K > 0 && q_logits_host &&
        cudaMemcpyAsync(h->st_q, q_logits_host, sizeof(float) * static_cast<size_t>(D.RQ) * D.V,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return SV_ERR_CUDA;
    if (cudaMemcpyAsync(h->st_u, uniforms_host, sizeof(float) * D.R, cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
      return SV_ERR_CUDA;
  }
  // the staging q buffer stands in for the caller's only if one was given
  // (no q_logits: point-mass drafts; at T == 0 q is not read)
  int rc = spec_verify_run(h, h->st_hidden, W_lm, D.K > 0 ? h->st_draft : nullptr,
                           q_logits_host ? h->st_q : nullptr, greedy ? nullptr : h->st_u,
                           temperature, h->st_tokens, h->st_n);
  if (rc != SV_OK) return rc;
  if (cudaMemcpyAsync(out_tokens_host, h->st_tokens, sizeof(int32_t) * D.R,
                      cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(out_n_accepted_host, h->st_n, sizeof(int32_t) * D.B,
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, h->w.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  return code == 0 ? SV_OK : spec_verify_status(h);
}

namespace {

// Staging buffers, pinned status words, events and the two copy streams of
// the double-buffered host rounds (first use only).
int pipe_setup(spec_verify_t *h) {
  if (h->pipe_ready) return SV_OK;
  const sv::Dims &D = h->dims;
  const size_t es = esize(h->cfg.dtype);
  bool ok = cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (auto &sl : h->slot) {
    ok = ok && dalloc(reinterpret_cast<uint8_t **>(&sl.hidden), static_cast<size_t>(D.R) * D.d * es) &&
         dalloc(&sl.draft, static_cast<size_t>(D.RQ)) &&
         dalloc(&sl.q, static_cast<size_t>(D.RQ) * D.V) && dalloc(&sl.u, D.R) &&
         dalloc(&sl.tokens, D.R) && dalloc(&sl.n, D.B) &&
         cudaMallocHost(reinterpret_cast<void **>(&sl.status_host), sizeof(int)) == cudaSuccess &&
         cudaEventCreateWithFlags(&sl.copied, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&sl.kernels, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) return SV_ERR_CUDA;
  h->pipe_ready = true;
  return SV_OK;
}

}  // namespace

int spec_verify_submit_host(spec_verify_t *h, int slot, const void *hidden_host,
                            const void *W_lm, const int32_t *draft_tokens_host,
                            const float *q_logits_host, const float *uniforms_host,
                            float temperature, int32_t *out_tokens_host,
                            int32_t *out_n_accepted_host) {
  if (!h || slot < 0 || slot > 1 || !hidden_host || !W_lm || !out_tokens_host ||
      !out_n_accepted_host)
    return SV_ERR_ARG;
  if (h->cfg.dtype == SV_FP8) return SV_ERR_ARG;  // no host path for the FP8 scales
  const sv::Dims &D = h->dims;
  const bool greedy = temperature == 0.0f;
  if (D.K > 0 && !draft_tokens_host) return SV_ERR_ARG;
  if (!greedy && !uniforms_host) return SV_ERR_ARG;
  if (int rc = pipe_setup(h)) return rc;
  auto &sl = h->slot[slot];
  if (sl.busy) return SV_ERR_ARG;  // wait for this slot's previous round first
  const size_t es = esize(h->cfg.dtype);
  // inputs: on the host-to-device stream, free to overlap the other slot's kernels
  if (cudaMemcpyAsync(sl.hidden, hidden_host, static_cast<size_t>(D.R) * D.d * es,
                      cudaMemcpyHostToDevice, h->h2d) != cudaSuccess ||
      (D.K > 0 && cudaMemcpyAsync(sl.draft, draft_tokens_host, sizeof(int32_t) * D.RQ,
                                  cudaMemcpyHostToDevice, h->h2d) != cudaSuccess) ||
      (!greedy && D.K > 0 && q_logits_host &&
       cudaMemcpyAsync(sl.q, q_logits_host, sizeof(float) * static_cast<size_t>(D.RQ) * D.V,
                       cudaMemcpyHostToDevice, h->h2d) != cudaSuccess) ||
      (!greedy && cudaMemcpyAsync(sl.u, uniforms_host, sizeof(float) * D.R,
                                  cudaMemcpyHostToDevice, h->h2d) != cudaSuccess) ||
      cudaEventRecord(sl.copied, h->h2d) != cudaSuccess ||
      cudaStreamWaitEvent(h->stream, sl.copied, 0) != cudaSuccess)
    return SV_ERR_CUDA;
  // the step, on the handle's stream (kernels only)
  const int rc = spec_verify_run(h, sl.hidden, W_lm, D.K > 0 ? sl.draft : nullptr,
                                 q_logits_host ? sl.q : nullptr, greedy ? nullptr : sl.u,
                                 temperature, sl.tokens, sl.n);
  if (rc != SV_OK) return rc;
  // outputs and the status word: on the device-to-host stream
  if (cudaEventRecord(sl.kernels, h->stream) != cudaSuccess ||
      cudaStreamWaitEvent(h->d2h, sl.kernels, 0) != cudaSuccess ||
      cudaMemcpyAsync(out_tokens_host, sl.tokens, sizeof(int32_t) * D.R, cudaMemcpyDeviceToHost,
                      h->d2h) != cudaSuccess ||
      cudaMemcpyAsync(out_n_accepted_host, sl.n, sizeof(int32_t) * D.B, cudaMemcpyDeviceToHost,
                      h->d2h) != cudaSuccess ||
      cudaMemcpyAsync(sl.status_host, h->w.status, sizeof(int), cudaMemcpyDeviceToHost,
                      h->d2h) != cudaSuccess ||
      cudaEventRecord(sl.done, h->d2h) != cudaSuccess)
    return SV_ERR_CUDA;
  sl.busy = true;
  return SV_OK;
}

int spec_verify_wait_host(spec_verify_t *h, int slot) {
  if (!h || slot < 0 || slot > 1 || !h->pipe_ready || !h->slot[slot].busy) return SV_ERR_ARG;
  auto &sl = h->slot[slot];
  sl.busy = false;
  if (cudaEventSynchronize(sl.done) != cudaSuccess) return SV_ERR_CUDA;
  // a device-side error: read and clear the status word (synchronises)
  return *sl.status_host == 0 ? SV_OK : spec_verify_status(h);
}

int spec_verify_debug_logits(spec_verify_t *h, float *dst) {
  if (!h || !dst) return SV_ERR_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return SV_ERR_CUDA;
  const size_t n = static_cast<size_t>(h->dims.R) * h->dims.V;
  return cudaMemcpy(dst, h->w.logits, n * sizeof(float), cudaMemcpyDefault) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify_debug_lse(spec_verify_t *h, double *dst) {
  if (!h || !dst) return SV_ERR_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return SV_ERR_CUDA;
  const size_t n = static_cast<size_t>(h->dims.R + h->dims.RQ);
  std::vector<float> m(n);
  std::vector<float2> s(n);
  std::vector<double> lse(n);
  if (cudaMemcpy(m.data(), h->w.row_m, n * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(s.data(), h->w.row_s, n * sizeof(float2), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SV_ERR_CUDA;
  for (size_t i = 0; i < n; ++i)
    lse[i] = static_cast<double>(m[i]) +
             std::log(static_cast<double>(s[i].x) + static_cast<double>(s[i].y));
  return cudaMemcpy(dst, lse.data(), n * sizeof(double), cudaMemcpyDefault) == cudaSuccess
             ? SV_OK
             : SV_ERR_CUDA;
}

int spec_verify_debug_stall(spec_verify_t *h, int enable) {
  if (!h) return SV_ERR_ARG;
  h->debug_stall = enable != 0;
  return SV_OK;
}

int spec_verify_timing(spec_verify_t *h, int enable) {
  if (!h) return SV_ERR_ARG;
  if (enable && h->ev0.empty()) {
    h->ev0.resize(kTimingRing);
    h->ev1.resize(kTimingRing);
    for (int i = 0; i < kTimingRing; ++i)
      if (cudaEventCreate(&h->ev0[i]) != cudaSuccess || cudaEventCreate(&h->ev1[i]) != cudaSuccess)
        return SV_ERR_CUDA;
  }
  if (h->timing) fold_timing(h, h->timed);
  h->timing = enable != 0;
  h->timed = 0;
  h->folded = 0;
  h->timed_ms = 0.0;
  return SV_OK;
}

int spec_verify_timing_read(spec_verify_t *h, double *total_ms, int64_t *launches) {
  if (!h || !total_ms || !launches) return SV_ERR_ARG;
  if (h->timed > 0) fold_timing(h, h->timed);
  *total_ms = h->timed_ms;
  *launches = h->timed;
  return SV_OK;
}

}  // extern "C"
