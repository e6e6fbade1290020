// sv_noalloc.cu -- the verify step for callers that cannot allocate device
// memory when they call in: a serving runtime that plans every device
// buffer ahead of time and forbids cudaMalloc at run time (cudaMalloc can
// synchronise the whole device and fragments a caching allocator), or a
// plugin host that hands the library nothing but its input and output
// pointers.  Instead of a handle with its own workspace, this entry point
// keeps its scratch in one file-scope device array of fixed size that every
// GPU which loads the library holds until the process exits.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "sv_internal.cuh"
#include "sv_kernels.h"

namespace {

// Largest scratch one call may use.  The Llama-8B-shaped step (V = 128256,
// d = 4096, B = 1, K = 4) needs about 5.5 MiB of it.
constexpr size_t kArenaBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_arena[kArenaBytes];

// Device address of g_arena per device.  Host code must not pass &g_arena:
// on the host that name is only a stand-in for the device symbol.
void *g_arena_ptr[kMaxDevices] = {};
std::mutex g_arena_mu;

int arena_address(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_arena_mu);
  if (!g_arena_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_arena) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_arena_ptr[dev] = p;
  }
  *out = g_arena_ptr[dev];
  return SV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Carves the arena in 256-byte steps; returns false if it does not fit.
struct Carver {
  unsigned char *base;
  size_t off = 0;
  bool ok = true;
  template <typename T>
  T *take(size_t count) {
    if (count == 0) count = 1;
    const size_t bytes = ((count * sizeof(T)) + 255) & ~size_t(255);
    if (off + bytes > kArenaBytes) {
      ok = false;
      return nullptr;
    }
    T *p = reinterpret_cast<T *>(base + off);
    off += bytes;
    return p;
  }
};

// cuTensorMapEncodeTiled from the driver, looked up once per process (a
// function-local static: its initialisation is thread-safe).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_local() {
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

int encode_w_local(CUtensorMap *map, const void *ptr, int64_t inner, int64_t outer,
                   uint32_t box_rows, int chunks) {
  const auto fn = encode_fn_local();
  if (!fn) return SV_ERR_CUDA;
  CUresult r;
  if (chunks > 1) {  // same 3-D view as the handle path
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(outer), static_cast<cuuint64_t>(inner / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, 128};
    cuuint32_t box[3] = {64, box_rows, static_cast<cuuint32_t>(chunks)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? SV_OK : SV_ERR_CUDA;
}

// TMA store map of the fp32 logits scratch (same box as the handle path).
int encode_logits_local(CUtensorMap *map, float *base, int64_t V, int64_t R) {
  const auto fn = encode_fn_local();
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

}  // namespace

extern "C" int spec_verify_run_noalloc(const sv_config_t *cfg, const void *hidden,
                                       const void *W_lm, const int32_t *draft_tokens,
                                       const float *q_logits, const float *uniforms,
                                       float temperature, int32_t *out_tokens,
                                       int32_t *out_n_accepted) {
  if (!cfg || !hidden || !W_lm || !out_tokens || !out_n_accepted) return SV_ERR_ARG;
  if (cfg->dtype != SV_BF16 && cfg->dtype != SV_FP32) return SV_ERR_ARG;
  if (!(temperature >= 0.0f) || !std::isfinite(temperature)) return SV_ERR_ARG;
  if (cfg->V < 1 || cfg->V > INT32_MAX || cfg->d < 1 || cfg->d > (1 << 20) || cfg->B < 1 ||
      cfg->B > SV_MAX_B || cfg->K < 0 || cfg->K > SV_MAX_K)
    return SV_ERR_SHAPE;
  if (cfg->d % (cfg->dtype == SV_BF16 ? 8 : 4) != 0) return SV_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(cfg->B) * (cfg->K + 1);
  if (cfg->dtype == SV_BF16 && R > SV_MAX_ROWS_BF16) return SV_ERR_SHAPE;
  const bool greedy = temperature == 0.0f;
  if (cfg->K > 0 && !draft_tokens) return SV_ERR_ARG;
  if (!greedy && !uniforms) return SV_ERR_ARG;  // q_logits == NULL: point-mass drafts
  const void *ptrs[] = {hidden, W_lm, draft_tokens, q_logits, uniforms, out_tokens,
                        out_n_accepted};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SV_ERR_ALIGN;

  int dev = 0, major = 0, minor = 0, sms = 0, smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SV_ERR_CUDA;
  if (major != 10 || minor != 3) return SV_ERR_ARCH;
  void *arena = nullptr;
  if (int rc = arena_address(dev, &arena)) return rc;

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
  sv::TcPlan plan{};
  if (cfg->dtype == SV_BF16) {
    plan = sv::plan_tc(D, sms, smem, 2);
    if (!plan.valid) return SV_ERR_SHAPE;
  }

  // Carve the arena: the words that must start at zero first, in one block.
  Carver c{static_cast<unsigned char *>(arena)};
  sv::Work w{};
  w.split_cnt = c.take<int>(static_cast<size_t>(sms) * 4);
  w.status = c.take<int>(1);
  w.abort_epoch = c.take<unsigned>(1);
  w.ticket = c.take<unsigned>(1);
  w.finished = c.take<unsigned>(1);
  w.row_count = c.take<int>(D.B);
  w.chunk_count = c.take<int>(D.B);
  w.seq_flag = c.take<unsigned>(D.B);
  w.seq_final = c.take<int>(D.B);
  w.chunk_done = c.take<int>(D.B);
  const size_t zero_bytes = c.off;
  w.logits = c.take<float>(static_cast<size_t>(R) * D.V);
  w.part_p = c.take<float2>(static_cast<size_t>(R) * D.nsub);
  w.part_q = c.take<float2>(static_cast<size_t>(D.RQ) * D.nsub);
  w.row_m = c.take<float>(static_cast<size_t>(R + D.RQ));
  w.row_s = c.take<float2>(static_cast<size_t>(R + D.RQ));
  w.seq = c.take<sv::SeqState>(D.B);
  w.chunk_mass = c.take<float2>(2 * static_cast<size_t>(D.B) * D.nchunk);
  w.cand = c.take<int>(static_cast<size_t>(R) * (1 + sv::kMaxCand));
  w.draft_logit = c.take<float2>(static_cast<size_t>(D.RQ));
  w.draft_q = c.take<float>(static_cast<size_t>(D.RQ));
  // per-CTA row statistics of the drain-mode contraction (fast tail)
  const bool fast = cfg->dtype == SV_BF16 && plan.ncol != 0 && !greedy && plan.grid <= 256;
  w.rowpart = fast ? c.take<float4>(static_cast<size_t>(R + D.RQ) * plan.grid) : nullptr;
  w.split_buf = c.take<float>(cfg->dtype == SV_BF16
                                  ? static_cast<size_t>(plan.grid) * 2 * sv::kTileM * plan.npad
                                  : 1);
  if (!c.ok) return SV_ERR_SHAPE;

  cudaStream_t st = static_cast<cudaStream_t>(cfg->stream);
  // The array keeps the previous call's contents: clear the counters, flags
  // and status word this call relies on starting at zero.
  if (cudaMemsetAsync(arena, 0, zero_bytes, st) != cudaSuccess) return SV_ERR_CUDA;
  // chunk masses start unset (all-ones bits): the cooperative selection waits for them
  if (cudaMemsetAsync(w.chunk_mass, 0xFF, sizeof(float2) * D.B * D.nchunk, st) != cudaSuccess)
    return SV_ERR_CUDA;

  const unsigned epoch = 1;  // flags were just cleared to 0
  const uint64_t wait_limit_ns = 1000000000ull;
  const float inv_t = greedy ? 1.0f : static_cast<float>(1.0 / static_cast<double>(temperature));
  cudaError_t e;
  if (cfg->dtype == SV_BF16) {
    CUtensorMap tmW, tmH, tmL{};
    const bool tma_logits = D.V % 4 == 0;
    if (encode_w_local(&tmW, W_lm, D.d, D.V, sv::kTileM, plan.chunks) != SV_OK ||
        encode_w_local(&tmH, hidden, D.d, D.R, static_cast<uint32_t>(plan.h_box_rows),
                       plan.chunks) != SV_OK ||
        (tma_logits && encode_logits_local(&tmL, w.logits, D.V, R) != SV_OK))
      return SV_ERR_CUDA;
    sv::TcParams P{};
    P.dims = D;
    P.w = w;
    P.q_logits = q_logits;
    P.inv_t = inv_t;
    P.greedy = greedy ? 1 : 0;
    P.npad = plan.npad;
    P.nkb = plan.nkb;
    P.kbk = plan.kbk;
    P.chunks = plan.chunks;
    P.stages = plan.stages;
    P.stage_bytes = plan.stage_bytes;
    P.h_boxes = plan.h_boxes;
    P.h_box_rows = plan.h_box_rows;
    P.nslot = plan.nslot;
    P.nbuf = plan.nbuf;
    P.half = plan.half;
    P.tma_logits = tma_logits ? 1 : 0;
    P.tmem_cols = plan.tmem_cols;
    P.wait_limit_ns = wait_limit_ns;
    P.epoch = epoch;
    P.row_stats = fast ? 1 : 0;
    P.H = hidden;
    P.W = W_lm;
    P.draft = draft_tokens;
    e = sv::launch_tc(plan, P, tmW, tmH, tmL, st);
  } else {
    sv::SimtParams P{};
    P.dims = D;
    P.w = w;
    P.H = static_cast<const float *>(hidden);
    P.W = static_cast<const float *>(W_lm);
    P.q_logits = q_logits;
    P.inv_t = inv_t;
    P.greedy = greedy ? 1 : 0;
    e = sv::launch_simt(P, st);
  }
  if (e != cudaSuccess) return SV_ERR_CUDA;
  sv::TailParams T{};
  T.dims = D;
  T.w = w;
  T.H = hidden;
  T.W = W_lm;
  T.dtype = cfg->dtype;
  T.draft = draft_tokens;
  T.q_logits = q_logits;
  T.u = uniforms;
  T.T = static_cast<double>(temperature);
  T.inv_t = inv_t;
  T.greedy = greedy ? 1 : 0;
  T.out_tokens = out_tokens;
  T.out_n = out_n_accepted;
  T.epoch = epoch;
  T.wait_limit_ns = wait_limit_ns;
  T.split_cnt_n = sms * 4;
  T.draft_logits_ready = cfg->dtype == SV_BF16 ? 1 : 0;
  T.fast = fast ? 1 : 0;
  T.grid_parts = plan.grid;
  const int64_t tail_ctas = static_cast<int64_t>(D.B) * D.nchunk;
  const int stage_bytes = fast ? sv::tail_stage_bytes(D, true) : 0;
  T.coop = 0;
  T.stage_rows = 0;
  if (stage_bytes > 0 && tail_ctas <= sv::tail_resident_ctas(sms, stage_bytes)) {
    T.coop = 1;
    T.stage_rows = D.K + 1 + (q_logits ? D.K : 0);
  } else if (fast && tail_ctas <= sv::tail_resident_ctas(sms, 0)) {
    T.coop = 1;
  }
  return sv::launch_tail(T, st) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
