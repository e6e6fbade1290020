"""Python binding of the GB300 verify-and-sample library (libspec_verify.so).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels behind the C ABI of ``include/spec_verify.h``; the functions here
carry the same names as the C entry points, take torch tensors (device
memory) and pass their pointers and the current CUDA stream through.
There is no fallback: if the library has not been built, importing the
entry points raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspec_verify.so")

SV_OK = 0
SV_ERR_ARG = -1
SV_ERR_ALIGN = -2
SV_ERR_SHAPE = -3
SV_ERR_CUDA = -4
SV_ERR_ARCH = -5
SV_ERR_TIMEOUT = -6
SV_ERR_TOKEN = -7
SV_ERR_NONFINITE = -8
SV_BF16 = 0
SV_FP32 = 1
SV_FP8 = 2
SV_MAX_K = 64
SV_MAX_B = 4096
SV_MAX_ROWS_BF16 = 384
SV_NGRAM_MAX = 16

# every symbol of include/spec_verify.h
EXPORTS = ("spec_verify_create", "spec_verify_run", "spec_verify_run_host",
           "spec_verify_status", "spec_verify_set_stream",
           "spec_verify_debug_logits", "spec_verify_debug_lse",
           "spec_verify_set_wait_limit", "spec_verify_timing",
           "spec_verify_timing_read", "spec_verify_launches_per_run",
           "spec_verify_strerror", "spec_verify_destroy",
           "spec_verify_run_noalloc", "spec_ngram_draft", "spec_verify_run_truncated",
           "spec_verify_tree_greedy", "spec_verify_run_fp8", "spec_verify_plan",
           "spec_verify_debug_stall", "spec_verify_submit_host", "spec_verify_wait_host")


class sv_plan_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "npad", "drain_cols", "half", "kblock_elems", "kblocks", "chunks", "stages",
        "stage_bytes", "smem_bytes", "grid", "tmem_cols", "tmem_buffers", "tmem_slots")]


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {spec_verify_strerror(code)} ({code})")
        self.code = code


class sv_config_t(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int64), ("d", ctypes.c_int64),
                ("B", ctypes.c_int32), ("K", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("stream", ctypes.c_void_p)]


_lib = None


def load_library():
    """Loads the in-tree CUDA library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(or python -m speculative_decoding_verification_22_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_float)
        lib.spec_verify_create.argtypes = [ctypes.POINTER(sv_config_t),
                                           ctypes.POINTER(vp)]
        lib.spec_verify_run.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp]
        lib.spec_verify_run_host.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp]
        lib.spec_verify_status.argtypes = [vp]
        lib.spec_verify_set_stream.argtypes = [vp, vp]
        lib.spec_verify_debug_logits.argtypes = [vp, vp]
        lib.spec_verify_debug_lse.argtypes = [vp, vp]
        lib.spec_verify_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
        lib.spec_verify_debug_stall.argtypes = [vp, ctypes.c_int]
        lib.spec_verify_submit_host.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, vp, f32, vp,
                                                vp]
        lib.spec_verify_wait_host.argtypes = [vp, ctypes.c_int]
        lib.spec_verify_timing.argtypes = [vp, ctypes.c_int]
        lib.spec_verify_timing_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double),
                                                ctypes.POINTER(i64)]
        lib.spec_verify_launches_per_run.argtypes = [vp, f32]
        lib.spec_verify_strerror.argtypes = [ctypes.c_int]
        lib.spec_verify_strerror.restype = ctypes.c_char_p
        lib.spec_verify_destroy.argtypes = [vp]
        lib.spec_verify_destroy.restype = None
        lib.spec_verify_run_noalloc.argtypes = [ctypes.POINTER(sv_config_t), vp, vp, vp, vp,
                                                vp, f32, vp, vp]
        i32 = ctypes.c_int32
        lib.spec_verify_run_truncated.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, f32, i32,
                                                  f32, vp, vp]
        lib.spec_verify_tree_greedy.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        lib.spec_verify_run_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp]
        lib.spec_ngram_draft.argtypes = [vp, ctypes.c_int64, vp, i32, i32, i32, i32, vp, vp,
                                         vp]
        lib.spec_verify_plan.argtypes = [ctypes.POINTER(sv_config_t), i32, i32,
                                         ctypes.POINTER(sv_plan_t)]
        for name in EXPORTS:
            if name not in ("spec_verify_strerror", "spec_verify_destroy"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(code: int, what: str):
    if code != SV_OK:
        raise SpecVerifyError(code, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def spec_verify_strerror(code: int) -> str:
    return load_library().spec_verify_strerror(int(code)).decode()


def spec_verify_plan(V: int, d: int, B: int, K: int, dtype="bf16", num_sms: int = 152,
                     smem_optin: int = 232448) -> dict:
    """The contraction's launch plan for a shape (host arithmetic, no GPU):
    accumulation mode, pipeline stages, shared and tensor memory layout."""
    code = {"bf16": SV_BF16, "fp8": SV_FP8}.get(dtype, dtype)
    cfg = sv_config_t(V, d, B, K, code, None)
    out = sv_plan_t()
    _check(load_library().spec_verify_plan(ctypes.byref(cfg), num_sms, smem_optin,
                                           ctypes.byref(out)), "spec_verify_plan")
    return {n: getattr(out, n) for n, _ in sv_plan_t._fields_}


def spec_verify_create(V: int, d: int, B: int, K: int, dtype="bf16", stream=None):
    """Creates a handle; ``dtype`` is "bf16"/"fp32" (or SV_BF16/SV_FP32)."""
    code = {"bf16": SV_BF16, "fp32": SV_FP32, "fp8": SV_FP8}.get(dtype, dtype)
    cfg = sv_config_t(int(V), int(d), int(B), int(K), int(code),
                      _stream_handle(stream))
    h = ctypes.c_void_p()
    _check(load_library().spec_verify_create(ctypes.byref(cfg), ctypes.byref(h)),
           "spec_verify_create")
    return h


def spec_verify_run(h, hidden, W_lm, draft_tokens, q_logits, uniforms,
                    temperature: float, out_tokens, out_n_accepted) -> None:
    _check(load_library().spec_verify_run(
        h, _ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(q_logits),
        _ptr(uniforms), float(temperature), _ptr(out_tokens),
        _ptr(out_n_accepted)), "spec_verify_run")


def spec_verify_run_host(h, hidden, W_lm, draft_tokens, q_logits, uniforms,
                         temperature: float, out_tokens, out_n_accepted) -> None:
    """Host-buffer variant: hidden/draft/q/uniforms/outputs are host
    (preferably pinned) tensors, W_lm a device tensor; returns after the
    outputs have been copied back."""
    _check(load_library().spec_verify_run_host(
        h, _ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(q_logits),
        _ptr(uniforms), float(temperature), _ptr(out_tokens),
        _ptr(out_n_accepted)), "spec_verify_run_host")


def spec_verify_submit_host(h, slot: int, hidden, W_lm, draft_tokens, q_logits, uniforms,
                            temperature: float, out_tokens, out_n_accepted) -> None:
    """Double-buffered host round: enqueue it in slot 0 or 1 (pinned host
    tensors for inputs and outputs, W_lm on the device) and return."""
    _check(load_library().spec_verify_submit_host(
        h, int(slot), _ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(q_logits),
        _ptr(uniforms), float(temperature), _ptr(out_tokens), _ptr(out_n_accepted)),
        "spec_verify_submit_host")


def spec_verify_wait_host(h, slot: int) -> int:
    """Waits for the round in `slot`; returns its status code."""
    return int(load_library().spec_verify_wait_host(h, int(slot)))


def spec_verify_status(h) -> int:
    return int(load_library().spec_verify_status(h))


def spec_verify_set_stream(h, stream=None) -> None:
    _check(load_library().spec_verify_set_stream(h, _stream_handle(stream)),
           "spec_verify_set_stream")


def spec_verify_debug_logits(h, dst) -> None:
    _check(load_library().spec_verify_debug_logits(h, _ptr(dst)),
           "spec_verify_debug_logits")


def spec_verify_debug_lse(h, dst) -> None:
    _check(load_library().spec_verify_debug_lse(h, _ptr(dst)),
           "spec_verify_debug_lse")


def spec_verify_set_wait_limit(h, limit_ns: int) -> None:
    _check(load_library().spec_verify_set_wait_limit(h, int(limit_ns)),
           "spec_verify_set_wait_limit")


def spec_verify_debug_stall(h, enable: bool) -> None:
    """Tests only: every run first waits for a flag nothing sets (bounded by
    the wait limit), so it reports SV_ERR_TIMEOUT and withdraws sequence 0."""
    _check(load_library().spec_verify_debug_stall(h, int(bool(enable))),
           "spec_verify_debug_stall")


def spec_verify_timing(h, enable: bool) -> None:
    _check(load_library().spec_verify_timing(h, int(bool(enable))),
           "spec_verify_timing")


def spec_verify_timing_read(h):
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    _check(load_library().spec_verify_timing_read(h, ctypes.byref(ms), ctypes.byref(n)),
           "spec_verify_timing_read")
    return ms.value, n.value


def spec_verify_launches_per_run(h, temperature: float) -> int:
    n = load_library().spec_verify_launches_per_run(h, float(temperature))
    if n < 0:
        raise SpecVerifyError(n, "spec_verify_launches_per_run")
    return n


def spec_verify_run_noalloc(V, d, B, K, dtype, hidden, W_lm, draft_tokens, q_logits,
                            uniforms, temperature: float, out_tokens, out_n_accepted,
                            stream=None) -> None:
    """The step without a handle or any allocation (scratch in a fixed
    device array inside the library); for callers that cannot allocate
    device memory at call time.  Calls that overlap on the GPU race."""
    code = {"bf16": SV_BF16, "fp32": SV_FP32, "fp8": SV_FP8}.get(dtype, dtype)
    cfg = sv_config_t(int(V), int(d), int(B), int(K), int(code), _stream_handle(stream))
    _check(load_library().spec_verify_run_noalloc(
        ctypes.byref(cfg), _ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(q_logits),
        _ptr(uniforms), float(temperature), _ptr(out_tokens), _ptr(out_n_accepted)),
        "spec_verify_run_noalloc")


def spec_verify_run_truncated(h, hidden, W_lm, draft_tokens, q_logits, uniforms,
                              temperature: float, target_top_k: int, target_top_p: float,
                              draft_top_k: int, draft_top_p: float, out_tokens,
                              out_n_accepted) -> None:
    """The step with truncated sampling (top-k, then top-p; per side)."""
    _check(load_library().spec_verify_run_truncated(
        h, _ptr(hidden), _ptr(W_lm), _ptr(draft_tokens), _ptr(q_logits), _ptr(uniforms),
        float(temperature), int(target_top_k), float(target_top_p), int(draft_top_k),
        float(draft_top_p), _ptr(out_tokens), _ptr(out_n_accepted)),
        "spec_verify_run_truncated")


def spec_verify_run_fp8(h, hidden8, hidden_scale, W8, w_scale, draft_tokens, q_logits,
                        uniforms, temperature: float, out_tokens, out_n_accepted) -> None:
    """The step with an FP8 E4M3 LM head (handle dtype "fp8")."""
    _check(load_library().spec_verify_run_fp8(
        h, _ptr(hidden8), _ptr(hidden_scale), _ptr(W8), _ptr(w_scale), _ptr(draft_tokens),
        _ptr(q_logits), _ptr(uniforms), float(temperature), _ptr(out_tokens),
        _ptr(out_n_accepted)), "spec_verify_run_fp8")


def spec_verify_tree_greedy(h, hidden, W_lm, tree_tokens, tree_parents, out_tokens,
                            out_nodes, out_n) -> None:
    """Greedy tree verification: the longest path whose tokens are the
    target's argmax choices (N = the handle's K nodes)."""
    _check(load_library().spec_verify_tree_greedy(
        h, _ptr(hidden), _ptr(W_lm), _ptr(tree_tokens), _ptr(tree_parents), _ptr(out_tokens),
        _ptr(out_nodes), _ptr(out_n)), "spec_verify_tree_greedy")


def spec_ngram_draft(tokens, lengths, K: int, n_min: int = 2, n_max: int = 5,
                     out_draft=None, out_len=None, stream=None):
    """Prompt-lookup drafts for B contexts (tokens [B, L] int32 on the GPU,
    lengths [B] int32): the up to K tokens that followed the latest earlier
    occurrence of the longest recurring suffix of n_max..n_min tokens.
    Returns (draft [B, K] with -1 after the proposal, length [B]); the
    draft feeds spec_verify_run with q_logits=None."""
    B, L = tokens.shape
    if out_draft is None:
        out_draft = torch.empty((B, K), dtype=torch.int32, device=tokens.device)
    if out_len is None:
        out_len = torch.empty((B,), dtype=torch.int32, device=tokens.device)
    _check(load_library().spec_ngram_draft(
        _ptr(tokens), int(L), _ptr(lengths), int(B), int(K), int(n_min), int(n_max),
        _ptr(out_draft), _ptr(out_len), _stream_handle(stream)), "spec_ngram_draft")
    return out_draft, out_len


def spec_verify_destroy(h) -> None:
    if h:
        load_library().spec_verify_destroy(h)


class SpecVerify:
    """Owns one handle; ``run`` writes tokens [B, K+1] and n_accepted [B]."""

    def __init__(self, V, d, B, K, dtype="bf16", device=None, stream=None):
        self.V, self.d, self.B, self.K, self.dtype = V, d, B, K, dtype
        self.device = torch.device("cuda" if device is None else device)
        with torch.cuda.device(self.device):
            self.h = spec_verify_create(V, d, B, K, dtype, stream)

    def run(self, hidden, W_lm, draft_tokens, q_logits, uniforms, temperature,
            out_tokens=None, out_n_accepted=None):
        if out_tokens is None:
            out_tokens = torch.empty((self.B, self.K + 1), dtype=torch.int32,
                                     device=self.device)
        if out_n_accepted is None:
            out_n_accepted = torch.empty((self.B,), dtype=torch.int32, device=self.device)
        spec_verify_run(self.h, hidden, W_lm, draft_tokens, q_logits, uniforms,
                        temperature, out_tokens, out_n_accepted)
        return out_tokens, out_n_accepted

    def run_truncated(self, hidden, W_lm, draft_tokens, q_logits, uniforms, temperature,
                      target_top_k=0, target_top_p=1.0, draft_top_k=0, draft_top_p=1.0,
                      out_tokens=None, out_n_accepted=None):
        if out_tokens is None:
            out_tokens = torch.empty((self.B, self.K + 1), dtype=torch.int32,
                                     device=self.device)
        if out_n_accepted is None:
            out_n_accepted = torch.empty((self.B,), dtype=torch.int32, device=self.device)
        spec_verify_run_truncated(self.h, hidden, W_lm, draft_tokens, q_logits, uniforms,
                                  temperature, target_top_k, target_top_p, draft_top_k,
                                  draft_top_p, out_tokens, out_n_accepted)
        return out_tokens, out_n_accepted

    def run_fp8(self, hidden8, hidden_scale, W8, w_scale, draft_tokens, q_logits, uniforms,
                temperature, out_tokens=None, out_n_accepted=None):
        if out_tokens is None:
            out_tokens = torch.empty((self.B, self.K + 1), dtype=torch.int32,
                                     device=self.device)
        if out_n_accepted is None:
            out_n_accepted = torch.empty((self.B,), dtype=torch.int32, device=self.device)
        spec_verify_run_fp8(self.h, hidden8, hidden_scale, W8, w_scale, draft_tokens, q_logits,
                            uniforms, temperature, out_tokens, out_n_accepted)
        return out_tokens, out_n_accepted

    def run_tree_greedy(self, hidden, W_lm, tree_tokens, tree_parents):
        """Returns (tokens [B, N+1], nodes [B, N], n [B])."""
        out_t = torch.empty((self.B, self.K + 1), dtype=torch.int32, device=self.device)
        out_nodes = torch.empty((self.B, max(self.K, 1)), dtype=torch.int32, device=self.device)
        out_n = torch.empty((self.B,), dtype=torch.int32, device=self.device)
        spec_verify_tree_greedy(self.h, hidden, W_lm, tree_tokens, tree_parents, out_t,
                                out_nodes, out_n)
        return out_t, out_nodes[:, :self.K], out_n

    def status(self) -> int:
        return spec_verify_status(self.h)

    def logits(self):
        out = torch.empty((self.B * (self.K + 1), self.V), dtype=torch.float32,
                          device=self.device)
        spec_verify_debug_logits(self.h, out)
        return out

    def lse(self):
        out = torch.empty((self.B * (self.K + 1) + self.B * self.K,), dtype=torch.float64,
                          device=self.device)
        spec_verify_debug_lse(self.h, out)
        return out

    def close(self):
        if getattr(self, "h", None):
            spec_verify_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
