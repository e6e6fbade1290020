"""Oracle for the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product (``speculative_decoding_verification_22_gb300``) never imports it,
and this package never imports the product.

The arithmetic lives in ``sv_oracle.c`` (plain C, fp64, one thread; built
with ``-O2 -ffp-contract=off`` and no fast-math).  This module only marshals
numpy arrays into it, plus two closed forms from the pages:

* ``expected_tokens(alpha, K)`` -- "Speculative Decoding: Two Models, One
  Voice", "How much faster" and Tool 2: with i.i.d. acceptance alpha, a round
  emits (1 - alpha^(K+1)) / (1 - alpha) tokens on average.
* ``expected_tokens_positions(alphas)`` -- "Speculative Decoding: The Algebra
  and the Proof", "The algebra": with conditional acceptance alpha_j at
  position j, E = 1 + sum_i prod_{j<=i} alpha_j.

Every C function is described (with its source passages) in ``sv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB = os.path.join(_HERE, "libsv_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EARG, ETOKEN, ENOMEM = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libsv_oracle.so`` (gcc, fp64, no
    fast-math, no FMA contraction so x86 and Arm round identically)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, vp, dbl = (ctypes.c_int64, ctypes.c_int32,
                                 ctypes.c_void_p, ctypes.c_double)
            lib.sv_oracle_logits.argtypes = [i64, i64, i64, i32, vp, vp, i64,
                                             i64, vp]
            lib.sv_oracle_logits.restype = ctypes.c_int
            lib.sv_oracle_lse.argtypes = [i64, vp, dbl]
            lib.sv_oracle_lse.restype = dbl
            lib.sv_oracle_softmax.argtypes = [i64, vp, dbl, vp]
            lib.sv_oracle_softmax.restype = None
            lib.sv_oracle_verify.argtypes = [i64, i64, i32, i32, i32, vp, vp,
                                             vp, vp, vp, dbl, vp, vp, vp, vp,
                                             vp, vp, vp, vp]
            lib.sv_oracle_verify.restype = ctypes.c_int
            lib.sv_oracle_rule_batch.argtypes = [i64, i32, vp, vp, i64, vp,
                                                 vp, vp, vp, vp, vp, vp]
            lib.sv_oracle_rule_batch.restype = ctypes.c_int
            lib.sv_oracle_emitted_law.argtypes = [i64, vp, vp, vp]
            lib.sv_oracle_emitted_law.restype = dbl
            lib.sv_oracle_ngram_draft.argtypes = [vp, i64, vp, i32, i32, i32,
                                                  i32, vp, vp]
            lib.sv_oracle_ngram_draft.restype = ctypes.c_int
            lib.sv_oracle_truncate.argtypes = [i64, vp, dbl, i32, dbl, vp, vp, vp, vp]
            lib.sv_oracle_truncate.restype = ctypes.c_int
            lib.sv_oracle_truncate_ex.argtypes = [i64, vp, dbl, i32, dbl, vp, vp, vp, vp, vp,
                                                  vp, vp]
            lib.sv_oracle_truncate_ex.restype = ctypes.c_int
            lib.sv_oracle_verify_truncated.argtypes = [i64, i64, i32, i32, i32, vp, vp, vp,
                                                       vp, vp, dbl, i32, dbl, i32, dbl, dbl,
                                                       dbl, vp, vp, vp, vp, vp]
            lib.sv_oracle_verify_truncated.restype = ctypes.c_int
            lib.sv_oracle_tree_greedy.argtypes = [i64, i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                                  vp, vp, vp]
            lib.sv_oracle_tree_greedy.restype = ctypes.c_int
            lib.sv_oracle_verify_fp8.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp,
                                                 vp, dbl, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.sv_oracle_verify_fp8.restype = ctypes.c_int
            lib.sv_oracle_e4m3_decode.argtypes = [i64, vp, vp]
            lib.sv_oracle_e4m3_decode.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _matrix(a):
    """bf16 matrices travel as their uint16 bit patterns (dtype code 0),
    fp32 as float32 (code 1), FP8 E4M3 as uint8 codes (code 2; logits()
    then returns the unscaled sums, see verify_fp8 for the scaled step)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 0
    if a.dtype == np.float32:
        return a, 1
    if a.dtype == np.uint8:
        return a, 2
    raise TypeError("matrices must be uint16 (bf16 bits), float32 or uint8 (E4M3)")


def logits(H, W, v0: int = 0, v1: int | None = None) -> np.ndarray:
    """fp64 logits H @ W[v0:v1].T, summed in k order (LM-head contraction)."""
    H, dt = _matrix(H)
    W, dt2 = _matrix(W)
    if dt != dt2:
        raise TypeError("H and W must share a dtype")
    R, d = H.shape
    V, d2 = W.shape
    if d != d2:
        raise ValueError("hidden size mismatch")
    v1 = V if v1 is None else v1
    out = np.empty((R, v1 - v0), dtype=np.float64)
    rc = _load().sv_oracle_logits(V, d, R, dt, _ptr(H), _ptr(W), v0, v1,
                                  _ptr(out))
    if rc != OK:
        raise ValueError(f"sv_oracle_logits failed ({rc})")
    return out


def lse(x, T: float = 1.0) -> float:
    """log-sum-exp of x / T (temperature softmax normaliser)."""
    x = _c(x, np.float64)
    return float(_load().sv_oracle_lse(x.size, _ptr(x), float(T)))


def softmax(x, T: float = 1.0) -> np.ndarray:
    """softmax(x / T) in fp64."""
    x = _c(x, np.float64)
    out = np.empty_like(x)
    _load().sv_oracle_softmax(x.size, _ptr(x), float(T), _ptr(out))
    return out


def verify(hidden, W, draft, q_logits, uniforms, temperature: float,
           want_logits: bool = False) -> dict:
    """The whole verify-and-sample step for B sequences.

    hidden [B, K+1, d] and W [V, d] as uint16 (bf16 bits) or float32;
    draft [B, K] int32; q_logits [B, K, V] float32, or None for drafts
    proposed with certainty (point-mass q; a -1 then ends a draft early);
    uniforms [B, K+1] float32.
    Returns tokens [B, K+1], n_accepted [B], dist [B] (with its two parts
    dist_accept [B], over the accept tests, and dist_draw [B], for the final
    draw), lse_p, lse_q, status and (optionally) fp64 logits [B*(K+1), V].
    """
    hidden, dt = _matrix(hidden)
    W, dt2 = _matrix(W)
    if dt != dt2:
        raise TypeError("hidden and W must share a dtype")
    B, rows, d = hidden.shape
    K = rows - 1
    V = W.shape[0]
    draft = _c(draft, np.int32).reshape(B, K)
    T = float(temperature)
    q = None if (K == 0 or q_logits is None) else _c(q_logits, np.float32).reshape(B, K, V)
    u = None if T == 0.0 else _c(uniforms, np.float32).reshape(B, rows)
    tokens = np.empty((B, rows), dtype=np.int32)
    n_acc = np.empty((B,), dtype=np.int32)
    dist = np.empty((B,), dtype=np.float64)
    dacc = np.empty((B,), dtype=np.float64)
    ddraw = np.empty((B,), dtype=np.float64)
    lg = np.empty((B * rows, V), dtype=np.float64) if want_logits else None
    lse_p = np.full((B * rows,), np.nan)
    lse_q = np.full((max(B * K, 1),), np.nan)
    rc = _load().sv_oracle_verify(V, d, B, K, dt, _ptr(hidden), _ptr(W),
                                  _ptr(draft), _ptr(q), _ptr(u), T,
                                  _ptr(tokens), _ptr(n_acc), _ptr(dist),
                                  _ptr(lg), _ptr(lse_p), _ptr(lse_q),
                                  _ptr(dacc), _ptr(ddraw))
    if rc not in (OK, ETOKEN):
        raise ValueError(f"sv_oracle_verify failed ({rc})")
    return {"tokens": tokens, "n_accepted": n_acc, "dist": dist, "dist_accept": dacc,
            "dist_draw": ddraw, "logits": lg, "lse_p": lse_p, "lse_q": lse_q[:B * K],
            "status": rc}


def rule_batch(p, q, x, u, split: bool = False):
    """The accept / residual / bonus rule for n independent rounds that
    share p [K+1, V] and q [K, V] (probabilities; None for point-mass
    drafts, where a -1 ends a draft early); x [n, K], u [n, K+1].
    Returns (tokens, n_accepted, dist), and with split=True also the two
    parts of dist (accept tests, final draw)."""
    p = _c(p, np.float64)
    K1, V = p.shape
    K = K1 - 1
    if q is not None:
        q = _c(q, np.float64).reshape(K, V) if K > 0 else np.zeros((1, V))
    x = _c(x, np.int32).reshape(-1, K) if K > 0 else np.zeros((len(u), 1), np.int32)
    u = _c(u, np.float64).reshape(-1, K1)
    n = u.shape[0]
    tokens = np.empty((n, K1), dtype=np.int32)
    n_acc = np.empty((n,), dtype=np.int32)
    dist = np.empty((n,), dtype=np.float64)
    dacc = np.empty((n,), dtype=np.float64)
    ddraw = np.empty((n,), dtype=np.float64)
    rc = _load().sv_oracle_rule_batch(V, K, _ptr(p), _ptr(q), n, _ptr(x),
                                      _ptr(u), _ptr(tokens), _ptr(n_acc),
                                      _ptr(dist), _ptr(dacc), _ptr(ddraw))
    if rc not in (OK, ETOKEN):
        raise ValueError(f"sv_oracle_rule_batch failed ({rc})")
    if split:
        return tokens, n_acc, dist, dacc, ddraw
    return tokens, n_acc, dist


def emitted_law(p, q):
    """Exact law of the token emitted at one draft position and the
    acceptance mass alpha = sum min(p, q)."""
    p = _c(p, np.float64)
    q = _c(q, np.float64)
    law = np.empty_like(p)
    alpha = _load().sv_oracle_emitted_law(p.size, _ptr(p), _ptr(q), _ptr(law))
    return law, float(alpha)


def expected_tokens(alpha: float, K: int) -> float:
    """(1 - alpha^(K+1)) / (1 - alpha); K + 1 at alpha == 1."""
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def expected_tokens_positions(alphas) -> float:
    """1 + sum_{i=1..K} prod_{j<=i} alpha_j (conditional acceptances)."""
    total, prod = 1.0, 1.0
    for a in alphas:
        prod *= float(a)
        total += prod
    return total


def ngram_draft(tokens, lengths, K: int, n_min: int = 2, n_max: int = 5):
    """Prompt-lookup drafts (reading R10 in sv_oracle.c): tokens [B, L]
    int32 contexts (row b holds lengths[b] tokens), K draft slots.
    Returns draft [B, K] (-1 after the proposal) and its length [B]."""
    tokens = _c(tokens, np.int32)
    if tokens.ndim == 1:
        tokens = tokens.reshape(1, -1)
    B, L = tokens.shape
    lengths = _c(lengths, np.int32).reshape(B)
    draft = np.empty((B, K), dtype=np.int32)
    n = np.empty((B,), dtype=np.int32)
    rc = _load().sv_oracle_ngram_draft(_ptr(tokens), L, _ptr(lengths), B, K,
                                       n_min, n_max, _ptr(draft), _ptr(n))
    if rc != OK:
        raise ValueError(f"sv_oracle_ngram_draft failed ({rc})")
    return draft, n


def truncate(logits, T: float, top_k: int = 0, top_p: float = 1.0, cut: bool = False):
    """Warped distribution of one row of logits (reading R11 in
    sv_oracle.c): temperature, top-k (0: off), then top-p (1: off), both
    cut by value with ties kept.  Returns (p, keep, gap, margin), and with
    cut=True also (cut_logit, last_kept, first_dropped): the logit of the
    last kept token in descending order, that token and the largest dropped
    one (-inf, -1, -1 when nothing is cut)."""
    x = _c(logits, np.float64)
    p = np.empty_like(x)
    keep = np.empty(x.size, dtype=np.uint8)
    gap, margin, cl = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    a0, a1 = ctypes.c_int64(), ctypes.c_int64()
    rc = _load().sv_oracle_truncate_ex(x.size, _ptr(x), float(T), int(top_k), float(top_p),
                                       _ptr(p), _ptr(keep), ctypes.byref(gap),
                                       ctypes.byref(margin), ctypes.byref(cl), ctypes.byref(a0),
                                       ctypes.byref(a1))
    if rc != OK:
        raise ValueError(f"sv_oracle_truncate failed ({rc})")
    if cut:
        return p, keep.astype(bool), gap.value, margin.value, cl.value, a0.value, a1.value
    return p, keep.astype(bool), gap.value, margin.value


def verify_truncated(hidden, W, draft, q_logits, uniforms, temperature: float,
                     p_top_k: int = 0, p_top_p: float = 1.0, q_top_k: int = 0,
                     q_top_p: float = 1.0, tol_gap: float = 0.0, tol_mass: float = 0.0) -> dict:
    """The verify step with truncated target and draft distributions (R11);
    arguments as verify().  Adds trunc_sens [B] (the largest warped mass of
    a token next to a cut within tol_gap / tol_mass of flipping) and
    trunc_xgap [B] (the smallest logit change that moves a draft token
    across its row's cut), see sv_oracle.c."""
    hidden, dt = _matrix(hidden)
    W, dt2 = _matrix(W)
    if dt != dt2:
        raise TypeError("hidden and W must share a dtype")
    B, rows, d = hidden.shape
    K = rows - 1
    V = W.shape[0]
    draft = _c(draft, np.int32).reshape(B, K)
    T = float(temperature)
    q = None if (K == 0 or q_logits is None) else _c(q_logits, np.float32).reshape(B, K, V)
    u = None if T == 0.0 else _c(uniforms, np.float32).reshape(B, rows)
    tokens = np.empty((B, rows), dtype=np.int32)
    n_acc = np.empty((B,), dtype=np.int32)
    dist = np.empty((B,), dtype=np.float64)
    sens = np.zeros((B,))
    xgap = np.full((B,), np.inf)
    rc = _load().sv_oracle_verify_truncated(V, d, B, K, dt, _ptr(hidden), _ptr(W), _ptr(draft),
                                            _ptr(q), _ptr(u), T, int(p_top_k), float(p_top_p),
                                            int(q_top_k), float(q_top_p), float(tol_gap),
                                            float(tol_mass), _ptr(tokens), _ptr(n_acc),
                                            _ptr(dist), _ptr(sens), _ptr(xgap))
    if rc not in (OK, ETOKEN):
        raise ValueError(f"sv_oracle_verify_truncated failed ({rc})")
    return {"tokens": tokens, "n_accepted": n_acc, "dist": dist, "trunc_sens": sens,
            "trunc_xgap": xgap, "status": rc}


def tree_greedy(hidden, W, tokens, parents) -> dict:
    """Greedy tree verification (reading R12 in sv_oracle.c): hidden
    [B, N+1, d], W [V, d] (uint16 bf16 bits or float32), tokens / parents
    [B, N] int32 (parents in [-1, j)).  Returns tokens [B, N+1], nodes
    [B, N] (the accepted path's node indices), n [B] and gap [B]."""
    hidden, dt = _matrix(hidden)
    W, dt2 = _matrix(W)
    if dt != dt2:
        raise TypeError("hidden and W must share a dtype")
    B, rows, d = hidden.shape
    N = rows - 1
    V = W.shape[0]
    tokens = _c(tokens, np.int32).reshape(B, N)
    parents = _c(parents, np.int32).reshape(B, N)
    out_t = np.empty((B, rows), dtype=np.int32)
    out_nodes = np.empty((B, max(N, 1)), dtype=np.int32)
    out_n = np.empty((B,), dtype=np.int32)
    gap = np.empty((B,), dtype=np.float64)
    rc = _load().sv_oracle_tree_greedy(V, d, B, N, dt, _ptr(hidden), _ptr(W), _ptr(tokens),
                                       _ptr(parents), _ptr(out_t), _ptr(out_nodes),
                                       _ptr(out_n), _ptr(gap))
    if rc not in (OK, ETOKEN):
        raise ValueError(f"sv_oracle_tree_greedy failed ({rc})")
    return {"tokens": out_t, "nodes": out_nodes[:, :N], "n": out_n, "gap": gap, "status": rc}


def e4m3_decode(codes) -> np.ndarray:
    """FP8 E4M3 bytes to float64 (reading R13 in sv_oracle.c)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _load().sv_oracle_e4m3_decode(codes.size, _ptr(codes), _ptr(out))
    return out


def verify_fp8(hidden8, hscale, W8, wscale, draft, q_logits, uniforms, temperature: float,
               want_logits: bool = False) -> dict:
    """The verify step with an FP8 LM head (R13): hidden8 [B, K+1, d] and
    W8 [V, d] E4M3 bytes (uint8), hscale [B, K+1] and wscale [V] float32.
    Other arguments and the result as verify()."""
    hidden8 = _c(hidden8, np.uint8)
    W8 = _c(W8, np.uint8)
    B, rows, d = hidden8.shape
    K = rows - 1
    V = W8.shape[0]
    hscale = _c(hscale, np.float32).reshape(B * rows)
    wscale = _c(wscale, np.float32).reshape(V)
    draft = _c(draft, np.int32).reshape(B, K)
    T = float(temperature)
    q = None if (K == 0 or q_logits is None) else _c(q_logits, np.float32).reshape(B, K, V)
    u = None if T == 0.0 else _c(uniforms, np.float32).reshape(B, rows)
    tokens = np.empty((B, rows), dtype=np.int32)
    n_acc = np.empty((B,), dtype=np.int32)
    dist = np.empty((B,), dtype=np.float64)
    dacc = np.empty((B,), dtype=np.float64)
    ddraw = np.empty((B,), dtype=np.float64)
    lg = np.empty((B * rows, V), dtype=np.float64) if want_logits else None
    lse_p = np.full((B * rows,), np.nan)
    lse_q = np.full((max(B * K, 1),), np.nan)
    rc = _load().sv_oracle_verify_fp8(V, d, B, K, _ptr(hidden8), _ptr(hscale), _ptr(W8),
                                      _ptr(wscale), _ptr(draft), _ptr(q), _ptr(u), T,
                                      _ptr(tokens), _ptr(n_acc), _ptr(dist), _ptr(lg),
                                      _ptr(lse_p), _ptr(lse_q), _ptr(dacc), _ptr(ddraw))
    if rc not in (OK, ETOKEN):
        raise ValueError(f"sv_oracle_verify_fp8 failed ({rc})")
    return {"tokens": tokens, "n_accepted": n_acc, "dist": dist, "dist_accept": dacc,
            "dist_draw": ddraw, "logits": lg, "lse_p": lse_p, "lse_q": lse_q[:B * K],
            "status": rc}
