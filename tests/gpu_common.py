"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI and the CPU oracle on the same seeded inputs, and compare."""
import concurrent.futures
import os

import numpy as np
import torch

import oracle
import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv

# A round is "flagged" when a uniform lies within this distance of a
# decision threshold it was compared with (sampling), or when the top two
# logits of a row that decided something are this close (greedy).
FLAG_SAMPLED = 1e-6
FLAG_GREEDY = 1e-7
LOGIT_TOL = 2e-2      # bf16 inputs, fp32 accumulation
PROB_TOL = 1e-5

_POOL = concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4))


def oracle_verify(hidden, W_np, draft, q_logits, uniforms, T, want_logits=False, rows=None):
    """The oracle on host copies of the inputs, one sequence per thread (the
    C oracle releases the GIL).  `rows` restricts it to some sequences."""
    H = si.to_oracle(hidden)
    X = si.to_oracle(draft)
    Q = None if q_logits is None else si.to_oracle(q_logits)
    U = si.to_oracle(uniforms)
    B = H.shape[0]
    seqs = list(range(B)) if rows is None else list(rows)

    def one(b):
        q = None if q_logits is None else (Q[b:b + 1] if Q.size else Q)
        return oracle.verify(H[b:b + 1], W_np, X[b:b + 1], q,
                             U[b:b + 1], T, want_logits=want_logits)

    res = list(_POOL.map(one, seqs))
    out = {k: np.concatenate([r[k] for r in res]) for k in
           ("tokens", "n_accepted", "dist", "dist_accept", "dist_draw", "lse_p")}
    out["lse_q"] = np.concatenate([r["lse_q"] for r in res])
    if want_logits:
        out["logits"] = np.concatenate([r["logits"] for r in res])
    out["status"] = min(r["status"] for r in res)
    out["seqs"] = seqs
    return out


def gpu_verify(eng, W, inp, T):
    tok, n = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"], T)
    code = eng.status()
    return {"tokens": tok.cpu().numpy(), "n_accepted": n.cpu().numpy(), "status": code}


def flagged(ref, T):
    return ref["dist"] <= (FLAG_SAMPLED if T > 0 else FLAG_GREEDY)


def compare_tokens(got, ref, T, seqs=None):
    """Bit-exact token ids and accept counts outside flagged rounds.
    Returns (mismatches outside flagged rounds, flagged rounds)."""
    gt, gn = got["tokens"], got["n_accepted"]
    if seqs is not None:
        gt, gn = gt[seqs], gn[seqs]
    fl = flagged(ref, T)
    bad = (np.any(gt != ref["tokens"], axis=1) | (gn != ref["n_accepted"])) & ~fl
    return int(bad.sum()), int(fl.sum())


def probs(logits, lse, T):
    return np.exp(logits / T - lse[:, None])


def check_numerics(eng, ref, wl, T):
    """logits within 2e-2 abs, probabilities within 1e-5 (sampling), and
    returns the max |d logit| for reporting."""
    lg = eng.logits().cpu().numpy().astype(np.float64)
    dl = np.abs(lg - ref["logits"]).max()
    assert dl <= LOGIT_TOL, dl
    if T > 0:
        R = wl.B * (wl.K + 1)
        lse = eng.lse().cpu().numpy()
        p_gpu = probs(lg, lse[:R], T)
        p_ref = probs(ref["logits"], ref["lse_p"], T)
        dp = np.abs(p_gpu - p_ref).max()
        assert dp <= PROB_TOL, dp
        if wl.K > 0:
            assert np.abs(lse[R:] - ref["lse_q"]).max() <= 1e-6
    return float(dl)
