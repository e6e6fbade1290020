"""GPU parity and statistics of truncated sampling (top-k, then top-p, each
side with its own settings; reading R11) against the CPU oracle.

* tokens and accept counts bit-exact except rounds within rounding of a
  decision.  Membership is decided on the step's fp32 logits (within ~7e-7
  of the exact ones) and fp32 exponentials, so a cut whose logit gap or
  top-p mass margin is below 4e-6 may fall either way; the oracle reports
  the largest warped mass of a token next to such a cut (moving it moves
  every threshold and CDF edge of the round by about that much) and the
  distance of each draft token's logit from its rows' cuts.  A round is
  flagged when a decision's uniform lies within 1e-6 plus twice that mass
  of its threshold, or a draft token lies within 4e-6 of a cut;
* no cut reproduces spec_verify_run bit for bit; top-1 on both sides is
  greedy verification (the pages' greedy corollary);
* over 2M rounds on the six-token example the emitted law is the warped
  target ("Speculative Decoding: Two Models, One Voice", three remarks).
"""
import numpy as np
import pytest
import torch

import oracle
import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import FLAG_SAMPLED

pytestmark = pytest.mark.gpu

GAP_FLAG = 4e-6
MASS_FLAG = 4e-6


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _oracle(inp, W, T, pk, pp, qk, qp):
    H = si.to_oracle(inp["hidden"])
    X = si.to_oracle(inp["draft"])
    Q = None if inp["q_logits"] is None else si.to_oracle(inp["q_logits"])
    U = si.to_oracle(inp["uniforms"])
    Wn = si.to_oracle(W)
    outs = [oracle.verify_truncated(H[b:b + 1], Wn, X[b:b + 1],
                                    None if Q is None else Q[b:b + 1], U[b:b + 1], T,
                                    pk, pp, qk, qp, GAP_FLAG, MASS_FLAG)
            for b in range(H.shape[0])]
    return {k: np.concatenate([o[k] for o in outs]) for k in
            ("tokens", "n_accepted", "dist", "trunc_sens", "trunc_xgap")}


def _compare(tok, n, ref):
    """(mismatches outside flagged rounds, flagged rounds); flagged rounds
    must still match in most cases (a systematic error would not)."""
    fl = ((ref["dist"] <= FLAG_SAMPLED + 2.0 * ref["trunc_sens"])
          | (ref["trunc_xgap"] < GAP_FLAG))
    diff = np.any(tok != ref["tokens"], axis=1) | (n != ref["n_accepted"])
    assert int((diff & fl).sum()) <= max(1, int(fl.sum()) // 2)
    return int((diff & ~fl).sum()), int(fl.sum())


SETTINGS = [(50, 1.0, 0, 1.0), (0, 0.9, 0, 1.0), (100, 0.8, 200, 0.95), (0, 1.0, 40, 0.7),
            (7, 0.5, 3, 1.0)]


@pytest.mark.parametrize("pk,pp,qk,qp", SETTINGS)
def test_truncated_parity_tiny(dev, pk, pp, qk, qp):
    wl = si.workload("tiny", B=40, K=4)
    T = 0.8
    W = si.make_weights(wl, seed=61, device=dev)
    inp = si.make_round(wl, W, seed=62, T=T)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    tok, n = eng.run_truncated(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"],
                               T, pk, pp, qk, qp)
    assert eng.status() == sv.SV_OK
    ref = _oracle(inp, W, T, pk, pp, qk, qp)
    bad, flagged = _compare(tok.cpu().numpy(), n.cpu().numpy(), ref)
    assert bad == 0 and flagged <= wl.B // 4, (bad, flagged)
    eng.close()


@pytest.mark.parametrize("B,K,T", [(1, 4, 1.0), (8, 7, 0.7)])
def test_truncated_parity_llama8b(dev, B, K, T):
    wl = si.workload("llama8b", B=B, K=K, T=T)
    W = si.make_weights(wl, seed=71 + B, device=dev)
    inp = si.make_round(wl, W, seed=72 + B, T=T)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    for pk, pp, qk, qp in ((50, 0.9, 50, 0.9), (0, 0.95, 1000, 1.0)):
        tok, n = eng.run_truncated(inp["hidden"], W, inp["draft"], inp["q_logits"],
                                   inp["uniforms"], T, pk, pp, qk, qp)
        assert eng.status() == sv.SV_OK
        ref = _oracle(inp, W, T, pk, pp, qk, qp)
        bad, flagged = _compare(tok.cpu().numpy(), n.cpu().numpy(), ref)
        assert bad == 0 and flagged <= max(1, B // 4), (pk, pp, qk, qp, bad, flagged)
    eng.close()


def test_no_cut_is_the_plain_run_and_top_one_is_greedy(dev):
    wl = si.workload("tiny", B=32, K=4)
    T = 1.0
    W = si.make_weights(wl, seed=81, device=dev)
    inp = si.make_round(wl, W, seed=82, T=T)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    tok0, n0 = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"], T)
    tok1, n1 = eng.run_truncated(inp["hidden"], W, inp["draft"], inp["q_logits"],
                                 inp["uniforms"], T, 0, 1.0, wl.V, 1.0)
    assert torch.equal(tok0, tok1) and torch.equal(n0, n1)
    # top-1 on both sides, with top-1 drafts: greedy verification
    x = torch.argmax(inp["q_logits"], dim=-1).to(torch.int32).contiguous()
    tg, ng = eng.run(inp["hidden"], W, x, None, None, 0.0)
    for seed in range(3):
        u = torch.rand((wl.B, wl.K + 1), device=dev,
                       generator=torch.Generator(device=dev).manual_seed(seed))
        tt, nt = eng.run_truncated(inp["hidden"], W, x, inp["q_logits"], u.contiguous(), T,
                                   1, 1.0, 1, 1.0)
        assert torch.equal(tt, tg) and torch.equal(nt, ng)
    assert eng.status() == sv.SV_OK
    eng.close()


def test_truncated_emitted_law_over_two_million_rounds(dev, golden):
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    V, d, B, K = len(P), 4, 1000, 1
    pk, pp, qk, qp = 4, 0.9, 5, 0.95
    p_w, _, _, _ = oracle.truncate(np.log(P), 1.0, pk, pp)
    q_w, _, _, _ = oracle.truncate(np.log(Q), 1.0, qk, qp)
    W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    W[:, 0] = torch.log(torch.tensor(P, dtype=torch.float64)).float().to(dev)
    hidden = torch.zeros((B, K + 1, d), dtype=torch.float32, device=dev)
    hidden[:, :, 0] = 1.0
    ql = torch.log(torch.tensor(Q, dtype=torch.float64)).float().to(dev).expand(B, K, V)
    ql = ql.contiguous()
    cdf = torch.cumsum(torch.tensor(q_w, dtype=torch.float64), 0).to(dev)
    eng = sv.SpecVerify(V, d, B, K, "fp32", device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    counts = torch.zeros(V, dtype=torch.int64, device=dev)
    launches = 2000
    for _ in range(launches):
        r = torch.rand((B, K), generator=gen, device=dev, dtype=torch.float64)
        x = torch.searchsorted(cdf, r, right=True).clamp_max(V - 1).to(torch.int32).contiguous()
        u = (torch.randint(0, 1 << 24, (B, K + 1), generator=gen, device=dev).float()
             * 2.0 ** -24).contiguous()
        tok, n = eng.run_truncated(hidden, W, x, ql, u, 1.0, pk, pp, qk, qp)
        counts += torch.bincount(tok[:, 0].long(), minlength=V)
    assert eng.status() == sv.SV_OK
    eng.close()
    from scipy import stats
    c = counts.cpu().numpy()
    total = c.sum()
    assert np.all(c[p_w == 0] == 0)
    emp = c / total
    assert 0.5 * np.abs(emp - p_w).sum() < 1.5e-3
    keep = p_w > 0
    assert stats.chisquare(c[keep], total * p_w[keep]).pvalue > 1e-4
