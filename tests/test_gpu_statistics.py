"""The method's statistical invariants reproduced through the GPU path.

The pages check the rule by simulation on small vocabularies ("Speculative
Decoding: Two Models, One Voice", 'Checking the math honestly': a six-token
p and q, K = 4, 200k rounds; "Speculative Decoding: Guess Several Tokens,
Check Them in One Pass", Step 3: a three-token p and q).  Here the same
distributions are fed to the CUDA library (fp32 path): hidden row e_0 and
W[v, 0] = log p(v) make the target logits log p, and q_logits = log q.
Draft tokens are drawn from q and uniforms are seeded.  Through 2M rounds
(1000 sequences per launch) the pooled emitted-token law must be within
TV 1e-3 of p, pass a chi-square test, and the mean round length must match
(1 - alpha^(K+1)) / (1 - alpha) within 4 standard errors.  A slice of the
rounds is also compared token for token with the CPU oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import FLAG_SAMPLED

pytestmark = pytest.mark.gpu

B = 1000


def _setup(P, Q, K, dev):
    V = len(P)
    d = 4
    W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    W[:, 0] = torch.log(torch.tensor(P, dtype=torch.float64)).float().to(dev)
    hidden = torch.zeros((B, K + 1, d), dtype=torch.float32, device=dev)
    hidden[:, :, 0] = 1.0
    ql = torch.log(torch.tensor(Q, dtype=torch.float64)).float().to(dev)
    q_logits = ql.expand(B, K, V).contiguous()
    cdf = torch.cumsum(torch.tensor(Q, dtype=torch.float64), 0).to(dev)
    return W, hidden, q_logits, cdf


def _draw(cdf, K, gen, dev):
    """Draft tokens from q by inverse CDF on seeded uniforms (the draft's
    own sampling) and the verify uniforms on the 2^-24 grid."""
    V = cdf.numel()
    r = torch.rand((B, K), generator=gen, device=dev, dtype=torch.float64)
    x = torch.searchsorted(cdf, r, right=True).clamp_max(V - 1).to(torch.int32)
    u = torch.randint(0, 1 << 24, (B, K + 1), generator=gen, device=dev).float() * 2.0 ** -24
    return x.contiguous(), u.contiguous()


def _run(P, Q, K, launches, seed, oracle_launches=0):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    V = len(P)
    W, hidden, q_logits, cdf = _setup(P, Q, K, dev)
    eng = sv.SpecVerify(V, 4, B, K, "fp32", device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    counts = torch.zeros(V, dtype=torch.int64, device=dev)
    lengths = torch.zeros(K + 2, dtype=torch.int64, device=dev)
    accepted_tests = torch.zeros((), dtype=torch.int64, device=dev)
    bad = flagged = 0
    for it in range(launches):
        x, u = _draw(cdf, K, gen, dev)
        tok, n = eng.run(hidden, W, x, q_logits, u, 1.0)
        valid = tok[tok >= 0].long()
        counts += torch.bincount(valid, minlength=V)
        lengths += torch.bincount((n + 1).long(), minlength=K + 2)
        accepted_tests += n.long().sum()
        if it < oracle_launches:
            ref = oracle.verify(hidden.cpu().numpy(), W.cpu().numpy(), x.cpu().numpy(),
                                q_logits.cpu().numpy(), u.cpu().numpy(), 1.0)
            fl = ref["dist"] <= FLAG_SAMPLED
            gt, gn = tok.cpu().numpy(), n.cpu().numpy()
            mism = (np.any(gt != ref["tokens"], axis=1) | (gn != ref["n_accepted"])) & ~fl
            bad += int(mism.sum())
            flagged += int(fl.sum())
    assert eng.status() == sv.SV_OK
    eng.close()
    return counts.cpu().numpy(), lengths.cpu().numpy(), int(accepted_tests.item()), bad, flagged


def _round_length_stats(alpha, K):
    ks = np.arange(1, K + 2)
    probs = np.array([alpha ** (k - 1) * (1 - alpha) for k in range(1, K + 1)] + [alpha ** K])
    mean = float(np.sum(ks * probs))
    return mean, float(np.sum((ks - mean) ** 2 * probs))


def _check_law(P, counts, lengths, K):
    from scipy import stats
    emp = counts / counts.sum()
    tv = 0.5 * np.abs(emp - np.array(P)).sum()
    assert tv < 1e-3, tv
    assert stats.chisquare(counts, counts.sum() * np.array(P)).pvalue > 1e-4
    rounds = lengths.sum()
    assert lengths[0] == 0
    return emp, rounds


def test_six_token_example_two_million_rounds(golden):
    g = golden("six_token_example.json")
    P, Q, K = g["p"], g["q"], g["K"]
    counts, lengths, _, bad, flagged = _run(P, Q, K, launches=2000, seed=1,
                                            oracle_launches=20)
    assert bad == 0 and flagged <= 2
    _, rounds = _check_law(P, counts, lengths, K)
    alpha = float(np.minimum(P, Q).sum())
    mean, var = _round_length_stats(alpha, K)
    assert round(oracle.expected_tokens(alpha, K), 3) == g["tokens_per_round_formula_printed"]
    measured = float((np.arange(K + 2) * lengths).sum() / rounds)
    assert abs(measured - mean) < 4 * math.sqrt(var / rounds), (measured, mean)


def test_three_token_example_two_million_rounds(golden):
    g = golden("three_token_example.json")
    P, Q, K = g["p"], g["q"], g["gamma"]
    counts, lengths, acc_tests, bad, flagged = _run(P, Q, K, launches=2000, seed=2,
                                                    oracle_launches=20)
    assert bad == 0 and flagged <= 2
    _, rounds = _check_law(P, counts, lengths, K)
    alpha = float(np.minimum(P, Q).sum())
    assert round(alpha, 3) == g["acceptance_printed"]
    mean, var = _round_length_stats(alpha, K)
    measured = float((np.arange(K + 2) * lengths).sum() / rounds)
    assert abs(measured - mean) < 4 * math.sqrt(var / rounds)
    assert round(mean, 3) == g["tokens_per_step_printed"]
    # acceptance rate of the accept tests actually taken: accepted / taken,
    # where a round with n accepted took min(n + 1, K) tests
    taken = int(sum(lengths[k] * min(k, K) for k in range(1, K + 2)))
    rate = acc_tests / taken
    assert abs(rate - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / taken)


def test_greedy_worked_example_on_the_gpu(golden):
    g = golden("greedy_example.json")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    V, K = g["V"], len(g["draft"])
    d = V + (4 - V % 4) % 4   # the fp32 path wants d % 4 == 0
    # W = identity (zero-padded), hidden row i = the target's logits at i
    Wp = torch.zeros((V, d), dtype=torch.float32, device=dev)
    Wp[:, :V] = torch.eye(V, dtype=torch.float32, device=dev)
    Hp = torch.zeros((1, K + 1, d), dtype=torch.float32, device=dev)
    Hp[0, torch.arange(K + 1), torch.tensor(g["target_argmax"])] = 1.0
    eng = sv.SpecVerify(V, d, 1, K, "fp32", device=dev)
    draft = torch.tensor([g["draft"]], dtype=torch.int32, device=dev)
    tok, n = eng.run(Hp, Wp, draft, None, None, 0.0)
    want = g["expected_tokens"] + [-1] * (K + 1 - len(g["expected_tokens"]))
    assert tok.cpu().tolist()[0] == want
    assert int(n.item()) == g["expected_n_accepted"]
    assert eng.status() == sv.SV_OK
    eng.close()
