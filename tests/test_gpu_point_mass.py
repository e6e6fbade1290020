"""GPU parity and statistics of the point-mass draft path (q_logits = NULL)
and of the prompt-lookup drafter, against the CPU oracle.

* drafter: bit-exact drafts and lengths on random contexts (small and large
  vocabularies, ragged lengths, a row stride above the lengths, empty and
  one-token contexts) and on the hand-derived cases of
  tests/golden/ngram_examples.json;
* verify with point-mass drafts: tokens and accept counts bit-exact except
  rounds within 1e-6 of a threshold, at the tiny fp32 shape (sampled and
  greedy) and at the Llama-8B shape (bf16), with short drafts (-1 tails);
* the emitted law of 2M point-mass rounds on the six-token example is p,
  and the acceptance frequency of the proposed token is p(x) ("Speculative
  Decoding: Two Models, One Voice", "The rule that makes it exact");
* the host-buffer entry point and an invalid short-draft pattern.
"""
import numpy as np
import pytest
import torch

import oracle
import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import compare_tokens, gpu_verify, oracle_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _drafter_case(dev, ctx, lens, K, n_min=2, n_max=5):
    t = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).to(dev)
    ln = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).to(dev)
    d, n = sv.spec_ngram_draft(t, ln, K, n_min, n_max)
    torch.cuda.synchronize()
    rd, rn = oracle.ngram_draft(ctx, lens, K, n_min, n_max)
    assert np.array_equal(d.cpu().numpy(), rd)
    assert np.array_equal(n.cpu().numpy(), rn)
    return rn


@pytest.mark.parametrize("vocab,L,K", [(3, 300, 4), (8, 4000, 16), (50000, 2048, 4),
                                       (2, 64, 1), (6, 60000, 4)])  # last: beyond smem
def test_drafter_matches_the_oracle(dev, vocab, L, K):
    rng = np.random.default_rng(vocab + L)
    B = 64
    ctx = rng.integers(0, vocab, size=(B, L)).astype(np.int32)
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    lens[:4] = [0, 1, 2, L]
    if vocab > 1000:
        # plant copies so that a large vocabulary still has matches
        for b in range(4, B, 2):
            if lens[b] > 40:
                s = rng.integers(0, lens[b] - 20)
                ctx[b, lens[b] - 6:lens[b]] = ctx[b, s:s + 6]
    rn = _drafter_case(dev, ctx, lens, K)
    assert (rn > 0).any()


def test_drafter_n_bounds_and_golden_cases(dev, golden):
    g = golden("ngram_examples.json")
    for c in g["cases"]:
        row = np.array([c["tokens"]], dtype=np.int32)
        _drafter_case(dev, row, [c["length"]], c["K"], c["n_min"], c["n_max"])
    rng = np.random.default_rng(9)
    ctx = rng.integers(0, 5, size=(32, 500)).astype(np.int32)
    lens = np.full(32, 500, np.int32)
    for lo, hi in ((1, 1), (3, 3), (1, 16), (16, 16)):
        _drafter_case(dev, ctx, lens, 8, lo, hi)


def _point_round(dev, wl, T, seed, short_every=3):
    W = si.make_weights(wl, seed=seed, device=dev)
    inp = si.make_round(wl, W, seed=seed + 1, T=T)
    draft = inp["draft"].clone()
    rng = np.random.default_rng(seed)
    for b in range(0, wl.B, short_every):
        kb = int(rng.integers(0, wl.K))
        draft[b, kb:] = -1
    inp = dict(inp, draft=draft.contiguous(), q_logits=None)
    return W, inp


@pytest.mark.parametrize("T", [1.0, 0.7, 0.0])
def test_point_mass_parity_tiny(dev, T):
    wl = si.workload("tiny", B=48, K=4)
    W, inp = _point_round(dev, wl, T, seed=31)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    got = gpu_verify(eng, W, inp, T)
    assert got["status"] == sv.SV_OK
    ref = oracle_verify(inp["hidden"], si.to_oracle(W), inp["draft"], None, inp["uniforms"], T)
    bad, flagged = compare_tokens(got, ref, T)
    assert bad == 0 and flagged <= 2
    kb = (inp["draft"].cpu().numpy() >= 0).sum(axis=1)
    assert np.all(got["n_accepted"] <= kb)
    eng.close()


@pytest.mark.parametrize("B,K,T", [(1, 4, 1.0), (8, 7, 0.7), (8, 7, 0.0)])
def test_point_mass_parity_llama8b(dev, B, K, T):
    wl = si.workload("llama8b", B=B, K=K, T=T)
    W, inp = _point_round(dev, wl, T, seed=41 + B, short_every=2)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    got = gpu_verify(eng, W, inp, T)
    assert got["status"] == sv.SV_OK
    ref = oracle_verify(inp["hidden"], si.to_oracle(W), inp["draft"], None, inp["uniforms"], T)
    bad, flagged = compare_tokens(got, ref, T)
    assert bad == 0 and flagged <= 1
    eng.close()


def test_point_mass_emits_p_over_two_million_rounds(dev, golden):
    g = golden("six_token_example.json")
    P = np.array(g["p"])
    V, d, B, K, x = len(P), 4, 1000, 1, 3
    W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    W[:, 0] = torch.log(torch.tensor(P, dtype=torch.float64)).float().to(dev)
    hidden = torch.zeros((B, K + 1, d), dtype=torch.float32, device=dev)
    hidden[:, :, 0] = 1.0
    draft = torch.full((B, K), x, dtype=torch.int32, device=dev)
    eng = sv.SpecVerify(V, d, B, K, "fp32", device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    counts = torch.zeros(V, dtype=torch.int64, device=dev)
    accepted = torch.zeros((), dtype=torch.int64, device=dev)
    launches = 2000
    for _ in range(launches):
        u = (torch.randint(0, 1 << 24, (B, K + 1), generator=gen, device=dev).float()
             * 2.0 ** -24).contiguous()
        tok, n = eng.run(hidden, W, draft, None, u, 1.0)
        # K = 1: the first token is x if accepted, else the residual draw
        counts += torch.bincount(tok[:, 0].long(), minlength=V)
        accepted += (n == 1).sum()
    assert eng.status() == sv.SV_OK
    eng.close()
    from scipy import stats
    c = counts.cpu().numpy()
    total = B * launches
    emp = c / total
    assert 0.5 * np.abs(emp - P).sum() < 1e-3
    assert stats.chisquare(c, total * P).pvalue > 1e-4
    rate = int(accepted.item()) / total
    assert abs(rate - P[x]) < 4 * np.sqrt(P[x] * (1 - P[x]) / total)


def test_point_mass_host_entry_and_bad_short_draft(dev):
    wl = si.workload("tiny", B=6, K=4)
    W, inp = _point_round(dev, wl, 1.0, seed=51, short_every=2)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    tok_d, n_d = eng.run(inp["hidden"], W, inp["draft"], None, inp["uniforms"], 1.0)
    host = {k: inp[k].cpu().pin_memory() for k in ("hidden", "draft", "uniforms")}
    ht = torch.empty((wl.B, wl.K + 1), dtype=torch.int32).pin_memory()
    hn = torch.empty((wl.B,), dtype=torch.int32).pin_memory()
    rc = sv.load_library().spec_verify_run_host(
        eng.h, host["hidden"].data_ptr(), W.data_ptr(), host["draft"].data_ptr(), None,
        host["uniforms"].data_ptr(), 1.0, ht.data_ptr(), hn.data_ptr())
    assert rc == sv.SV_OK
    assert torch.equal(ht, tok_d.cpu()) and torch.equal(hn, n_d.cpu())
    # a token after the first -1 makes that sequence's draft invalid
    bad = inp["draft"].clone()
    bad[1] = torch.tensor([int(bad[1, 0]), -1, 5, -1], dtype=torch.int32)
    got = gpu_verify(eng, W, dict(inp, draft=bad), 1.0)
    assert got["status"] == sv.SV_ERR_TOKEN
    assert got["n_accepted"][1] == -1 and np.all(got["tokens"][1] == -1)
    # -1 is never a terminator when the draft comes with q_logits
    full = si.make_round(wl, W, seed=52, T=1.0)
    neg = full["draft"].clone()
    neg[2, 3] = -1
    got = gpu_verify(eng, W, dict(full, draft=neg), 1.0)
    assert got["status"] == sv.SV_ERR_TOKEN and got["n_accepted"][2] == -1
    assert eng.status() == sv.SV_OK
    eng.close()
