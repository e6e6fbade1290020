"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.

Contract checked here:
  * logits within 2e-2 absolute (bf16 inputs, fp32 accumulation) and the
    target probabilities within 1e-5;
  * token ids and accept counts bit-exact, except rounds whose uniform lies
    within 1e-6 of a decision threshold (sampling) or whose deciding rows
    have top-two logits within 1e-7 (greedy); those are counted;
  * all five configurations at full size, plus small shapes that span
    several tiles with ragged tails, K = 0, and the degenerate inputs.
"""
import numpy as np
import pytest
import torch

import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import (check_numerics, compare_tokens, gpu_verify, oracle_verify)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _case(dev, wl, T, seed, want_logits=True, rows=None, W=None, W_np=None):
    if W is None:
        W = si.make_weights(wl, seed=seed, device=dev)
        W_np = si.to_oracle(W)
    inp = si.make_round(wl, W, seed=seed + 1, T=T)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    got = gpu_verify(eng, W, inp, T)
    assert got["status"] == sv.SV_OK
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"],
                        T, want_logits=want_logits, rows=rows)
    return eng, got, ref, inp


SMALL = [
    # (overrides, T): several 128-row tiles, ragged V and d, every
    # accumulator mode of the tensor-core path, K = 0, greedy
    (dict(dtype="bf16", B=1, K=4, V=1000, d=256), 1.0),
    (dict(dtype="bf16", B=2, K=3, V=777, d=136), 0.7),
    (dict(dtype="bf16", B=4, K=4, V=4096, d=512), 0.0),
    (dict(dtype="bf16", B=1, K=0, V=300, d=64), 1.0),
    (dict(dtype="bf16", B=1, K=0, V=300, d=64), 0.0),
    (dict(dtype="bf16", B=3, K=1, V=33, d=8), 1.0),
    (dict(dtype="bf16", B=16, K=3, V=1152, d=64), 1.0),
    (dict(dtype="bf16", B=8, K=3, V=5000, d=1024, w_std=1 / 32), 1.0),
    (dict(dtype="bf16", B=20, K=4, V=1500, d=128), 1.0),
    (dict(dtype="bf16", B=20, K=4, V=1500, d=512), 2.0),
    (dict(dtype="bf16", B=40, K=5, V=3000, d=256), 1.0),
    (dict(dtype="bf16", B=64, K=5, V=2000, d=128), 1.0),
    (dict(dtype="bf16", B=64, K=5, V=2000, d=128), 0.0),
    # column halves whose second half runs past the last row, with an odd
    # number of 64-wide k blocks (single-block stages)
    (dict(dtype="bf16", B=53, K=4, V=1300, d=192), 0.9),
    (dict(B=1, K=4), 1.0),
    (dict(B=5, K=2, V=97), 0.5),
    (dict(B=5, K=2, V=97), 0.0),
]


@pytest.mark.parametrize("over,T", SMALL)
def test_small_shapes_match_oracle(dev, over, T):
    wl = si.workload("tiny", **over)
    eng, got, ref, _ = _case(dev, wl, T, seed=11)
    check_numerics(eng, ref, wl, T)
    bad, _ = compare_tokens(got, ref, T)
    assert bad == 0
    eng.close()


def test_tiny_fp32_thousand_rounds(dev):
    # V=1000, d=256, B=1, K=4, fp32, T=1, draft noise 0.5, 1000 rounds
    wl = si.workload("tiny")
    W = si.make_weights(wl, seed=1000, device=dev)
    W_np = si.to_oracle(W)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    bad = flagged = 0
    tokens = 0
    for r in range(1000):
        inp = si.make_round(wl, W, seed=1000 + r)
        got = gpu_verify(eng, W, inp, 1.0)
        assert got["status"] == sv.SV_OK
        ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"],
                            inp["uniforms"], 1.0)
        b, f = compare_tokens(got, ref, 1.0)
        bad += b
        flagged += f
        tokens += int(got["n_accepted"][0]) + 1
    assert bad == 0
    assert flagged <= 2
    # acceptance near the configured draft quality (noise 0.5 ~ alpha 0.8)
    assert 2.5 < tokens / 1000 < 4.5
    eng.close()


@pytest.fixture(scope="module")
def w8b(dev):
    wl = si.workload("llama8b")
    W = si.make_weights(wl, seed=2024, device=dev)
    return W, si.to_oracle(W)


@pytest.mark.parametrize("alpha", [0.6, 0.7, 0.8])
def test_llama8b_shape(dev, w8b, alpha):
    W, W_np = w8b
    wl = si.workload("llama8b", alpha=alpha)
    for seed in (1, 2):
        eng, got, ref, _ = _case(dev, wl, 1.0, seed=100 * seed + int(alpha * 10), W=W, W_np=W_np)
        check_numerics(eng, ref, wl, 1.0)
        bad, _ = compare_tokens(got, ref, 1.0)
        assert bad == 0
        eng.close()


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_llama8b_b8_k7(dev, w8b, T):
    W, W_np = w8b
    wl = si.workload("llama8b_b8k7")
    eng, got, ref, _ = _case(dev, wl, T, seed=5, W=W, W_np=W_np)
    check_numerics(eng, ref, wl, T)
    bad, _ = compare_tokens(got, ref, T)
    assert bad == 0
    eng.close()


@pytest.mark.parametrize("B,K", [(1, 3), (2, 4), (4, 5), (8, 3), (16, 4), (32, 5), (64, 3),
                                 (64, 4), (64, 5)])
def test_llama8b_batch_sweep_sampled_sequences(dev, w8b, B, K):
    # full-size launches; the oracle checks the first and last sequence and
    # the logits of every row on a sample of vocabulary entries
    W, W_np = w8b
    wl = si.workload("sweep", B=B, K=K)
    rows = sorted({0, B - 1})
    eng, got, ref, inp = _case(dev, wl, 1.0, seed=B * 10 + K, want_logits=False, rows=rows,
                               W=W, W_np=W_np)
    bad, _ = compare_tokens(got, ref, 1.0, seqs=rows)
    assert bad == 0
    import oracle
    lg = eng.logits().cpu().numpy()
    cols = np.random.default_rng(B + K).choice(wl.V, 64, replace=False)
    H = si.to_oracle(inp["hidden"]).reshape(B * (K + 1), wl.d)
    for c in cols:
        exact = oracle.logits(H, W_np, int(c), int(c) + 1)[:, 0]
        assert np.abs(lg[:, c] - exact).max() <= 2e-2
    # every emitted sequence is an accepted prefix and one more token
    n = got["n_accepted"]
    assert np.all((got["tokens"] >= 0).sum(axis=1) == n + 1)
    eng.close()


def test_llama70b_shape(dev):
    wl = si.workload("llama70b")
    eng, got, ref, _ = _case(dev, wl, 1.0, seed=70)
    check_numerics(eng, ref, wl, 1.0)
    bad, _ = compare_tokens(got, ref, 1.0)
    assert bad == 0
    eng.close()


def test_repeated_runs_are_bitwise_identical(dev):
    wl = si.workload("tiny", dtype="bf16", B=4, K=4, V=20000, d=1024, w_std=1 / 32)
    W = si.make_weights(wl, seed=3, device=dev)
    inp = si.make_round(wl, W, seed=4)
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    first = None
    for _ in range(50):
        tok, n = eng.run(inp["hidden"], W, inp["draft"], inp["q_logits"], inp["uniforms"], 1.0)
        cur = (tok.clone(), n.clone(), eng.logits(), eng.lse())
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert torch.equal(a, b)
    assert eng.status() == sv.SV_OK
    eng.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_masked_draft_logits(dev, dtype):
    # draft logits of -inf (tokens the draft can never propose) are valid
    # inputs: q = 0 there, and those tokens reach the output only through
    # the residual
    over = dict(B=4, K=4, V=2000, d=256) if dtype == "bf16" else dict(B=4, K=4)
    wl = si.workload("tiny", dtype=dtype, **over)
    W = si.make_weights(wl, seed=31, device=dev)
    W_np = si.to_oracle(W)
    inp = si.make_round(wl, W, seed=32)
    q = inp["q_logits"].clone()
    mask = torch.rand(q.shape, generator=torch.Generator(device=dev).manual_seed(3),
                      device=dev) < 0.3
    drafted = torch.zeros_like(mask)
    drafted.scatter_(2, inp["draft"].long().unsqueeze(-1), True)
    q[mask & ~drafted] = float("-inf")
    inp["q_logits"] = q
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    got = gpu_verify(eng, W, inp, 1.0)
    assert got["status"] == sv.SV_OK
    ref = oracle_verify(inp["hidden"], W_np, inp["draft"], inp["q_logits"], inp["uniforms"],
                        1.0, want_logits=True)
    check_numerics(eng, ref, wl, 1.0)
    assert compare_tokens(got, ref, 1.0)[0] == 0
    eng.close()
