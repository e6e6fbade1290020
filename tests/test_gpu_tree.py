"""GPU parity of greedy tree verification (reading R12) against the CPU
oracle: the pages' two-branch tree worked by hand, the chain tree (linear
greedy verification), random trees of 15 to 63 nodes at the tiny shape, a
Medusa-like tree at the Llama-8B shape, and invalid trees.  Tokens, the
accepted path's nodes and its length must match exactly except in rounds
whose deciding rows have top-two logits within 1e-7 (flagged)."""
import numpy as np
import pytest
import torch

import oracle
import spec_inputs as si
import speculative_decoding_verification_22_gb300 as sv
from gpu_common import FLAG_GREEDY

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _tree_case(dev, eng, hidden, W, tok, par):
    t = torch.from_numpy(np.ascontiguousarray(tok, np.int32)).to(dev)
    p = torch.from_numpy(np.ascontiguousarray(par, np.int32)).to(dev)
    got_t, got_nodes, got_n = eng.run_tree_greedy(hidden, W, t, p)
    status = eng.status()
    ref = oracle.tree_greedy(si.to_oracle(hidden), si.to_oracle(W), tok, par)
    return (got_t.cpu().numpy(), got_nodes.cpu().numpy(), got_n.cpu().numpy(), status, ref)


def _compare(got_t, got_nodes, got_n, ref):
    fl = ref["gap"] <= FLAG_GREEDY
    bad = ((np.any(got_t != ref["tokens"], axis=1) | np.any(got_nodes != ref["nodes"], axis=1)
            | (got_n != ref["n"])) & ~fl)
    return int(bad.sum()), int(fl.sum())


def test_two_branch_tree_by_hand(dev, golden):
    g = golden("tree_example.json")
    V, N = g["V"], len(g["parents"])
    d = 12  # the fp32 path wants d % 4 == 0
    W = torch.zeros((V, d), dtype=torch.float32, device=dev)
    W[:, :V] = torch.eye(V, device=dev)
    H = torch.zeros((1, N + 1, d), dtype=torch.float32, device=dev)
    H[0, torch.arange(N + 1), torch.tensor(g["row_argmax"])] = 1.0
    eng = sv.SpecVerify(V, d, 1, N, "fp32", device=dev)
    for c in g["cases"]:
        gt, gn, gl, status, ref = _tree_case(dev, eng, H, W, np.array([c["tokens"]]),
                                             np.array([g["parents"]]))
        assert status == sv.SV_OK
        assert gt[0].tolist() == c["out_tokens"] and gn[0].tolist() == c["nodes"]
        assert int(gl[0]) == c["n"]
    eng.close()


def _biased_tree(rng, L, N, branch_p=0.7):
    """A random tree whose tokens follow the target's choice (from a plain
    torch matmul, input shaping only) with probability branch_p."""
    arg = L.argmax(axis=-1)
    par = np.array([rng.integers(-1, j) if j > 0 else -1 for j in range(N)], np.int32)
    tok = rng.integers(0, L.shape[-1], size=N).astype(np.int32)
    for j in range(N):
        if rng.random() < branch_p:
            tok[j] = arg[par[j] + 1]
    return tok, par


@pytest.mark.parametrize("N", [15, 31, 63])
def test_random_trees_tiny(dev, N):
    wl = si.workload("tiny", B=6, K=N)
    W = si.make_weights(wl, seed=91 + N, device=dev)
    inp = si.make_round(wl, W, seed=92 + N, T=0.0)
    L = (inp["hidden"].float() @ W.float().T).cpu().numpy()
    rng = np.random.default_rng(N)
    toks, pars = zip(*[_biased_tree(rng, L[b], N) for b in range(wl.B)])
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, N, wl.dtype, device=dev)
    gt, gn, gl, status, ref = _tree_case(dev, eng, inp["hidden"], W, np.stack(toks),
                                         np.stack(pars))
    assert status == sv.SV_OK
    bad, flagged = _compare(gt, gn, gl, ref)
    assert bad == 0 and flagged <= 1
    assert (gl > 0).any()
    # the chain tree is linear greedy verification
    chain = np.tile(np.arange(-1, N - 1, dtype=np.int32), (wl.B, 1))
    gt2, gn2, gl2, status, _ = _tree_case(dev, eng, inp["hidden"], W, np.stack(toks), chain)
    lt, ln = eng.run(inp["hidden"], W, torch.from_numpy(np.stack(toks)).to(dev), None, None, 0.0)
    assert np.array_equal(gt2, lt.cpu().numpy()) and np.array_equal(gl2, ln.cpu().numpy())
    eng.close()


def test_medusa_like_tree_llama8b(dev):
    # three levels of three branches (3 + 9 + 27 = 39 nodes), B = 2
    par = []
    level = [-1]
    for depth in range(3):
        nxt = []
        for p in level:
            for _ in range(3):
                par.append(p)
                nxt.append(len(par) - 1)
        level = nxt
    N = len(par)
    wl = si.workload("llama8b", B=2, K=N, T=0.0)
    W = si.make_weights(wl, seed=101, device=dev)
    inp = si.make_round(wl, W, seed=102, T=0.0)
    L = (inp["hidden"].float() @ W.float().T).cpu().numpy()
    rng = np.random.default_rng(3)
    toks = []
    for b in range(wl.B):
        arg = L[b].argmax(axis=-1)
        tok = rng.integers(0, wl.V, size=N).astype(np.int32)
        for j, p in enumerate(par):
            if j % 3 == 0:  # the first child of every node follows the target
                tok[j] = arg[p + 1]
        toks.append(tok)
    pars = np.tile(np.array(par, np.int32), (wl.B, 1))
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, N, wl.dtype, device=dev)
    gt, gn, gl, status, ref = _tree_case(dev, eng, inp["hidden"], W, np.stack(toks), pars)
    assert status == sv.SV_OK
    bad, flagged = _compare(gt, gn, gl, ref)
    assert bad == 0 and flagged <= 1
    assert np.all(gl[ref["gap"] > FLAG_GREEDY] == 3)  # the following branch is accepted
    eng.close()


def test_invalid_trees_are_reported(dev):
    wl = si.workload("tiny", B=3, K=4)
    W = si.make_weights(wl, seed=111, device=dev)
    inp = si.make_round(wl, W, seed=112, T=0.0)
    tok = np.array([[1, 2, 3, 4]] * 3, np.int32)
    par = np.array([[-1, 0, 1, 2], [-1, 0, 3, 1], [-1, -1, 0, 1]], np.int32)  # row 1: 3 >= 2
    tok[2, 1] = wl.V                                                           # row 2: bad token
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, wl.dtype, device=dev)
    gt, gn, gl, status, ref = _tree_case(dev, eng, inp["hidden"], W, tok, par)
    assert status == sv.SV_ERR_TOKEN
    assert gl.tolist()[1:] == [-1, -1] and ref["n"].tolist()[1:] == [-1, -1]
    assert np.all(gt[1:] == -1) and np.all(gn[1:] == -1)
    assert gl[0] == ref["n"][0] and np.array_equal(gt[0], ref["tokens"][0])
    assert eng.status() == sv.SV_OK
    eng.close()
