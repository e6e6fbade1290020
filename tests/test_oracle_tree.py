"""Pins of the oracle's greedy tree verification (reading R12): the pages'
two-branch tree worked by hand, the chain tree (which is linear greedy
verification, pinned by the pages' greedy example in test_oracle_pins.py),
and a brute-force enumeration of root-to-node paths on random small trees."""
import numpy as np

import oracle


def _one_hot_rows(argmax, V):
    H = np.zeros((1, len(argmax), V), dtype=np.float32)
    H[0, np.arange(len(argmax)), np.array(argmax)] = 1.0
    return H, np.eye(V, dtype=np.float32)


def test_two_branch_tree_by_hand(golden):
    g = golden("tree_example.json")
    H, W = _one_hot_rows(g["row_argmax"], g["V"])
    par = np.array([g["parents"]], dtype=np.int32)
    for c in g["cases"]:
        out = oracle.tree_greedy(H, W, np.array([c["tokens"]], np.int32), par)
        assert out["tokens"][0].tolist() == c["out_tokens"], c["name"]
        assert out["nodes"][0].tolist() == c["nodes"], c["name"]
        assert int(out["n"][0]) == c["n"], c["name"]


def test_chain_tree_is_linear_greedy_verification():
    rng = np.random.default_rng(12)
    V, d, B, N = 30, 6, 40, 5
    W = rng.standard_normal((V, d)).astype(np.float32)
    H = rng.standard_normal((B, N + 1, d)).astype(np.float32)
    L = oracle.logits(H.reshape(-1, d), W).reshape(B, N + 1, V)
    arg = L.argmax(axis=-1)
    # drafts that follow the target for a random number of steps
    x = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):
        m = rng.integers(0, N + 1)
        x[b, :m] = arg[b, :m]
    chain = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tree = oracle.tree_greedy(H, W, x, chain)
    lin = oracle.verify(H, W, x, np.zeros((B, N, V), np.float32), None, 0.0)
    assert np.array_equal(tree["tokens"], lin["tokens"])
    assert np.array_equal(tree["n"], lin["n_accepted"])


def test_random_trees_against_path_enumeration():
    rng = np.random.default_rng(13)
    V, d, N = 6, 5, 12
    for trial in range(200):
        W = rng.standard_normal((V, d)).astype(np.float32)
        H = rng.standard_normal((1, N + 1, d)).astype(np.float32)
        par = np.array([rng.integers(-1, j) if j > 0 else -1 for j in range(N)], np.int32)
        arg = oracle.logits(H[0], W).argmax(axis=-1)
        tok = rng.integers(0, V, size=N).astype(np.int32)
        # bias the tokens toward the target's choices so that paths survive
        for j in range(N):
            if rng.random() < 0.6:
                tok[j] = arg[par[j] + 1]
        out = oracle.tree_greedy(H, W, tok[None], par[None])
        # every node's root path, checked token by token
        best, best_path = 0, []
        for j in range(N):
            path, r = [], j
            while r >= 0:
                path.append(r)
                r = par[r]
            path.reverse()
            ok = all(tok[node] == arg[(par[node] + 1)] for node in path)
            if ok and len(path) > best:
                best, best_path = len(path), path
        assert int(out["n"][0]) == best
        want = [int(tok[n]) for n in best_path]
        last_row = best_path[-1] + 1 if best_path else 0
        want += [int(arg[last_row])]
        assert out["tokens"][0].tolist() == want + [-1] * (N + 1 - len(want))
        assert out["nodes"][0].tolist() == best_path + [-1] * (N - len(best_path))


def test_invalid_trees_are_reported():
    V, N = 8, 3
    H, W = _one_hot_rows([1, 2, 3, 4], V)
    out = oracle.tree_greedy(H, W, np.array([[1, 2, 3]], np.int32),
                             np.array([[-1, 1, 0]], np.int32))   # parent not before child
    assert out["n"][0] == -1 and np.all(out["tokens"][0] == -1)
    out = oracle.tree_greedy(H, W, np.array([[1, 9, 3]], np.int32),
                             np.array([[-1, 0, 1]], np.int32))   # token out of range
    assert out["n"][0] == -1
