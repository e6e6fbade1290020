"""Pins of the oracle's point-mass draft rule (readings R8, R9) and its
prompt-lookup drafter (R10), against things other than the oracle itself:

* the general rule of the pages (pinned by their worked examples in
  test_oracle_pins.py) given one-hot q rows -- a draft proposed with
  certainty is exactly that q ("Speculative Decoding: The Algebra and the
  Proof", "Where it breaks": q is the distribution that actually generated
  the proposal);
* the method's exactness ("Speculative Decoding: Two Models, One Voice",
  "The rule that makes it exact"): over a deterministic grid of uniforms the
  emitted law is p, and the acceptance frequency is p(x);
* hand-derived draws and hand-derived prompt-lookup drafts
  (tests/golden/ngram_examples.json);
* brute-force properties of the drafter on random small contexts.
"""
import numpy as np
import pytest

import oracle


def _rand_p(rng, K, V):
    p = rng.random((K + 1, V)) ** 3
    return p / p.sum(axis=1, keepdims=True)


def test_point_mass_equals_the_general_rule_with_one_hot_q():
    rng = np.random.default_rng(11)
    V, K, n = 12, 4, 4000
    p = _rand_p(rng, K, V)
    x = rng.integers(0, V, size=(n, K)).astype(np.int32)
    u = rng.random((n, K + 1))
    # one sequence of x at a time: the general rule needs q rows per round
    for r in range(0, n, 500):
        q = np.zeros((K, V))
        q[np.arange(K), x[r]] = 1.0
        xr = np.repeat(x[r:r + 1], 500, axis=0)
        ur = u[r:r + 500]
        t_gen, n_gen, _ = oracle.rule_batch(p, q, xr, ur)
        t_pm, n_pm, _ = oracle.rule_batch(p, None, xr, ur)
        assert np.array_equal(t_gen, t_pm) and np.array_equal(n_gen, n_pm)


def test_point_mass_emits_p_over_a_uniform_grid():
    """K = 1, x fixed: P(emit v) = p(v) exactly; the grid's step bounds the
    error."""
    p = np.array([0.05, 0.25, 0.1, 0.4, 0.2])
    P = np.stack([p, np.full(5, 0.2)])      # row 1 (bonus) unused when rejected
    x = 3
    g = (np.arange(2000) + 0.5) / 2000.0
    u0, u1 = np.meshgrid(g, g, indexing="ij")
    u = np.stack([u0.ravel(), u1.ravel()], axis=1)
    xs = np.full((u.shape[0], 1), x, dtype=np.int32)
    tok, n, _ = oracle.rule_batch(P, None, xs, u)
    accepted = n == 1
    assert abs(accepted.mean() - p[x]) < 1e-3
    first = tok[:, 0].copy()
    rejected = ~accepted
    emitted = np.where(accepted, x, tok[:, 0])
    # a rejected round never emits x (its residual entry is removed)
    assert not np.any(first[rejected] == x)
    law = np.bincount(emitted, minlength=5) / emitted.size
    assert np.abs(law - p).max() < 2e-3


def test_point_mass_residual_draw_by_hand():
    # p = (0.1, 0.2, 0.3, 0.4), x = 2, u0 = 0.5 >= p(2) = 0.3: rejected.
    # residual weights (0.1, 0.2, 0, 0.4), S = 0.7, C = (0.1, 0.3, 0.3, 0.7)
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.25] * 4])
    x = np.array([[2], [2]], dtype=np.int32)
    u = np.array([[0.5, 0.5],     # target 0.35 -> first C > 0.35 is v = 3
                  [0.5, 0.2]])    # target 0.14 -> v = 1
    tok, n, _ = oracle.rule_batch(p, None, x, u)
    assert n.tolist() == [0, 0]
    assert tok[:, 0].tolist() == [3, 1]
    # accepted at u0 = 0.29 < 0.3, bonus from row 1 with u1 = 0.6 -> v = 2
    tok, n, _ = oracle.rule_batch(p, None, x[:1], np.array([[0.29, 0.6]]))
    assert n.tolist() == [1] and tok[0].tolist() == [2, 2]


def test_short_draft_ends_the_walk_and_draws_the_bonus_from_its_row():
    V, K = 6, 4
    p = np.full((K + 1, V), 1.0 / V)
    p[2] = 0.0
    p[2, 5] = 1.0                          # row 2 is a point mass at 5
    x = np.array([[1, 4, -1, -1]], dtype=np.int32)
    u = np.array([[0.01, 0.01, 0.9, 0.9, 0.3]])  # both proposals survive
    tok, n, _ = oracle.rule_batch(p, None, x, u)
    assert n.tolist() == [2] and tok[0].tolist() == [1, 4, 5, -1, -1]
    # a -1 must end the draft: a later token is an invalid draft
    tok, n, _ = oracle.rule_batch(p, None, np.array([[1, -1, 4, -1]], np.int32), u)
    assert n.tolist() == [-1]
    # with a draft distribution, -1 is never a terminator
    q = np.full((K, V), 1.0 / V)
    tok, n, _ = oracle.rule_batch(p, q, x, u)
    assert n.tolist() == [-1]


def test_short_draft_in_greedy_mode(golden):
    """The greedy worked example with the draft cut after two tokens: both
    match the target's argmax, so the round emits them and the argmax of
    target row 2."""
    g = golden("greedy_example.json")
    V, K = g["V"], len(g["draft"])
    W = np.eye(V, dtype=np.float32)
    H = np.zeros((1, K + 1, V), dtype=np.float32)
    H[0, np.arange(K + 1), np.array(g["target_argmax"])] = 1.0
    draft = np.array([g["draft"][:2] + [-1] * (K - 2)], dtype=np.int32)
    ref = oracle.verify(H, W, draft, None, None, 0.0)
    want = g["target_argmax"][:3] + [-1] * (K + 1 - 3)
    assert g["draft"][:2] == g["target_argmax"][:2]
    assert ref["tokens"][0].tolist() == want and ref["n_accepted"][0] == 2


def test_verify_without_q_matches_softmax_and_the_point_mass_rule():
    rng = np.random.default_rng(3)
    V, d, K, T = 50, 8, 3, 0.8
    W = rng.standard_normal((V, d)).astype(np.float32)
    H = rng.standard_normal((1, K + 1, d)).astype(np.float32)
    L = oracle.logits(H[0], W)
    p = np.stack([oracle.softmax(L[i], T) for i in range(K + 1)])
    for seed in range(20):
        r = np.random.default_rng(100 + seed)
        x = r.integers(0, V, size=(1, K)).astype(np.int32)
        if seed % 3 == 0:
            x[0, 2:] = -1
        u = (r.integers(0, 1 << 24, size=(1, K + 1)) * 2.0 ** -24).astype(np.float32)
        got = oracle.verify(H, W, x, None, u, T)
        tok, n, _ = oracle.rule_batch(p, None, x, u.astype(np.float64))
        assert np.array_equal(got["tokens"], tok) and np.array_equal(got["n_accepted"], n)


def test_ngram_drafts_by_hand(golden):
    g = golden("ngram_examples.json")
    for c in g["cases"]:
        draft, n = oracle.ngram_draft(np.array([c["tokens"]]), [c["length"]], c["K"],
                                      c["n_min"], c["n_max"])
        assert draft[0].tolist() == c["draft"], c["name"]
        assert int(n[0]) == c["n"], c["name"]


def test_ngram_drafts_brute_force_properties():
    """On random small contexts: the draft follows an occurrence of the
    chosen suffix, no longer suffix has an occurrence, and no later
    occurrence of the chosen one exists."""
    rng = np.random.default_rng(5)
    B, L, K = 300, 40, 4
    ctx = rng.integers(0, 4, size=(B, L)).astype(np.int32)
    lens = rng.integers(1, L + 1, size=B).astype(np.int32)
    draft, n = oracle.ngram_draft(ctx, lens, K, 2, 5)

    def occ(t, m):
        ln = len(t)
        pat = t[ln - m:]
        return [j for j in range(0, ln - m) if list(t[j:j + m]) == list(pat)]

    for b in range(B):
        t = ctx[b, :lens[b]]
        chosen = None
        for m in range(5, 1, -1):
            if m < len(t) and occ(t, m):
                chosen = m
                break
        if chosen is None:
            assert n[b] == 0 and np.all(draft[b] == -1)
            continue
        j = max(occ(t, chosen))
        want = list(t[j + chosen: j + chosen + K])
        assert n[b] == len(want) >= 1
        assert draft[b].tolist() == want + [-1] * (K - len(want))
