"""Pins of the oracle's truncated sampling (reading R11): hand-derived kept
sets, the untruncated special case (the plain rule, pinned by the pages'
worked examples), the top-1 special case (the pages' greedy corollary:
point-mass distributions turn the rule into greedy verification), and the
method's exactness for the warped target over a grid of uniforms
("Speculative Decoding: Two Models, One Voice", three remarks: warping
before forming p and q preserves exactness for the warped target)."""
import numpy as np

import oracle


def _embed(L):
    """hidden rows e_i and W = L^T: the logits of row i are L[i]."""
    R, V = L.shape
    W = np.ascontiguousarray(L.T, dtype=np.float32)
    H = np.eye(R, dtype=np.float32)[None]
    return H, W


def test_kept_sets_by_hand(golden):
    g = golden("truncation_examples.json")
    for c in g["cases"]:
        p, keep, gap, margin = oracle.truncate(np.array(c["logits"]), c["T"], c["top_k"],
                                               c["top_p"])
        assert np.flatnonzero(keep).tolist() == c["keep"], c["name"]
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p[~keep] == 0.0)
        x = np.array(c["logits"]) / c["T"]
        kept = x[keep]
        assert np.allclose(p[keep], np.exp(kept - kept.max()) / np.exp(kept - kept.max()).sum())
        if "gap" in c:
            assert abs(gap - c["gap"]) < 1e-12


def test_cut_description_by_hand(golden):
    """The final cut's description: the kept token with the smallest logit
    (the last in descending order, ties by index), the dropped token with
    the largest, and the former's logit."""
    g = golden("truncation_examples.json")
    for c in g["cases"]:
        L = np.array(c["logits"])
        _, keep, _, _, cut, a0, a1 = oracle.truncate(L, c["T"], c["top_k"], c["top_p"], cut=True)
        if keep.all():
            assert (cut, a0, a1) == (-np.inf, -1, -1), c["name"]
            continue
        kept, dropped = np.flatnonzero(keep), np.flatnonzero(~keep)
        lo = kept[L[kept] == L[kept].min()].max()
        hi = dropped[L[dropped] == L[dropped].max()].min()
        assert (a0, a1) == (lo, hi), c["name"]
        assert abs(cut - L[lo]) <= 1e-12 * max(1.0, abs(L[lo]))


def test_no_cut_is_the_plain_rule():
    rng = np.random.default_rng(2)
    V, K, B = 40, 3, 30
    L = rng.standard_normal((B * (K + 1), V)) * 2.0
    ql = (L.reshape(B, K + 1, V)[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    W = rng.standard_normal((V, 8)).astype(np.float32)
    H = rng.standard_normal((B, K + 1, 8)).astype(np.float32)
    x = rng.integers(0, V, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    for T in (1.0, 0.6):
        ref = oracle.verify(H, W, x, ql, u, T)
        got = oracle.verify_truncated(H, W, x, ql, u, T, 0, 1.0, 0, 1.0)
        assert np.array_equal(ref["tokens"], got["tokens"])
        assert np.array_equal(ref["n_accepted"], got["n_accepted"])
        got_v = oracle.verify_truncated(H, W, x, ql, u, T, V, 1.0, V + 5, 1.0)  # k >= V
        assert np.array_equal(ref["tokens"], got_v["tokens"])


def test_top_one_on_both_sides_is_greedy_verification():
    rng = np.random.default_rng(4)
    V, K, B = 25, 4, 60
    L = rng.standard_normal((B, K + 1, V)) * 3.0
    H = np.zeros((B, K + 1, V), dtype=np.float32)
    W = np.eye(V, dtype=np.float32)
    H[:] = L.astype(np.float32)
    ql = (L[:, :K] + rng.standard_normal((B, K, V)) * 2.0).astype(np.float32)
    # a top-1 draft proposes its argmax
    x = np.argmax(ql, axis=-1).astype(np.int32)
    greedy = oracle.verify(H, W, x, None, None, 0.0)
    for trial in range(5):
        u = rng.random((B, K + 1)).astype(np.float32)
        got = oracle.verify_truncated(H, W, x, ql, u, 1.0, 1, 1.0, 1, 1.0)
        assert np.array_equal(got["tokens"], greedy["tokens"])
        assert np.array_equal(got["n_accepted"], greedy["n_accepted"])


def test_emitted_law_is_the_warped_target():
    """K = 1: averaging the emitted token over x ~ q_w (exactly) and a grid
    of uniforms gives p_w, the truncated target."""
    lp = np.array([[1.2, 0.3, -0.4, 0.8, -1.5, 0.0], [0.0] * 6])
    lq = np.array([[0.4, 1.1, -0.2, 0.9, -0.6, 0.2]], dtype=np.float32)
    T, pk, pp, qk, qp = 0.9, 4, 0.85, 5, 0.9
    p_w, _, _, _ = oracle.truncate(lp[0], T, pk, pp)
    q_w, _, _, _ = oracle.truncate(lq[0].astype(np.float64), T, qk, qp)
    H, W = _embed(lp)
    g = (np.arange(400) + 0.5) / 400.0
    u0, u1 = np.meshgrid(g, g, indexing="ij")
    U = np.stack([u0.ravel(), u1.ravel()], axis=1).astype(np.float32)
    n = U.shape[0]
    law = np.zeros(6)
    for xv in np.flatnonzero(q_w > 0):
        got = oracle.verify_truncated(np.repeat(H, n, axis=0), W, np.full((n, 1), xv, np.int32),
                                      np.repeat(lq[None], n, axis=0), U, T, pk, pp, qk, qp)
        law += q_w[xv] * np.bincount(got["tokens"][:, 0], minlength=6) / n
    assert np.abs(law - p_w).max() < 6e-3
    assert np.all(law[p_w == 0] == 0)


def test_draft_token_cut_distance_by_hand():
    """trunc_xgap: how far a draft token's logit must move to cross its
    row's cut.  Target row 0 keeps {0,1,2} (top-3; first dropped 3 at 2.5),
    the draft row keeps {3,4,5} (last kept 3 at logit 3.0)."""
    lp = np.array([[5.0, 4.0, 3.0, 2.5, 1.0, 0.0], [0.0, 0.5, 1.0, 1.5, 2.0, 2.5]])
    lq = np.array([[[0.0, 1.0, 2.0, 3.0, 4.0, 5.0]]], dtype=np.float32)
    H, W = _embed(lp)
    u = np.full((1, 2), 0.5, np.float32)
    # token: (target side, draft side) -> the smaller
    want = {2: min(3.0 - 2.5, 3.0 - 2.0),   # kept / dropped
            0: min(5.0 - 2.5, 3.0 - 0.0),   # kept / dropped
            3: min(3.0 - 2.5, 3.0 - 2.0),   # dropped / kept
            5: min(3.0 - 0.0, 5.0 - 2.0)}   # dropped / kept
    for xv, d in want.items():  # fp32-exact logits
        got = oracle.verify_truncated(H, W, np.array([[xv]], np.int32), lq, u, 1.0, 3, 1.0, 3,
                                      1.0, 4e-6, 4e-6)
        assert abs(got["trunc_xgap"][0] - d) < 1e-12, (xv, got["trunc_xgap"][0], d)
        assert got["trunc_sens"][0] == 0.0
    # a top-p cut that lands on a cumulative mass of exactly top_p (up to
    # rounding): the last kept and first dropped tokens are at distance 0,
    # and their masses are reported as sensitivity (logits rounded to fp32)
    P = np.array([0.5, 0.3, 0.2])
    lp2 = np.log(np.stack([P, P]))
    H2, W2 = _embed(lp2)
    lq2 = np.zeros((1, 1, 3), np.float32)
    u2 = np.full((1, 2), 0.5, np.float32)
    for xv, d in ((1, 0.0), (2, 0.0), (0, np.log(0.5 / 0.2))):
        got = oracle.verify_truncated(H2, W2, np.array([[xv]], np.int32), lq2, u2, 1.0, 0, 0.8,
                                      0, 1.0, 4e-6, 4e-6)
        assert abs(got["trunc_xgap"][0] - d) < 1e-6, (xv, got["trunc_xgap"][0], d)
        assert abs(got["trunc_sens"][0] - 0.375) < 1e-7  # 0.3 / (0.5 + 0.3), kept
