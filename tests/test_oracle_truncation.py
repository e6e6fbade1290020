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
