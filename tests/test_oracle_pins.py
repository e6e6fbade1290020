"""Pins for the CPU oracle, against what the pages and the mathematics fix.

Each test names the page passage it checks.  The oracle is treated as a
black box: it is fed inputs and its outputs are compared with printed
values, closed forms, exact grid quadratures, library routines and Monte
Carlo bounds, so that a dropped term, a wrong sign, a swapped p/q or an
off-by-one index in it fails at least one test here.
"""
import math

import numpy as np
import pytest

import oracle


def midgrid(n):
    return (np.arange(n, dtype=np.float64) + 0.5) / n


def bf16_bits(x):
    """Round float32 values to bf16 (round to nearest even), as bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> 16) & np.uint32(1))) >> 16
    return rounded.astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Step 1: LM-head contraction
# --------------------------------------------------------------------------

def test_logits_basis_rows_select_hidden_entries():
    # W[v] = e_{v mod d}: logit (r, v) must be H[r, v mod d] exactly.  V != d
    # and R != d, so a transposed operand or a dropped last k fails.
    rng = np.random.default_rng(1)
    R, d, V = 3, 5, 12
    H = rng.standard_normal((R, d)).astype(np.float32)
    W = np.zeros((V, d), dtype=np.float32)
    W[np.arange(V), np.arange(V) % d] = 1.0
    L = oracle.logits(H, W)
    assert L.shape == (R, V)
    np.testing.assert_array_equal(L, H.astype(np.float64)[:, np.arange(V) % d])


def test_logits_bf16_bit_patterns_decode_exactly():
    # d = 1, H = 1.0: each logit is one W entry, widened from its bf16 bits.
    bits = np.array([[0x3F80], [0xC000], [0x0001], [0x4049], [0x7F7F], [0x8000]],
                    dtype=np.uint16)
    H = np.array([[0x3F80]], dtype=np.uint16)
    L = oracle.logits(H, bits)[0]
    assert L[0] == 1.0 and L[1] == -2.0
    assert L[2] == 2.0 ** -133
    assert L[3] == 3.140625
    assert L[4] == (2 - 2.0 ** -7) * 2.0 ** 127
    assert L[5] == 0.0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_logits_match_library_matmul(dtype):
    rng = np.random.default_rng(2)
    R, d, V = 5, 256, 300
    Hf = rng.standard_normal((R, d)).astype(np.float32)
    Wf = (0.02 * rng.standard_normal((V, d))).astype(np.float32)
    if dtype == "bf16":
        H, W = bf16_bits(Hf), bf16_bits(Wf)
        H64, W64 = bf16_value(H), bf16_value(W)
    else:
        H, W = Hf, Wf
        H64, W64 = Hf.astype(np.float64), Wf.astype(np.float64)
    L = oracle.logits(H, W)
    ref = H64 @ W64.T
    bound = 1e-13 * (np.abs(H64) @ np.abs(W64).T)
    assert np.all(np.abs(L - ref) <= bound)


def test_logits_vocab_slice_and_row_permutation():
    rng = np.random.default_rng(3)
    R, d, V = 4, 64, 97
    H = bf16_bits(rng.standard_normal((R, d)))
    W = bf16_bits(0.02 * rng.standard_normal((V, d)))
    full = oracle.logits(H, W)
    np.testing.assert_array_equal(oracle.logits(H, W, 10, 60), full[:, 10:60])
    perm = rng.permutation(V)
    np.testing.assert_array_equal(oracle.logits(H, W[perm]), full[:, perm])


# --------------------------------------------------------------------------
# Step 2: temperature softmax
# --------------------------------------------------------------------------

def test_softmax_recovers_a_distribution_from_its_logs(golden):
    g = golden("six_token_example.json")
    P = np.array(g["p"])
    np.testing.assert_allclose(oracle.softmax(np.log(P)), P, rtol=0, atol=1e-15)
    # shifting the logits by a constant changes nothing
    np.testing.assert_allclose(oracle.softmax(np.log(P) + 40.0), P, rtol=0,
                               atol=1e-15)


@pytest.mark.parametrize("T", [0.25, 0.7, 1.0, 2.0])
def test_softmax_two_tokens_is_the_logistic_function(T):
    for a in (-3.0, -0.1, 0.0, 0.5, 7.0):
        p = oracle.softmax(np.array([0.0, a]), T)
        want = 1.0 / (1.0 + math.exp(-a / T))
        assert abs(p[1] - want) < 1e-14  # exp of an argument near 28: a few ulp
        assert abs(p[0] + p[1] - 1.0) < 1e-14


def test_lse_closed_forms():
    assert abs(oracle.lse(np.full(1000, 2.0), 0.5) - (4.0 + math.log(1000))) < 1e-12
    # large logits do not overflow
    assert abs(oracle.lse(np.array([1000.0, 1000.0]), 1.0) - (1000 + math.log(2))) < 1e-12
    x = np.random.default_rng(4).standard_normal(50)
    assert abs(oracle.lse(x + 3.0, 2.0) - (oracle.lse(x, 2.0) + 1.5)) < 1e-13


# --------------------------------------------------------------------------
# Steps 3-5: the rule on the pages' worked examples
# --------------------------------------------------------------------------

N_GRID = 1 << 20


def accept_fraction(P, Q, x):
    """Fraction of a midpoint grid of u_1 values that accepts token x (K=1)."""
    u = np.stack([midgrid(N_GRID), np.full(N_GRID, 0.5)], axis=1)
    xs = np.full((N_GRID, 1), x, dtype=np.int32)
    p = np.stack([P, P])
    _, n_acc, _ = oracle.rule_batch(p, Q[None, :], xs, u)
    return float(np.mean(n_acc == 1))


def final_draw_law(P, Q, x, u1):
    """Law of the final token over a midpoint grid of u_f, for fixed x, u_1."""
    u = np.stack([np.full(N_GRID, u1), midgrid(N_GRID)], axis=1)
    xs = np.full((N_GRID, 1), x, dtype=np.int32)
    tokens, n_acc, _ = oracle.rule_batch(np.stack([P, P]), Q[None, :], xs, u)
    slot = int(n_acc[0])
    assert np.all(n_acc == slot)
    return np.bincount(tokens[:, slot], minlength=len(P)) / N_GRID, slot


def test_six_token_alpha_and_emitted_law(golden):
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    law, alpha = oracle.emitted_law(P, Q)
    assert round(alpha, g["alpha_printed_decimals"]) == g["alpha_printed"]
    np.testing.assert_allclose(law, P, rtol=0, atol=1e-15)


def test_six_token_accept_probabilities_on_a_grid(golden):
    # accept x with probability min(1, p(x)/q(x))
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    for x in range(len(P)):
        assert abs(accept_fraction(P, Q, x) - min(1.0, P[x] / Q[x])) <= 1.0 / N_GRID


def test_six_token_residual_on_a_grid(golden):
    # after a rejection the replacement follows norm(max(0, p - q)); the
    # figure prints 0.53, 0.11, 0.37 on the three under-weighted tokens
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    resid = np.maximum(P - Q, 0.0)
    resid /= resid.sum()
    printed = g["residual_printed"]
    for x in (0, 4, 5):  # every token that can be rejected (q > p)
        u1 = 0.5 * (P[x] / Q[x] + 1.0)  # strictly above the threshold
        law, slot = final_draw_law(P, Q, x, u1)
        assert slot == 0
        assert np.max(np.abs(law - resid)) <= 2.0 / N_GRID
        for i, v in zip(printed["indices"], printed["values"]):
            assert round(law[i], printed["decimals"]) == v
        assert law[0] == 0 and law[4] == 0 and law[5] == 0


def test_six_token_bonus_draw_follows_p(golden):
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    law, slot = final_draw_law(P, Q, 1, 0.999)  # token 1 has p > q: always kept
    assert slot == 1
    assert np.max(np.abs(law - P)) <= 2.0 / N_GRID


def test_six_token_joint_grid_reproduces_p(golden):
    # black-box quadrature over x ~ q and a joint (u_1, u_f) grid: no
    # assumption about which uniform drives which decision
    g = golden("six_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    n = 1 << 9
    u1, uf = np.meshgrid(midgrid(n), midgrid(n), indexing="ij")
    u = np.stack([u1.ravel(), uf.ravel()], axis=1)
    law = np.zeros(len(P))
    for x in range(len(P)):
        xs = np.full((n * n, 1), x, dtype=np.int32)
        tokens, _, _ = oracle.rule_batch(np.stack([P, P]), Q[None, :], xs, u)
        law += Q[x] * np.bincount(tokens[:, 0], minlength=len(P)) / (n * n)
    assert np.max(np.abs(law - P)) <= (len(P) + 2) / n


def _mc(P, Q, K, n, seed, u_dtype=np.float64):
    rng = np.random.default_rng(seed)
    x = rng.choice(len(Q), p=Q, size=(n, K)).astype(np.int32)
    u = rng.random((n, K + 1)).astype(u_dtype).astype(np.float64)
    p = np.tile(P, (K + 1, 1))
    q = np.tile(Q, (K, 1))
    return oracle.rule_batch(p, q, x, u)


def _round_length_var(alpha, K):
    ks = np.arange(1, K + 2)
    probs = np.array([alpha ** (k - 1) * (1 - alpha) for k in range(1, K + 1)]
                     + [alpha ** K])
    mean = float(np.sum(ks * probs))
    return mean, float(np.sum((ks - mean) ** 2 * probs))


def test_six_token_monte_carlo_two_million_rounds(golden):
    # the pages' simulation (200k rounds, K = 4) scaled to 2M rounds so that
    # a correct sampler's TV sits well below 1e-3
    from scipy import stats
    g = golden("six_token_example.json")
    P, Q, K = np.array(g["p"]), np.array(g["q"]), g["K"]
    tokens, n_acc, _ = _mc(P, Q, K, 2_000_000, seed=11, u_dtype=np.float32)
    emitted = tokens[tokens >= 0]
    counts = np.bincount(emitted, minlength=len(P))
    emp = counts / counts.sum()
    tv = 0.5 * np.abs(emp - P).sum()
    assert tv < 1e-3
    chi2 = stats.chisquare(counts, counts.sum() * P)
    assert chi2.pvalue > 1e-4
    alpha = float(np.minimum(P, Q).sum())
    mean, var = _round_length_var(alpha, K)
    assert abs(mean - oracle.expected_tokens(alpha, K)) < 1e-12
    measured = float(np.mean(n_acc + 1))
    assert abs(measured - mean) < 4 * math.sqrt(var / len(n_acc))
    # every emitted sequence is an accepted prefix plus one token
    assert np.all((tokens >= 0).sum(axis=1) == n_acc + 1)


def test_six_token_printed_simulation_is_within_noise(golden):
    # the page's printed 200k-round output lies where a correct sampler puts
    # it, and so does ours
    g = golden("six_token_example.json")
    P, Q, K = np.array(g["p"]), np.array(g["q"]), g["K"]
    n = g["rounds_simulated"]
    tokens, n_acc, _ = _mc(P, Q, K, n, seed=1)
    emitted = tokens[tokens >= 0]
    emp = np.bincount(emitted, minlength=len(P)) / emitted.size
    se = np.sqrt(P * (1 - P) / emitted.size)
    assert np.all(np.abs(emp - P) < 5 * se)
    assert np.all(np.abs(np.array(g["empirical_law_printed"]) - P) < 5 * se)
    alpha = float(np.minimum(P, Q).sum())
    mean, var = _round_length_var(alpha, K)
    assert round(mean, 3) == g["tokens_per_round_formula_printed"]
    for val in (float(np.mean(n_acc + 1)), g["tokens_per_round_simulated_printed"]):
        assert abs(val - mean) < 4 * math.sqrt(var / n) + 5e-4


def test_three_token_example(golden):
    g = golden("three_token_example.json")
    P, Q = np.array(g["p"]), np.array(g["q"])
    law, alpha = oracle.emitted_law(P, Q)
    assert round(alpha, 3) == g["acceptance_printed"]
    np.testing.assert_allclose(law, P, rtol=0, atol=1e-15)
    # the over-proposed token survives 40% of the time
    grey = g["grey_index"]
    assert abs(accept_fraction(P, Q, grey) - g["grey_survival_printed"]) <= 1.0 / N_GRID
    # replacements come from blue and clear in the ratio 2:1
    u1 = 0.5 * (P[grey] / Q[grey] + 1.0)
    rlaw, _ = final_draw_law(P, Q, grey, u1)
    ratio = rlaw[g["blue_index"]] / rlaw[g["clear_index"]]
    assert abs(ratio - g["residual_ratio_blue_to_clear"]) < 1e-4
    assert rlaw[grey] == 0.0
    # 1M single-draft draws, as on the page
    tokens, n_acc, _ = _mc(P, Q, 1, g["draws_simulated"], seed=5)
    first = tokens[:, 0]
    emp = np.bincount(first, minlength=3) / len(first)
    se = np.sqrt(P * (1 - P) / len(first))
    assert np.all(np.abs(emp - P) < 4 * se)
    assert np.all(np.abs(np.array(g["law_printed"]) - P) < 4 * se)
    acc = float(np.mean(n_acc == 1))
    assert abs(acc - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / len(first))


def test_three_token_tokens_per_step_gamma3(golden):
    g = golden("three_token_example.json")
    P, Q, K = np.array(g["p"]), np.array(g["q"]), g["gamma"]
    alpha = float(np.minimum(P, Q).sum())
    assert round(oracle.expected_tokens(alpha, K), 3) == g["tokens_per_step_printed"]
    mean, var = _round_length_var(alpha, K)
    _, n_acc, _ = _mc(P, Q, K, 2_000_000, seed=7)
    assert abs(float(np.mean(n_acc + 1)) - mean) < 4 * math.sqrt(var / len(n_acc))


def test_exact_law_over_random_dirichlet_pairs():
    # The Algebra and the Proof, 'The proof': the emitted law equals p to
    # rounding over 10k random pairs, and alpha = 1 - TV(p, q)
    rng = np.random.default_rng(0)
    worst = 0.0
    for _ in range(10_000):
        V = int(rng.integers(2, 50))
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V) * 0.3)
        law, alpha = oracle.emitted_law(p, q)
        assert abs(alpha - (1.0 - 0.5 * np.abs(p - q).sum())) < 1e-12
        worst = max(worst, float(np.max(np.abs(law - p))))
    assert worst < 1e-15


def test_identical_draft_edge_case():
    # p = q = [1, 0]: alpha = 1, the residual is empty, and the sampler never
    # divides by zero; every proposal is kept and the bonus is token 0
    p = np.array([1.0, 0.0])
    law, alpha = oracle.emitted_law(p, p)
    assert alpha == 1.0
    np.testing.assert_array_equal(law, p)
    n = 4096
    u = np.stack([midgrid(n), midgrid(n)[::-1]], axis=1)
    tokens, n_acc, _ = oracle.rule_batch(np.stack([p, p]), p[None, :],
                                         np.zeros((n, 1), np.int32), u)
    assert np.all(n_acc == 1) and np.all(tokens == 0)


def test_zero_draft_probability_enters_through_the_residual():
    # The Algebra and the Proof, 'Where it breaks': tokens with q = 0, p > 0
    # cannot be proposed and are delivered by the residual
    P, Q = np.array([0.5, 0.5]), np.array([1.0, 0.0])
    law, alpha = oracle.emitted_law(P, Q)
    assert alpha == 0.5
    np.testing.assert_array_equal(law, P)
    assert abs(accept_fraction(P, Q, 0) - 0.5) <= 1.0 / N_GRID
    rlaw, _ = final_draw_law(P, Q, 0, 0.75)
    np.testing.assert_array_equal(rlaw, [0.0, 1.0])
    # a token with q = 0 and p > 0 that is forced in is accepted
    assert accept_fraction(P, Q, 1) == 1.0


def test_strict_accept_test_and_threshold_distance():
    P, Q = np.array([0.5, 0.5]), np.array([1.0, 0.0])
    tokens, n_acc, dist = oracle.rule_batch(np.stack([P, P]), Q[None, :],
                                            np.zeros((2, 1), np.int32),
                                            np.array([[0.5, 0.2], [0.4999, 0.2]]))
    assert n_acc[0] == 0 and tokens[0, 0] == 1 and dist[0] == 0.0
    assert n_acc[1] == 1 and tokens[1, 0] == 0
    assert abs(dist[1] - 1e-4) < 1e-12


def test_threshold_distance_parts():
    # The round's distance splits into its accept tests (|u_i - p/q|) and its
    # final draw (the chosen token's CDF interval edges).  Two-token p, q:
    # t = p(0)/q(0) = 0.5 for draft token 0; the bonus is drawn from p with
    # edges 0, 0.5, 1; after a rejection the residual max(0, p - q) = (0, 0.5)
    # normalises to (0, 1), edges 0 and 1.
    P, Q = np.array([0.5, 0.5]), np.array([1.0, 0.0])
    u = np.array([[0.4999, 0.2],          # accepted 1e-4 below t; bonus 0.2 into [0, 0.5)
                  [0.3, 0.5 + 3e-7],      # accepted; bonus 3e-7 above the edge at 0.5
                  [0.9, 0.75]])           # rejected 0.4 above t; residual draw at 0.75
    tokens, n_acc, dist, dacc, ddraw = oracle.rule_batch(
        np.stack([P, P]), Q[None, :], np.zeros((3, 1), np.int32), u, split=True)
    assert list(n_acc) == [1, 1, 0]
    assert tokens.tolist() == [[0, 0], [0, 1], [1, -1]]
    np.testing.assert_allclose(dacc, [1e-4, 0.2, 0.4], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ddraw, [0.2, 3e-7, 0.25], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(dist, np.minimum(dacc, ddraw))
    # no accept test at all (K = 0): only the draw counts
    _, _, dist0, dacc0, ddraw0 = oracle.rule_batch(P[None, :], None, np.zeros((1, 0), np.int32),
                                                   np.array([[0.7]]), split=True)
    assert dacc0[0] == np.inf and abs(ddraw0[0] - 0.2) < 1e-12 and dist0[0] == ddraw0[0]


def test_zero_residual_falls_back_to_p():
    # p <= q everywhere with a rejection: the residual is empty, the
    # replacement is drawn from p itself (the zero-residual fallback)
    P, Q = np.array([0.25, 0.75]), np.array([0.5, 0.75])
    u = np.array([[0.9, 0.1], [0.9, 0.6]])
    tokens, n_acc, _ = oracle.rule_batch(np.stack([P, P]), Q[None, :],
                                         np.zeros((2, 1), np.int32), u)
    assert list(n_acc) == [0, 0]
    assert list(tokens[:, 0]) == [0, 1]


def test_rows_used_by_the_residual_and_the_bonus():
    # row i of p scores draft position i+1 and row K is position K+1: a
    # rejection at position j draws from (p_j - q_j)+, a full accept draws
    # the bonus from p_{K+1} ("One speculation round", steps 3-5)
    V, K = 4, 2
    p = np.array([[0.25, 0.25, 0.25, 0.25],
                  [0.00, 0.50, 0.00, 0.50],
                  [0.00, 0.00, 1.00, 0.00]])
    q = np.array([[0.25, 0.25, 0.25, 0.25],
                  [0.50, 0.00, 0.50, 0.00]])
    u = np.array([[0.3, 0.3, 0.10],    # accept x1 (t=1), reject x2=0 (t=0)
                  [0.3, 0.3, 0.90],
                  [0.3, 0.3, 0.50]])
    x = np.array([[1, 0], [1, 0], [1, 1]], np.int32)
    tokens, n_acc, _ = oracle.rule_batch(p, q, x, u)
    assert list(n_acc) == [1, 1, 2]
    # residual of row 1 is (p1 - q1)+ = [0, .5, 0, .5]: u_f = .1 -> 1, .9 -> 3
    assert list(tokens[0]) == [1, 1, -1] and list(tokens[1]) == [1, 3, -1]
    # both accepted (x2 = 1 has q = 0, p = .5): the bonus comes from row 2
    assert list(tokens[2]) == [1, 1, 2]


def test_positionwise_acceptance_expected_tokens():
    # The Algebra and the Proof, 'The algebra': with per-position p_j, q_j
    # the mean round length is 1 + sum_i prod_{j<=i} alpha_j
    rng = np.random.default_rng(9)
    K, V, n = 3, 8, 1_000_000
    p = rng.dirichlet(np.ones(V), size=K + 1)
    q = rng.dirichlet(np.ones(V) * 0.7, size=K)
    alphas = [oracle.emitted_law(p[j], q[j])[1] for j in range(K)]
    want = oracle.expected_tokens_positions(alphas)
    x = np.stack([rng.choice(V, p=q[j], size=n) for j in range(K)], axis=1)
    u = rng.random((n, K + 1))
    _, n_acc, _ = oracle.rule_batch(p, q, x.astype(np.int32), u)
    lengths = n_acc + 1.0
    assert abs(lengths.mean() - want) < 4 * lengths.std() / math.sqrt(n)
    # with equal alphas it reduces to the i.i.d. closed form
    assert abs(oracle.expected_tokens_positions([0.7] * 3)
               - oracle.expected_tokens(0.7, 3)) < 1e-15


def test_closed_forms_printed_values(golden):
    g = golden("closed_forms.json")
    for case in g["iid"]:
        val = oracle.expected_tokens(case["alpha"], case["K"])
        assert round(val, case["decimals"]) == case["printed"], case
    cap = g["cap"]
    # the supremum 1 / (1 - alpha) is approached from below (and reached
    # only after rounding, at very long drafts)
    assert all(oracle.expected_tokens(cap["alpha"], k) < cap["bound"]
               for k in range(1, 60))
    assert abs(oracle.expected_tokens(cap["alpha"], 200) - cap["bound"]) < 1e-12
    pos = g["positions"]
    terms = [1.0] + list(np.cumprod(pos["alphas"]))
    np.testing.assert_allclose(terms, pos["terms_printed"], rtol=0, atol=1e-15)
    assert abs(oracle.expected_tokens_positions(pos["alphas"]) - pos["printed"]) < 1e-12
    assert oracle.expected_tokens(1.0, 4) == 5.0


def test_inverse_cdf_special_cases():
    # one-hot p always yields its token; uniform p over 7 tokens yields
    # floor(7 u) away from the cell edges
    n = 7 * 1000
    u = midgrid(n)[:, None]
    onehot = np.zeros((1, 9))
    onehot[0, 4] = 1.0
    tokens, n_acc, _ = oracle.rule_batch(onehot, None, None, u)
    assert np.all(tokens[:, 0] == 4) and np.all(n_acc == 0)
    flat = np.full((1, 7), 1.0 / 7)
    tokens, _, _ = oracle.rule_batch(flat, None, None, u)
    np.testing.assert_array_equal(tokens[:, 0], np.floor(7 * u[:, 0]).astype(int))


def test_out_of_range_draft_token_is_reported():
    P = np.array([0.5, 0.5])
    tokens, n_acc, _ = oracle.rule_batch(np.stack([P, P]), P[None, :],
                                         np.array([[2]], np.int32),
                                         np.array([[0.1, 0.1]]))
    assert n_acc[0] == -1 and np.all(tokens == -1)


# --------------------------------------------------------------------------
# The composed step (logits -> softmax -> rule) and the greedy rule
# --------------------------------------------------------------------------

def _embed_logits(rows_logits):
    """fp32 hidden/W such that the logits are exactly `rows_logits`:
    W = identity, hidden row i = desired logit row i."""
    R, V = rows_logits.shape
    H = rows_logits.astype(np.float32)
    W = np.eye(V, dtype=np.float32)
    return H, W


def test_greedy_worked_example(golden):
    g = golden("greedy_example.json")
    V, K = g["V"], len(g["draft"])
    L = np.zeros((K + 1, V))
    L[np.arange(K + 1), g["target_argmax"]] = 1.0
    H, W = _embed_logits(L)
    out = oracle.verify(H[None], W, np.array([g["draft"]]), None, None, 0.0)
    want = g["expected_tokens"] + [-1] * (K + 1 - len(g["expected_tokens"]))
    assert list(out["tokens"][0]) == want
    assert out["n_accepted"][0] == g["expected_n_accepted"]
    # every guess matched: the fifth pick is a free bonus
    out = oracle.verify(H[None], W, np.array([g["target_argmax"][:K]]), None, None, 0.0)
    assert list(out["tokens"][0]) == g["target_argmax"] and out["n_accepted"][0] == K
    # first guess wrong: one correction, nothing accepted
    bad = [g["target_argmax"][0] + 1] + g["draft"][1:]
    out = oracle.verify(H[None], W, np.array([bad]), None, None, 0.0)
    assert out["n_accepted"][0] == 0
    assert list(out["tokens"][0]) == [g["target_argmax"][0]] + [-1] * K


def test_greedy_ties_go_to_the_smallest_index():
    L = np.array([[0.0, 2.0, 2.0, 1.0]])
    H, W = _embed_logits(L)
    out = oracle.verify(H[None], W, np.zeros((1, 0), np.int32), None, None, 0.0)
    assert out["tokens"][0, 0] == 1 and out["dist"][0] == 0.0


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_composed_step_on_the_six_token_example(golden, T):
    # logits = T log P and q_logits = T log Q give p = P and q = Q at
    # temperature T; the composed step must then match the rule on P, Q
    g = golden("six_token_example.json")
    P, Q, K = np.array(g["p"]), np.array(g["q"]), g["K"]
    V = len(P)
    L = np.tile(T * np.log(P), (K + 1, 1))
    H, W = _embed_logits(L)
    rng = np.random.default_rng(21)
    B = 4000
    x = rng.choice(V, p=Q, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    ql = np.tile((T * np.log(Q)).astype(np.float32), (B, K, 1))
    out = oracle.verify(np.tile(H[None], (B, 1, 1)), W, x, ql, u, T)
    tokens, n_acc, dist = oracle.rule_batch(np.tile(P, (K + 1, 1)),
                                            np.tile(Q, (K, 1)), x, u.astype(np.float64))
    same = dist > 1e-9  # the step's p, q differ from P, Q by rounding only
    assert same.mean() > 0.999
    np.testing.assert_array_equal(out["tokens"][same], tokens[same])
    np.testing.assert_array_equal(out["n_accepted"][same], n_acc[same])
    # sum(P) = sum(Q) = 1, so both normalisers are log 1 = 0 up to the fp32
    # rounding of the embedded logits
    np.testing.assert_allclose(out["lse_p"], 0.0, rtol=0, atol=1e-6)
    np.testing.assert_allclose(out["lse_q"], 0.0, rtol=0, atol=1e-6)
