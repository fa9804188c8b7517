"""Pins of the oracle's sequence-wise balance statistics against what the pages and the
mathematics fix ("DeepSeek-V3" book, ch. 8, "The complementary sequence loss")."""

import numpy as np

import oracle


def test_plain_topk_matches_brute_force_and_breaks_ties_low():
    rng = np.random.default_rng(3)
    s = rng.integers(0, 4, (50, 12)).astype(np.float32) / 4      # many ties
    got = oracle.plain_topk(s, 5)
    for t in range(50):
        want = sorted(range(12), key=lambda i: (-s[t, i], i))[:5]
        assert list(got[t]) == want
    assert list(oracle.plain_topk(np.ones((1, 9), np.float32), 3)[0]) == [0, 1, 2]


def test_uniform_usage_gives_fair_share_and_loss_alpha():
    # E=8, K=2, L=4: token t picks experts 2t, 2t+1 (affinity 0.75, others 0.25), so each
    # expert is picked once: f_i = 8 * 1 / (2 * 4) = 1; D_t = 3, s' = 1/4 or 1/12, and
    # P_i = (1/4 + 3/12) / 4 = 1/8 = 1/E; loss = alpha * sum_i 1 * 1/8 = alpha
    E, K, L = 8, 2, 4
    s = np.full((L, E), 0.25, np.float32)
    for t in range(L):
        s[t, 2 * t:2 * t + 2] = 0.75
    f, P, loss = oracle.seq_balance_stats(s, K, L, alpha=1e-4, scores_are_affinities=True)
    assert np.array_equal(f, np.ones((1, E), np.float32))
    assert np.allclose(P, 1.0 / E, rtol=0, atol=1e-15)
    assert abs(loss[0] - 1e-4) < 1e-18


def test_concentrated_usage_closed_form():
    # every token puts all its mass on the same K experts: f = E/K there, P = 1/K there,
    # loss = alpha * K * (E/K) * (1/K) = alpha * E / K
    E, K, L = 16, 4, 6
    s = np.zeros((L, E), np.float32)
    s[:, [3, 7, 8, 15]] = 1.0
    f, P, loss = oracle.seq_balance_stats(s, K, L, alpha=1e-4, scores_are_affinities=True)
    assert f[0, 3] == E / K and f[0, 0] == 0
    assert P[0, 7] == 1.0 / K and P[0, 1] == 0
    assert abs(loss[0] - 1e-4 * E / K) < 1e-16


def test_hand_worked_example():
    # E=4, K=1, L=2.  Token 0 picks expert 0, token 1 picks expert 2: f = [2, 0, 2, 0].
    # D = 1.7 and 1.2; loss = alpha * 2 * (P_0 + P_2)
    #      = alpha * (0.9/1.7 + 0.1/1.2 + 0.2/1.7 + 0.6/1.2) = alpha * 1.2303921568627...
    s = np.array([[0.9, 0.5, 0.2, 0.1], [0.1, 0.3, 0.6, 0.2]], np.float32)
    f, P, loss = oracle.seq_balance_stats(s, 1, 2, alpha=1e-4, scores_are_affinities=True)
    assert np.array_equal(f[0], np.array([2, 0, 2, 0], np.float32))
    assert abs(P[0, 1] - (0.5 / 1.7 + 0.3 / 1.2) / 2) < 1e-7
    assert abs(loss[0] / 1e-4 - 1.2303921568627) < 1e-6


def test_invariants_and_sequences_are_independent():
    rng = np.random.default_rng(5)
    E, K, L, S = 64, 6, 37, 3
    z = rng.standard_normal((S * L, E)).astype(np.float32) * 3
    f, P, loss = oracle.seq_balance_stats(z, K, L, alpha=1e-4)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)          # s' sums to 1 per token
    assert np.allclose(f.astype(np.float64).sum(axis=1), E, rtol=1e-6)
    assert (f >= 0).all() and (f <= E / K).all()
    for q in range(S):                                          # one sequence at a time
        fq, Pq, lq = oracle.seq_balance_stats(z[q * L:(q + 1) * L], K, L, alpha=1e-4)
        assert np.array_equal(fq[0], f[q]) and np.array_equal(Pq[0], P[q]) and lq[0] == loss[q]
    # logits go through the router's sigmoid
    fa, Pa, la = oracle.seq_balance_stats(oracle.sigmoid_f32(z), K, L, alpha=1e-4,
                                          scores_are_affinities=True)
    assert np.array_equal(fa, f) and np.array_equal(Pa, P) and np.array_equal(la, loss)


def test_frequency_uses_plain_topk_not_the_biased_dispatch():
    # a bias that moves the router's choice does not move f: f follows the original
    # affinities' top-K over all experts
    s = np.array([[0.6, 0.8, 0.1, 0.05]], np.float32)
    bias = np.array([0.5, 0.0, 0.0, 0.0], np.float32)
    idx, _ = oracle.route(s, bias, 1, 1, 1, 1, scores_are_affinities=True)
    assert idx[0, 0] == 0                                       # router follows s + b
    f, _, _ = oracle.seq_balance_stats(s, 1, 1, scores_are_affinities=True)
    assert f[0, 1] == 4 and f[0, 0] == 0                        # f follows s alone
