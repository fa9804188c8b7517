"""Pins of the oracle router: the pages' worked examples, brute-force enumeration of
group-limited top-k on tiny inputs, the textbook top-k special case, gates summing to
1, bias entering only the selection, at most M groups per token, tie rules, sigmoid
against scipy, and the bias update's closed form and balancing behaviour."""

import itertools
import json
import os

import numpy as np
import scipy.special

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def test_bias_selection_worked_example():
    g = GOLD["bias_selection"]
    s = np.array([g["affinity"]], np.float32)
    b = np.array(g["bias"], np.float32)
    idx, gate = oracle.route(s, b, 1, 1, g["k"], g["k"], scores_are_affinities=True)
    assert sorted(idx[0] + 1) == g["chosen_one_based"]
    assert np.allclose(s[0] + b, g["selection_scores"], atol=1e-6)
    # the gates use the original affinities 0.80 and 0.60, not the biased 0.65
    assert list(np.round(gate[0], g["gate_decimals"])) == g["gates_approx"]
    idx0, _ = oracle.route(s, np.zeros(4, np.float32), 1, 1, 2, 2, scores_are_affinities=True)
    assert sorted(idx0[0] + 1) == g["chosen_without_bias_one_based"]


def test_toy_mixture_worked_example():
    g = GOLD["toy_mixture"]
    s = np.array([g["affinity"]], np.float32)
    idx, gate = oracle.route(s, np.zeros(4, np.float32), 1, 1, 2, g["k"],
                             scores_are_affinities=True)
    assert sorted(idx[0] + 1) == g["chosen_one_based"]
    assert list(np.round(gate[0], g["gate_decimals"])) == g["gates_approx"]
    Y = np.array(g["expert_outputs"], np.float32)[:, None]              # one output column
    y = oracle.combine(Y, np.array([[0, 1]], np.int32), gate, shared_row_base=-1)
    assert abs(float(y[0, 0]) - g["routed_contribution_approx"]) < 1e-6


def _brute_force(c, n_groups, M, n_top, K):
    """Selection by exhaustive search: the best M-group set maximises the total group
    score, a group's score being the largest sum over its n_top-subsets; the chosen
    experts are the K-subset of allowed experts with the largest total score."""
    E = len(c)
    gs = E // n_groups
    gscore = [max(sum(float(c[g * gs + j]) for j in sub)
                  for sub in itertools.combinations(range(gs), n_top)) for g in range(n_groups)]
    best_groups = max(itertools.combinations(range(n_groups), M),
                      key=lambda gset: sum(gscore[g] for g in gset))
    allowed = [e for e in range(E) if e // gs in best_groups]
    best = max(itertools.combinations(allowed, K), key=lambda sub: sum(float(c[e]) for e in sub))
    return set(best), set(best_groups)


def test_route_matches_brute_force():
    rng = np.random.default_rng(0)
    for (E, G, M, K) in [(16, 4, 2, 4), (12, 4, 3, 3), (16, 8, 2, 4), (8, 2, 1, 2)]:
        n_top = max(1, K // M)
        z = rng.standard_normal((40, E)).astype(np.float32) * 2
        b = (rng.uniform(-0.3, 0.3, E)).astype(np.float32)
        idx, gate = oracle.route(z, b, G, M, n_top, K)
        s = oracle.sigmoid_f32(z)
        c = (s + b).astype(np.float32)
        for t in range(40):
            chosen, groups = _brute_force(c[t], G, M, n_top, K)
            assert set(idx[t]) == chosen
            assert {e // (E // G) for e in idx[t]} <= groups


def test_group_score_over_every_expert_of_the_group():
    # the variant that scores a group by the sum of all its members' scores is the
    # group_topn = E / n_groups case; pinned against exhaustive search
    rng = np.random.default_rng(2)
    for (E, G, M, K) in [(16, 4, 2, 4), (12, 3, 2, 3), (16, 8, 3, 5)]:
        z = rng.standard_normal((40, E)).astype(np.float32) * 2
        b = (rng.uniform(-0.3, 0.3, E)).astype(np.float32)
        idx, _ = oracle.route(z, b, G, M, E // G, K)
        c = (oracle.sigmoid_f32(z) + b).astype(np.float32)
        for t in range(40):
            chosen, groups = _brute_force(c[t], G, M, E // G, K)
            assert set(idx[t]) == chosen
            gs = E // G
            sums = [float(c[t, g * gs:(g + 1) * gs].astype(np.float64).sum()) for g in range(G)]
            assert groups == set(sorted(range(G), key=lambda g: (-sums[g], g))[:M])


def test_no_group_limit_reduces_to_textbook_topk():
    rng = np.random.default_rng(1)
    s = rng.uniform(0, 1, (64, 32)).astype(np.float32)
    idx, _ = oracle.route(s, np.zeros(32, np.float32), 4, 4, 2, 6, scores_are_affinities=True)
    ref = np.argsort(-s, axis=1, kind="stable")[:, :6]
    assert (idx == ref).all()


def test_gates_sum_to_one_and_at_most_M_groups():
    rng = np.random.default_rng(2)
    E, G, M, K = 64, 8, 4, 8
    z = rng.standard_normal((200, E)).astype(np.float32) * 3
    b = rng.uniform(-0.01, 0.01, E).astype(np.float32)
    idx, gate = oracle.route(z, b, G, M, K // M, K)
    assert (np.abs(gate.astype(np.float64).sum(1) - 1) <= K * 2.0 ** -23).all()
    groups = idx // (E // G)
    assert max(len(set(r)) for r in groups) <= M
    assert all(len(set(r)) == K for r in idx)                      # distinct experts
    s = oracle.sigmoid_f32(z)
    ratio = gate[:, 0].astype(np.float64) / gate[:, 1]
    srat = np.take_along_axis(s, idx[:, :1], 1)[:, 0].astype(np.float64) / np.take_along_axis(s, idx[:, 1:2], 1)[:, 0]
    assert np.allclose(ratio, srat, rtol=1e-6)                     # gates proportional to s


def test_bias_only_changes_selection_never_gate_values():
    rng = np.random.default_rng(3)
    E = 32
    z = rng.standard_normal((300, E)).astype(np.float32)
    b = rng.uniform(-0.05, 0.05, E).astype(np.float32)
    idx_b, gate_b = oracle.route(z, b, 4, 2, 2, 4)
    idx_0, gate_0 = oracle.route(z, np.zeros(E, np.float32), 4, 2, 2, 4)
    same = np.array([set(a) == set(c) for a, c in zip(idx_b, idx_0)])
    assert same.mean() > 0.3 and (~same).any()
    for t in np.nonzero(same)[0]:
        gb = dict(zip(idx_b[t], gate_b[t]))
        g0 = dict(zip(idx_0[t], gate_0[t]))
        assert all(abs(gb[e] - g0[e]) <= 2 * 2.0 ** -24 for e in gb)
    # a bias shared by every expert changes nothing
    idx_c, gate_c = oracle.route(z, np.full(E, 0.25, np.float32), 4, 2, 2, 4)
    assert (idx_c == idx_0).all() and (gate_c == gate_0).all()


def test_ties_go_to_lower_index():
    z = np.zeros((1, 8), np.float32)
    z[0, [1, 3, 5, 6]] = 40.0                       # sigmoid saturates to exactly 1.0f
    assert oracle.sigmoid_f32(np.float32(40.0)) == 1.0
    idx, gate = oracle.route(z, np.zeros(8, np.float32), 2, 2, 1, 3)
    assert list(idx[0]) == [1, 3, 5]
    assert (gate == np.float32(1.0) / np.float32(3.0)).all()
    # groups with equal scores: the lower group wins
    idx, _ = oracle.route(z, np.zeros(8, np.float32), 4, 1, 1, 2)
    assert list(idx[0]) == [1, 0]


def test_sigmoid_against_scipy():
    z = np.random.default_rng(4).standard_normal(100000).astype(np.float32) * 8
    ref = scipy.special.expit(z.astype(np.float64)).astype(np.float32)
    assert (oracle.sigmoid_f32(z) == ref).all()
    assert oracle.sigmoid_f32(np.float32(0)) == 0.5


def test_bias_update_closed_form():
    T, K, E = 10, 4, 8                               # mean load 5
    counts = np.array([5, 6, 4, 0, 40, 5, 0, 0], np.int32)
    b = np.array([0.5, 0, 0, -1, 1e-3, 1e8, 0, 0], np.float32)
    nb = oracle.bias_update(b, counts, T, K, 0.001)
    g = np.float32(0.001)
    expect = np.array([0.5, -g, g, np.float32(-1) + g, 0.0, 1e8, g, g], np.float32)
    assert (nb == expect).all()


def test_bias_update_balances_a_skewed_router():
    """Repeated route -> count -> update shrinks the max/min load spread (the page's
    thermostat behaviour), while the gates stay the normalised affinities."""
    rng = np.random.default_rng(5)
    T, E, K = 512, 16, 2
    pref = np.log(1.0 / np.arange(1, E + 1) ** 1.1)          # Zipf-skewed demand
    z = (rng.standard_normal((T, E)) * 0.5 + pref).astype(np.float32)
    b = np.zeros(E, np.float32)
    spread = []
    for _ in range(60):
        idx, _ = oracle.route(z, b, 1, 1, K, K)
        counts = np.bincount(idx.reshape(-1), minlength=E)
        spread.append(counts.max() / max(counts.min(), 1))
        b = oracle.bias_update(b, counts, T, K, 0.02)
    assert spread[0] > 4 and np.mean(spread[-10:]) < spread[0] / 2


# ---- router logits z = x . E^T ([book] ch. 7 "The router's affinity scores") ----------

def test_router_logits_hand_worked_non_square():
    # d = 5 channels, E = 3 centroids; every product and sum is exact in float32
    x = np.array([[1, 2, 0, -1, 3], [0, 0, 4, 0, 0]], np.float32)
    cen = np.array([[1, 0, 0, 0, 0], [0, 1, 1, 0, 0], [2, -1, 0, 1, 0.5]], np.float32)
    z = oracle.router_logits(x, cen)
    assert z.shape == (2, 3) and z.dtype == np.float32
    # worked by hand: row 0: 1; 2 + 0; 2 - 2 + 0 - 1 + 1.5.  row 1: 0; 4; 0
    assert z.tolist() == [[1.0, 2.0, 0.5], [0.0, 4.0, 0.0]]
    # the operands are not interchangeable: [T, d] . [E, d]^T with T != E and d != E
    try:
        zz = oracle.router_logits(cen, x)
    except ValueError:
        zz = None
    assert zz is None or zz.shape != z.shape


def test_router_logits_one_hot_rows_pick_centroid_entries():
    rng = np.random.default_rng(3)
    E, d = 16, 384
    cen = (rng.standard_normal((E, d)) * 0.02).astype(np.float32)
    chans = np.array([0, 5, 127, 128, 383])
    x = np.zeros((len(chans), d), np.float32)
    x[np.arange(len(chans)), chans] = 1.0
    z = oracle.router_logits(x, cen)
    assert np.array_equal(z, cen[:, chans].T)            # exactly the centroid entries


def test_router_logits_constant_row_is_scaled_centroid_sum():
    import math
    rng = np.random.default_rng(4)
    E, d = 8, 512
    cen = (rng.standard_normal((E, d)) * 0.02).astype(np.float32)
    alpha = 0.75
    x = np.full((1, d), alpha, np.float32)
    z = oracle.router_logits(x, cen)
    want = np.array([math.fsum(alpha * float(v) for v in cen[i]) for i in range(E)])
    # fsum is the exact sum; the oracle rounds its float64 sum once to float32
    assert np.allclose(z[0], want.astype(np.float32), rtol=2 ** -22, atol=0)


def test_router_logits_additive_in_x():
    rng = np.random.default_rng(5)
    E, d = 4, 256
    # small integers: every product and partial sum is exact
    cen = rng.integers(-8, 9, (E, d)).astype(np.float32)
    x1 = rng.integers(-4, 5, (3, d)).astype(np.float32)
    x2 = rng.integers(-4, 5, (3, d)).astype(np.float32)
    assert np.array_equal(oracle.router_logits(x1 + x2, cen),
                          oracle.router_logits(x1, cen) + oracle.router_logits(x2, cen))


def test_route_scale_multiplies_gates_only():
    """The release config's routed scaling factor ([book] ch. 3 and ch. 7: 2.5) multiplies
    the normalised gates and nothing else: the same experts in the same order, and every
    gate equal to fl32(2.5 * the unscaled gate), so the gates sum to 2.5 (within the
    float32 rounding of K products)."""
    rng = np.random.default_rng(12)
    T, E, G, M, K = 64, 32, 8, 4, 8
    s = rng.uniform(0, 1, (T, E)).astype(np.float32)
    b = rng.uniform(-0.01, 0.01, E).astype(np.float32)
    i1, g1 = oracle.route(s, b, G, M, K // M, K, scores_are_affinities=True)
    i25, g25 = oracle.route(s, b, G, M, K // M, K, route_scale=2.5, scores_are_affinities=True)
    assert np.array_equal(i1, i25)
    assert np.array_equal(g25, (g1 * np.float32(2.5)).astype(np.float32))
    assert np.allclose(g25.astype(np.float64).sum(1), 2.5, atol=K * 2.5 * 2.0 ** -23)
