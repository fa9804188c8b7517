"""Router: logits, sigmoid affinity, bias-for-selection, group-limited top-k, gates,
and the auxiliary-loss-free bias update.

Oracle module (test infrastructure only).

What the pages fix:
* affinity s_i = sigmoid(u . e_i), applied per expert, so affinities do not sum to 1
  ("DeepSeek-V3", core idea 1; DeepSeek-V3 book, ch. 7 "The router's affinity
  scores");
* gating stays in higher precision, not FP8 ("DeepSeek-V3", core idea 6; book ch. 17
  "High-precision exceptions", "Router precision has discrete consequences");
* the bias b_i enters only the selection score s_i + b_i; the gate uses the original
  s_i (book ch. 8 "V3's routing-only bias", worked example in "A selection-versus-
  weighting example"; "DeepSeek-V3: the recipe...", "Auxiliary-loss-free balancing");
* a token may use at most M groups; a group is scored by the sum of its highest K/M
  scores ("DeepSeek-V3", core idea 1 "Node-limited routing"; book ch. 8 "Restricting
  target nodes");
* gates are the chosen affinities normalised to sum to 1 (book ch. 7 "Selecting and
  combining experts", toy mixture);
* after a step, an overloaded expert's bias drops by gamma and an underloaded one's
  rises by gamma, gamma = 0.001 ("DeepSeek-V3", core idea 2; book ch. 8 "The feedback
  update"; "DeepSeek-V3: the recipe...", bias_balance_step description).

Readings taken where the pages are silent:
* the group score sums the top-n BIASED scores c = s + b (group choice is selection);
  the n values are added in float32 in descending order;
* ties in every ranking go to the lower index (groups and experts alike);
* the chosen experts are listed in descending c, which fixes the order of the gate
  denominator sum D and of the combine;
* logits z are float32; s = fl32(1 / (1 + exp(-z))) computed in float64;
  c = fl32(s + b); D = float32 running sum of the chosen s in list order;
  g = fl32(s / D), then fl32(g * route_scale) (route_scale defaults to 1);
* bias update: load_i = number of (token, slot) pairs sent to routed expert i,
  mean = T*K/E, b_i <- fl32(b_i + gamma * sign(mean - load_i)), sign(0) = 0.
"""

import numpy as np


def router_logits(x, centroids):
    """z[t, i] = fl32(sum_k x[t,k] * e_i[k]) with the sum in float64.

    x: float32 [T, d] (BF16 values), centroids: float32 [E, d].
    """
    z = np.asarray(x, dtype=np.float64) @ np.asarray(centroids, dtype=np.float64).T
    return z.astype(np.float32)


def sigmoid_f32(z):
    """fl32(1 / (1 + exp(-z))) evaluated in float64."""
    zd = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return (1.0 / (1.0 + np.exp(-zd))).astype(np.float32)


def _desc_order(values, index):
    """Positions sorting ``values`` descending, ties by ascending ``index``."""
    return np.lexsort((index, -values))


def route_token(s, c, n_groups, topk_groups, group_topn, k, route_scale=1.0):
    """Route one token.

    s, c: float32 [E] affinities and selection scores.  Returns (idx int32[k],
    gate float32[k], kept_groups int[topk_groups]).
    """
    E = s.shape[0]
    gs = E // n_groups
    gscore = np.empty(n_groups, dtype=np.float32)
    for g in range(n_groups):
        vals = c[g * gs:(g + 1) * gs]
        order = _desc_order(vals, np.arange(gs))
        acc = vals[order[0]]
        for j in order[1:group_topn]:
            acc = np.float32(acc + vals[j])
        gscore[g] = acc
    kept = _desc_order(gscore, np.arange(n_groups))[:topk_groups]
    cand = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in sorted(kept)])
    chosen = cand[_desc_order(c[cand], cand)[:k]]
    denom = s[chosen[0]]
    for i in chosen[1:]:
        denom = np.float32(denom + s[i])
    gate = (s[chosen] / denom).astype(np.float32)
    if route_scale != 1.0:
        gate = (gate * np.float32(route_scale)).astype(np.float32)
    return chosen.astype(np.int32), gate, kept


def route(scores, bias, n_groups, topk_groups, group_topn, k, route_scale=1.0,
          scores_are_affinities=False):
    """Route every token.

    scores: float32 [T, E] logits (or affinities if ``scores_are_affinities``);
    bias: float32 [E].  Returns (idx int32[T, k], gate float32[T, k]).
    """
    scores = np.asarray(scores, dtype=np.float32)
    s = scores if scores_are_affinities else sigmoid_f32(scores)
    c = (s + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    T = s.shape[0]
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        idx[t], gate[t], _ = route_token(s[t], c[t], n_groups, topk_groups, group_topn,
                                         k, route_scale)
    return idx, gate


def bias_update(bias, counts, T, k, gamma):
    """b_i <- fl32(b_i + gamma * sign(T*k/E - counts_i)); sign taken exactly in integers."""
    bias = np.asarray(bias, dtype=np.float32)
    E = bias.shape[0]
    sgn = np.sign(np.int64(T) * np.int64(k) - np.int64(E) * np.asarray(counts, np.int64))
    step = np.float64(np.float32(gamma)) * sgn.astype(np.float64)
    return (bias.astype(np.float64) + step).astype(np.float32)
