"""Sequence-wise balance statistics of the complementary balance loss (forward only).

Oracle module (test infrastructure only).

What the pages fix ("DeepSeek-V3" book, ch. 8 "Routing and Load Balancing", section
"The complementary sequence loss"; "DeepSeek-V3" summary, core idea 2, the "safety net"
paragraph):
* the loss is alpha times the sum over the N_r routed experts of f_i * P_i, with
  alpha = 0.0001 in the V3 configuration, taken over one sequence;
* f_i is expert i's frequency of selection in the sequence, scaled by N_r / K_r so
  that a fair share is 1;
* P_i is expert i's affinity normalised over all routed experts of the token,
  averaged over the sequence's tokens;
* the frequency counts selection among the ORIGINAL affinities (the plain top-K_r of
  s over all routed experts), not the biased, group-limited dispatch;
* under uniform usage every f_i is about 1 and every P_i about 1/N_r, so the sum is
  about 1.

Readings taken where the pages are silent:
* s_{i,t} is the sigmoid affinity fl32(1 / (1 + exp(-z))) (same as the router), or
  the affinity itself when affinities are given;
* the top-K_r ranking breaks ties toward the lower expert index, as the router does;
* f_i = fl32(N_r * count_i) / fl32(K_r * L) in float32 (both operands exact), where L
  is the sequence length; P_i and the loss are computed in float64;
* a batch of T tokens is T / L consecutive sequences of L tokens; the statistics are
  reported per sequence (the pages do not say how sequences are combined).
"""

import numpy as np

from .router import sigmoid_f32


def plain_topk(s, k):
    """Indices of the k largest entries of each row, ties to the lower index."""
    s = np.asarray(s)
    order = np.lexsort((np.broadcast_to(np.arange(s.shape[1]), s.shape), -s.astype(np.float64)),
                       axis=1)
    return order[:, :k]


def seq_balance_stats(scores, k, seq_len, alpha=1e-4, scores_are_affinities=False):
    """Per-sequence f [S, E] (float32), P [S, E] (float64) and loss [S] (float64) for
    scores [T, E] (logits, or affinities if scores_are_affinities), T = S * seq_len."""
    scores = np.asarray(scores, dtype=np.float32)
    T, E = scores.shape
    if seq_len < 1 or T % seq_len:
        raise ValueError("T must be a multiple of seq_len")
    s = scores if scores_are_affinities else sigmoid_f32(scores)
    S = T // seq_len
    f = np.zeros((S, E), np.float32)
    P = np.zeros((S, E), np.float64)
    loss = np.zeros(S, np.float64)
    chosen = plain_topk(s, k)
    sd = s.astype(np.float64)
    for q in range(S):
        rows = slice(q * seq_len, (q + 1) * seq_len)
        count = np.bincount(chosen[rows].ravel(), minlength=E)
        f[q] = (count * E).astype(np.float32) / np.float32(k * seq_len)
        share = sd[rows] / sd[rows].sum(axis=1, keepdims=True)     # s' = s / sum_j s_j
        P[q] = share.mean(axis=0)
        loss[q] = alpha * float(np.dot(f[q].astype(np.float64), P[q]))
    return f, P, loss
