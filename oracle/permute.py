"""Grouping of token rows by expert (dispatch metadata).

Oracle module (test infrastructure only).

What the pages fix: the receiver groups rows by expert so each expert's weights see a
contiguous batch, and keeps metadata naming the original token and its mixture weight
so outputs can be restored and combined (DeepSeek-V3 book, ch. 15 "What dispatch must
do", "What combine must do"; ch. 7 "Batches change what is active"); no token is
dropped ("DeepSeek-V3", core idea 1 "No token dropping").

Reading taken: a stable counting sort of the flattened (t, k) pairs keyed by expert.
Rows of segment e are ordered by token; within one token the experts are distinct, so
no two of its pairs share a segment.  When the shared expert is included it forms
segment E after the routed rows, with row T*K + t holding token t.

Outputs:
  counts    int32[E]       pairs per routed expert
  offsets   int32[E + 2]   offsets[e] = first row of segment e (e = E is the shared
                           segment), offsets[E + 1] = total rows
  row_token int32[rows]    token of each row
  row_of    int32[T, K]    row holding pair (t, k)
"""

import numpy as np


def permute(idx, n_experts, include_shared=True):
    idx = np.asarray(idx, dtype=np.int64)
    T, K = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=n_experts).astype(np.int32)
    offsets = np.zeros(n_experts + 2, dtype=np.int64)
    offsets[1:n_experts + 1] = np.cumsum(counts)
    offsets[n_experts + 1] = offsets[n_experts] + (T if include_shared else 0)
    rows = int(offsets[n_experts + 1])
    row_token = np.empty(rows, dtype=np.int32)
    row_of = np.empty((T, K), dtype=np.int32)
    cursor = offsets[:n_experts].copy()
    for p in range(T * K):
        t, k = divmod(p, K)
        e = flat[p]
        r = cursor[e]
        cursor[e] += 1
        row_token[r] = t
        row_of[t, k] = r
    if include_shared:
        base = T * K
        row_token[base:base + T] = np.arange(T, dtype=np.int32)
    return counts, offsets.astype(np.int32), row_token, row_of
