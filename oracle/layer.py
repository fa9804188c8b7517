"""The whole MoE FFN layer forward, and a per-token variant for large shapes.

Oracle module (test infrastructure only).

The layer follows the order the pages give for one MoE layer (DeepSeek-V3 book, ch. 7
and ch. 15; "DeepSeek-V3", core ideas 1 and 6): router logits in high precision,
sigmoid affinities, biased group-limited top-k selection, normalised gates, FP8
quantisation of the activations before dispatch, grouping of rows by expert, SwiGLU
experts as block-scaled FP8 GEMMs, and a BF16 gate-weighted combine plus the shared
expert.  Each step is the oracle function of the same name; nothing is fused.
"""

import numpy as np

from .quant import quant_1x128, quant_128x128, quant_1x128_pow2, quant_128x128_pow2
from .router import router_logits, route, route_token, sigmoid_f32
from .permute import permute
from .gemm import swiglu_expert, combine


def moe_layer(x, centroids, bias, experts, n_groups, topk_groups, k, route_scale=1.0,
              logits=None, pow2=False):
    """Forward of one layer on every token.

    x: float32 [T, d] (BF16 values); centroids float32 [E, d]; bias float32 [E];
    experts: sequence of E + 1 tuples (w1q, s1, w3q, s3, w2q, s2), the last one the
    shared expert (already block-quantised with ``quant_128x128``).
    ``logits``: optional float32 [T, E] to route from instead of computing them.
    ``pow2``: the MX-native variant -- activations and h quantised with power-of-two
    scales (the experts must then come from ``quant_128x128_pow2``).
    Returns a dict with every intermediate the CUDA path also produces.
    """
    x = np.asarray(x, dtype=np.float32)
    T, d = x.shape
    E = centroids.shape[0]
    z = router_logits(x, centroids) if logits is None else np.asarray(logits, np.float32)
    idx, gate = route(z, bias, n_groups, topk_groups, k // topk_groups, k, route_scale)
    counts, offsets, row_token, row_of = permute(idx, E, include_shared=True)
    xq, sx = quant_1x128_pow2(x) if pow2 else quant_1x128(x)
    rows = int(offsets[E + 1])
    f = experts[0][0].shape[0]
    hq = np.zeros((rows, f), dtype=np.uint8)
    sh = np.zeros((f // 128, rows), dtype=np.float32)
    Y = np.zeros((rows, d), dtype=np.float32)
    for e in range(E + 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        toks = row_token[r0:r1]
        hq_e, sh_e, y_e = swiglu_expert(xq[toks], sx[:, toks], *experts[e], pow2=pow2)
        hq[r0:r1], sh[:, r0:r1], Y[r0:r1] = hq_e, sh_e, y_e
    y = combine(Y, row_of, gate, shared_row_base=T * k)
    return dict(z=z, idx=idx, gate=gate, counts=counts, offsets=offsets,
                row_token=row_token, row_of=row_of, xq=xq, sx=sx, hq=hq, sh=sh, Y=Y, y=y)


def moe_layer_tokens(tokens, x_rows, centroids, bias, expert_weights_f32, n_groups,
                     topk_groups, k, route_scale=1.0, expert_quantised=None, pow2=False):
    """Layer output for a few tokens only (for shapes too large to run whole).

    Rows of a segment never interact, so a token's output depends only on its own row,
    its chosen experts and the shared expert.  ``x_rows`` float32 [n, d] holds the
    tokens' inputs; ``expert_weights_f32(e)`` returns float32 (w1 [f,d], w3 [f,d],
    w2 [d,f]) for expert e (e = E is the shared expert); the oracle quantises them
    itself.  ``expert_quantised(e)``, when given, returns expert e already quantised
    with ``quant_128x128`` as (w1q, s1, w3q, s3, w2q, s2) and replaces that step (it lets a
    caller run the quantisation of many experts in parallel).
    ``pow2``: the MX-native variant (power-of-two scales everywhere).
    Returns dict(idx [n,k], gate [n,k], y [n,d], s [n,E]).
    """
    x_rows = np.asarray(x_rows, dtype=np.float32)
    E = centroids.shape[0]
    z = router_logits(x_rows, centroids)
    s = sigmoid_f32(z)
    c = (s + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
    cache = {}

    def quantised(e):
        if expert_quantised is not None:
            return expert_quantised(e)
        if e not in cache:
            w1, w3, w2 = expert_weights_f32(e)
            qw = quant_128x128_pow2 if pow2 else quant_128x128
            cache[e] = (*qw(w1), *qw(w3), *qw(w2))
        return cache[e]

    xq, sx = quant_1x128_pow2(x_rows) if pow2 else quant_1x128(x_rows)
    n = len(tokens)
    idx = np.empty((n, k), np.int32)
    gate = np.empty((n, k), np.float32)
    ys = []
    for i in range(n):
        idx[i], gate[i], _ = route_token(s[i], c[i], n_groups, topk_groups,
                                         k // topk_groups, k, route_scale)
        rows = [swiglu_expert(xq[i:i + 1], sx[:, i:i + 1], *quantised(int(e)), pow2=pow2)[2]
                for e in list(idx[i]) + [E]]
        Y = np.concatenate(rows, axis=0)                 # k routed rows, then shared
        row_of = np.arange(k, dtype=np.int32)[None, :]
        ys.append(combine(Y, row_of, gate[i:i + 1], shared_row_base=k)[0])
    return dict(idx=idx, gate=gate, y=np.stack(ys), s=s, z=z)
