"""Block-scaled FP8 GEMM with per-128-K promotion, the SwiGLU expert, and combine.

Oracle module (test infrastructure only).

What the pages fix:
* with scales that vary along K, each K-block partial sum needs its own product of
  group scales before it joins the result (DeepSeek-V3 book, ch. 16 "Scales along the
  GEMM inner dimension");
* partial sums are promoted to FP32 every N_C = 128 elements of K, and the group scales
  are applied during that promotion ("DeepSeek-V3", core idea 6(b); book ch. 16
  "Periodic high-precision promotion");
* a SwiGLU expert is W_down(SiLU(W_gate x) * W_up x) with d = 7168, f = 2048 (book ch. 2
  "RMSNorm and SwiGLU", ch. 7 "What one expert computes");
* the input of the down projection is FP8 with 1x128 tiles like any activation
  ("DeepSeek-V3", core idea 6(a));
* combine adds each expert's output weighted by the token's gate, plus the shared
  expert, and stays BF16 (book ch. 7 "Selecting and combining experts", ch. 15 "What
  combine must do", ch. 17 "FP8 dispatch, BF16 combine").

The definition computed here, for C = A . B^T with A [M, K] (scales sa[K/128][M]) and
B [N, K] (scales sb[N/128][K/128]):

    C[m, n] = sum_kb  (sa[kb, m] * sb[n // 128, kb]) * P_kb[m, n]
    P_kb    = sum_{k in block kb} dec(qa[m, k]) * dec(qb[n, k])

P_kb is exact in float64: every E4M3 value is a multiple of 2**-9, so each product is a
multiple of 2**-18 below 2**18 in magnitude, and a 128-term sum needs fewer than 44 bits.
The scale products and the sum over blocks are carried in float64.

Readings taken: expert outputs Y are rounded to BF16 (RNE); gate and up outputs are
rounded to float32 before h = fl32(silu(g) * u) with silu in float64; h is requantised
1x128 along f from float32; the layer output excludes the residual u (the caller adds
it) and is rounded to BF16 once, after the float64 sum shared + sum_k g_k * Y_k.
"""

import numpy as np

from .formats import e4m3_decode, bf16_round
from .quant import quant_1x128, quant_1x128_pow2


def blockscaled_gemm(qa, sa, qb, sb):
    """float64 C[M, N] per the definition in the module docstring.

    qa uint8 [M, K], sa float32 [K/128, M]; qb uint8 [N, K], sb float32 [N/128, K/128].
    """
    M, K = qa.shape
    N = qb.shape[0]
    assert K % 128 == 0 and N % 128 == 0 and qb.shape[1] == K
    A = e4m3_decode(qa)
    B = e4m3_decode(qb)
    C = np.zeros((M, N), dtype=np.float64)
    for kb in range(K // 128):
        ks = slice(kb * 128, (kb + 1) * 128)
        P = A[:, ks] @ B[:, ks].T                                      # exact
        scale = (np.asarray(sa[kb], np.float64)[:, None]
                 * np.repeat(np.asarray(sb[:, kb], np.float64), 128)[None, :N])
        C += scale * P
    return C


def swiglu_expert(xq, sx, w1q, s1, w3q, s3, w2q, s2, pow2=False):
    """One SwiGLU expert on FP8 rows.

    xq uint8 [m, d] with sx float32 [d/128, m]; w1q/w3q uint8 [f, d] (gate / up) with
    s1/s3 float32 [f/128, d/128]; w2q uint8 [d, f] with s2 float32 [d/128, f/128].
    Returns (hq uint8 [m, f], sh float32 [f/128, m], Y float32 [m, d] of BF16 values).
    pow2: h is requantised with power-of-two scales (the MX-native variant).
    """
    g = blockscaled_gemm(xq, sx, w1q, s1).astype(np.float32)
    u = blockscaled_gemm(xq, sx, w3q, s3).astype(np.float32)
    gd = g.astype(np.float64)
    with np.errstate(over="ignore"):
        silu = gd / (1.0 + np.exp(-gd))
    h = (silu * u.astype(np.float64)).astype(np.float32)
    hq, sh = quant_1x128_pow2(h) if pow2 else quant_1x128(h)
    y = bf16_round(blockscaled_gemm(hq, sh, w2q, s2))
    return hq, sh, y


def combine(y_rows, row_of, gate, shared_row_base):
    """y[t] = bf16( Y[shared_row_base + t] + sum_k gate[t, k] * Y[row_of[t, k]] ).

    The sum is carried in float64; ``shared_row_base < 0`` means no shared expert.
    """
    T, K = row_of.shape
    Y = np.asarray(y_rows, dtype=np.float64)
    acc = np.zeros((T, Y.shape[1]), dtype=np.float64)
    if shared_row_base >= 0:
        acc += Y[shared_row_base:shared_row_base + T]
    for k in range(K):
        acc += np.asarray(gate[:, k], np.float64)[:, None] * Y[row_of[:, k]]
    return bf16_round(acc)
