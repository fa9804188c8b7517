"""Backward pass of the SwiGLU experts in FP8: Dgrad and Wgrad GEMMs, the 1x128 -> 128x1
regrouping of activations, and SwiGLU recomputation from its cached FP8 inputs.

Oracle module (test infrastructure only).

What the pages fix (DeepSeek-V3 book, ch. 17 "One linear layer creates three GEMMs",
"SwiGLU recomputation", "Attention-related saved activations", "Backward grouping and
gradient sensitivity"; ch. 16 "Why transposition is not trivial"; "DeepSeek-V3" summary,
core idea 6):
* a linear layer Y = X W needs, given dY, the input gradient dX = dY W^T (Dgrad) and the
  weight gradient dW = X^T dY (Wgrad); all three GEMMs take FP8 inputs, with outputs in
  BF16 or FP32 and the same promotion of partial sums as the forward;
* activation gradients keep 1x128 tiles (128x128 blocks for them diverged);
* backward GEMMs may need the transposed orientation of an activation, which changes
  which elements share a scale: V3 regroups 1x128 tiles into 128x1 tiles there, with
  power-of-two scales to avoid extra quantisation error;
* the MoE caches the SwiGLU inputs in FP8 and recomputes the SwiGLU output in backward.

Definitions used here, for one expert e whose rows are r in [seg[e], seg[e+1]) (rows in
segment order, as in the forward), with the forward's quantised weights w1q/w3q [f, d]
(gate/up), w2q [d, f] and their 128x128 block scales:

  forward cache  g = fl32(G), u = fl32(U) from the gate/up GEMM, each quantised 1x128
                 along f (the FP32-scale rule) -> guq [R, 2f] = [gq | uq], sgu [2f/128, R]
  1  dYq, sdY   = quant_1x128(dY)                                  (dY BF16 [R, d])
  2  dh         = bf16( GEMM(dYq, W2^T) )     Dgrad of the down projection, contraction
                  over d; W2^T [f, d] keeps W2's 128x128 blocks (scales transposed)
  3  g, u       = fl32(dec(guq) * sgu)        the cached SwiGLU inputs, dequantised
  4  recompute  sig = 1/(1+exp(-g)),  h = g*sig*u;
     backward   dU = dh * g * sig,    dG = dh * u * sig * (1 + g*(1 - sig))   (float64,
                  then fl32)
  5  dGUq, sdGU = quant_1x128([dG | dU])      [R, 2f]
  6  dX         = bf16( GEMM(dGUq, [W1; W3]^T) )   Dgrad of gate/up, contraction over 2f
  7  regroup    dY, h, dG, dU and the input rows X into 128x1 tiles with power-of-two
                scales: per expert, its rows are cut into 128-row blocks starting at the
                segment's first row (a block never holds two experts' rows; the last one
                is zero-padded), one scale per (block, column); stored transposed
                [C][R_pad], R_pad = sum_e ceil(count_e / 128) * 128
  8  dW2 = fl32( WGRAD(dY^T, h^T) ) [d, f];  dW1 = fl32( WGRAD(dG^T, X^T) ) [f, d];
     dW3 = fl32( WGRAD(dU^T, X^T) ) [f, d]
     WGRAD(A^T, B^T)[i, j] = sum_rb sA[rb, i] * sB[rb, j] * sum_{p in rb} dec(A^T[i, p]) *
                             dec(B^T[j, p])   over the expert's row blocks rb (exact
                             per-block products, float64 sum)

Readings taken where the pages are silent: dh and dX are BF16 GEMM outputs and the
weight gradients FP32; the 128x1 tiles are quantised from the higher-precision tensor
(BF16 dY and X, FP32 h, dG and dU) rather than requantised from the 1x128 codes; the
power-of-two rule is the forward variant's (smallest 2^k >= 2^-126 with 448 * 2^k >=
amax); the routing gates are applied before dY reaches the experts (dY is the gradient
of the expert output rows), and the gating and router backward are not part of this
module.
"""

import numpy as np

from .formats import e4m3_decode, e4m3_encode, bf16_round
from .quant import quant_1x128, _pow2_scale_from_amax
from .gemm import blockscaled_gemm


def combine_backward_rows(dy, gate, row_of, shared_row_base, n_rows):
    """Gradient of the combine y_t = Y[shared_row_base + t] + sum_k g_tk * Y[row_of[t, k]]
    with respect to the expert output rows, as the expert backward's BF16 input:
    dY[row_of[t, k]] = bf16(fl32(g_tk * dy_t)), dY[shared_row_base + t] = dy_t (float32
    array of BF16 values; rows nobody uses stay 0)."""
    dy = np.asarray(dy, np.float32)
    T, d = dy.shape
    out = np.zeros((n_rows, d), np.float32)
    for t in range(T):
        if shared_row_base >= 0:
            out[shared_row_base + t] = dy[t]
        for k in range(row_of.shape[1]):
            out[row_of[t, k]] = bf16_round((np.float32(gate[t, k]) * dy[t]).astype(np.float32))
    return out


def padded_offsets(seg):
    """Start of every expert's 128-row-aligned block range: pad[e] = sum over e' < e of
    ceil(count_e' / 128) * 128; pad[G] = R_pad."""
    seg = np.asarray(seg, dtype=np.int64)
    cnt = np.diff(seg)
    return np.concatenate([[0], np.cumsum((cnt + 127) // 128 * 128)]).astype(np.int64)


def quant_128x1_pow2_segments(x, seg):
    """Regroup rows of x (float32 [R, C], rows in segment order) into 128x1 tiles with
    power-of-two scales, per segment, stored transposed.

    Returns (qT uint8 [C, R_pad], sT float32 [R_pad/128, C], pad [G+1]).  Padded rows
    hold code 0.  A block's scale is the power-of-two rule applied to the max |x| over
    its (real) rows in that column; an all-zero column of a block gets scale 1.
    """
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    pad = padded_offsets(seg)
    R_pad = int(pad[-1])
    qT = np.zeros((C, R_pad), dtype=np.uint8)
    sT = np.ones((R_pad // 128, C), dtype=np.float32)
    for e in range(len(seg) - 1):
        r0, r1 = int(seg[e]), int(seg[e + 1])
        for b0 in range(r0, r1, 128):
            b1 = min(b0 + 128, r1)
            blk = x[b0:b1]                                         # [<=128, C]
            s = _pow2_scale_from_amax(np.abs(blk).max(axis=0))     # [C]
            q = e4m3_encode((blk / s[None, :]).astype(np.float32))  # exact division
            p0 = int(pad[e]) + (b0 - r0)
            qT[:, p0:p0 + (b1 - b0)] = q.T
            sT[p0 // 128] = s
    return qT, sT, pad


def wgrad(aT, saT, bT, sbT, pad):
    """Per expert e: C_e[i, j] = sum_rb saT[rb, i] * sbT[rb, j] * sum_{p in rb}
    dec(aT[i, p]) * dec(bT[j, p]) over the row blocks rb of e, in float64.

    aT uint8 [I, R_pad], saT float32 [R_pad/128, I]; bT uint8 [J, R_pad], sbT float32
    [R_pad/128, J]; pad [G+1].  Returns float64 [G, I, J] (zero for an empty expert)."""
    A = e4m3_decode(aT)
    B = e4m3_decode(bT)
    G = len(pad) - 1
    out = np.zeros((G, A.shape[0], B.shape[0]), dtype=np.float64)
    for e in range(G):
        for p0 in range(int(pad[e]), int(pad[e + 1]), 128):
            rb = p0 // 128
            P = A[:, p0:p0 + 128] @ B[:, p0:p0 + 128].T               # exact
            out[e] += (np.asarray(saT[rb], np.float64)[:, None] *
                       np.asarray(sbT[rb], np.float64)[None, :]) * P
    return out


def swiglu_backward(g, u, dh):
    """SwiGLU recomputed from its inputs and differentiated (float64, rounded to float32):
    h = silu(g) * u,  dU = dh * silu(g),  dG = dh * u * sig(g) * (1 + g * (1 - sig(g)))."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    dh = np.asarray(dh, np.float64)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    h = silu * u
    du = dh * silu
    dg = dh * u * sig * (1.0 + g * (1.0 - sig))
    return h.astype(np.float32), dg.astype(np.float32), du.astype(np.float32)


def dequant_rows_1x128_f32(q, s):
    """fl32(dec(q) * s) for 1x128 tiles: q uint8 [R, C], s float32 [C/128, R]."""
    R, C = q.shape
    sc = np.repeat(np.asarray(s, np.float32).T, 128, axis=1)[:, :C]
    return (e4m3_decode(q).astype(np.float32) * sc).astype(np.float32)


def swiglu_cache(xq, sx, w1q, s1, w3q, s3):
    """The forward's FP8 cache of the SwiGLU inputs for a training step: g, u from the
    gate/up GEMMs (float32) quantised 1x128 along f.  Returns (guq [R, 2f], sgu [2f/128, R])
    with the gate columns first."""
    g = blockscaled_gemm(xq, sx, w1q, s1).astype(np.float32)
    u = blockscaled_gemm(xq, sx, w3q, s3).astype(np.float32)
    gq, sg = quant_1x128(g)
    uq, su = quant_1x128(u)
    return np.concatenate([gq, uq], axis=1), np.concatenate([sg, su], axis=0)


def expert_backward(seg, x_rows, dy_rows, guq, sgu, experts):
    """Backward of the SwiGLU experts over expert segments, step by step as in the module
    docstring.

    seg [G+1] row offsets; x_rows float32 [R, d] (BF16 values: the experts' input rows);
    dy_rows float32 [R, d] (BF16 values: gradient of the expert output rows); guq uint8
    [R, 2f], sgu float32 [2f/128, R] (the forward cache); experts[e] = (w1q, s1, w3q, s3,
    w2q, s2), the forward's quantised weights.

    Returns a dict: dh (float32 of BF16 values [R, f]), h, dg, du (float32 [R, f]),
    dx (float32 of BF16 values [R, d]), dw1, dw3 (float32 [G, f, d]), dw2 (float32
    [G, d, f]) and the intermediate quantised tensors.
    """
    seg = np.asarray(seg, dtype=np.int64)
    G = len(seg) - 1
    R, d = dy_rows.shape
    f = guq.shape[1] // 2
    dyq, sdy = quant_1x128(dy_rows)                                          # step 1
    dh = np.zeros((R, f), np.float32)
    for e in range(G):                                                       # step 2
        r0, r1 = int(seg[e]), int(seg[e + 1])
        if r1 > r0:
            w2q, s2 = experts[e][4], experts[e][5]
            dh[r0:r1] = bf16_round(blockscaled_gemm(dyq[r0:r1], sdy[:, r0:r1],
                                                    np.ascontiguousarray(w2q.T),
                                                    np.ascontiguousarray(s2.T)))
    gu = dequant_rows_1x128_f32(guq, sgu)                                    # step 3
    h, dg, du = swiglu_backward(gu[:, :f], gu[:, f:], dh)                     # step 4
    dguq, sdgu = quant_1x128(np.concatenate([dg, du], axis=1))                # step 5
    dx = np.zeros((R, d), np.float32)
    for e in range(G):                                                       # step 6
        r0, r1 = int(seg[e]), int(seg[e + 1])
        if r1 > r0:
            w1q, s1, w3q, s3 = experts[e][:4]
            wcat_t = np.ascontiguousarray(np.concatenate([w1q, w3q], axis=0).T)   # [d, 2f]
            scat_t = np.ascontiguousarray(np.concatenate([s1, s3], axis=0).T)     # [d/128, 2f/128]
            dx[r0:r1] = bf16_round(blockscaled_gemm(dguq[r0:r1], sdgu[:, r0:r1], wcat_t,
                                                    scat_t))
    dyT, sdyT, pad = quant_128x1_pow2_segments(dy_rows, seg)                 # step 7
    hT, shT, _ = quant_128x1_pow2_segments(h, seg)
    dgT, sdgT, _ = quant_128x1_pow2_segments(dg, seg)
    duT, sduT, _ = quant_128x1_pow2_segments(du, seg)
    xT, sxT, _ = quant_128x1_pow2_segments(x_rows, seg)
    dw2 = wgrad(dyT, sdyT, hT, shT, pad).astype(np.float32)                  # step 8
    dw1 = wgrad(dgT, sdgT, xT, sxT, pad).astype(np.float32)
    dw3 = wgrad(duT, sduT, xT, sxT, pad).astype(np.float32)
    return dict(dh=dh, h=h, dg=dg, du=du, dx=dx, dw1=dw1, dw3=dw3, dw2=dw2,
                dyq=dyq, sdy=sdy, dguq=dguq, sdgu=sdgu, pad=pad,
                dyT=dyT, sdyT=sdyT, hT=hT, shT=shT, dgT=dgT, sdgT=sdgT, duT=duT, sduT=sduT,
                xT=xT, sxT=sxT)
