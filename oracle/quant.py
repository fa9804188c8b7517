"""Fine-grained FP8 quantisation with online max-abs scales.

Oracle module (test infrastructure only).

What the pages fix:
* one FP32 scale per 1x128 activation tile (per token, per 128 channels) and per
  128x128 weight block ("DeepSeek-V3", core idea 6(a); DeepSeek-V3 book, ch. 16
  "V3's grouping");
* the scale comes from the max-abs of the current tile, not from history
  ("DeepSeek-V3", core idea 6(d); book ch. 16 "Online scales");
* choose s so that x/s fits the E4M3 range, and reconstruct x_hat = s * q (book
  ch. 16 "Scaling a group"; the stored scale is the dequantisation multiplier,
  like the release checkpoint's weight_scale_inv).

Reading taken (the formula itself is lost in the page text):
  amax = max |x| over the group (exact in float32)
  s    = fl32(amax / 448)           correctly rounded float32 division
  q    = E4M3_rne_satfinite(fl32(x / s))
  amax == 0  ->  s = 1, q = 0
Saturation is required: x/s for the max element can round to just above 448.

Layouts: activation scales are stored K-block-major, ``s[col_block][row]``; weight
scales ``s[row_block][col_block]``.

Power-of-two variant (the MX-native path).  The pages note that the 1x128 / 128x128
groups match the microscaling formats Blackwell tensor cores take natively ("DeepSeek-V3"
summary, core idea 6(a)), list native group-scaled MMA on the hardware wishlist (core
idea 8), and mention power-of-two scales as a way to avoid extra quantisation error
(DeepSeek-V3 book, ch. 17 "Attention-related saved activations").  Reading taken:
  s = the smallest power of two with 448 * s >= amax, at least 2^-126 (the smallest
      normal float32; s = 1 when amax == 0)
  q = E4M3_rne(x / s)        (the division is exact; |x / s| <= 448, so no saturation)
with the same group shapes and layouts; the tensor core reads the scale's exponent byte.
"""

import numpy as np

from .formats import E4M3_MAX, e4m3_encode, e4m3_decode


def _scale_from_amax(amax):
    amax = np.asarray(amax, dtype=np.float32)
    s = amax / np.float32(E4M3_MAX)                 # float32 / float32 -> float32, RNE
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def _pow2_scale_from_amax(amax):
    """Smallest power of two s >= 2^-126 with 448 * s >= amax (exact comparisons); 1 for
    amax == 0."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.ones(amax.shape, dtype=np.float64)
    for i, a in np.ndenumerate(amax):
        if a == 0:
            continue
        e = int(np.ceil(np.log2(a / E4M3_MAX)))
        while E4M3_MAX * 2.0 ** (e - 1) >= a:         # step down while still large enough
            e -= 1
        while E4M3_MAX * 2.0 ** e < a:                # step up until large enough
            e += 1
        out[i] = 2.0 ** max(e, -126)                  # kept a normal float32
    return out.astype(np.float32)


def _quant_groups(x, group_shape, scale_fn):
    """Shared shape handling: x [rows, cols] in (gr, gc) groups -> (q, s[rows/gr, cols/gc])."""
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    gr, gc = group_shape
    xb = x.reshape(rows // gr, gr, cols // gc, gc)
    amax = np.abs(xb).max(axis=(1, 3))
    s = scale_fn(amax)
    v = (xb / s[:, None, :, None]).astype(np.float32)
    return e4m3_encode(v).reshape(rows, cols), s


def quant_1x128_pow2(x):
    """Power-of-two-scale variant of quant_1x128: (q uint8[rows, cols], s[cols/128, rows])."""
    q, s = _quant_groups(x, (1, 128), _pow2_scale_from_amax)
    return q, np.ascontiguousarray(s.T)


def quant_128x128_pow2(w):
    """Power-of-two-scale variant of quant_128x128: (q, s[rows/128, cols/128])."""
    return _quant_groups(w, (128, 128), _pow2_scale_from_amax)


def quant_1x128(x):
    """Quantise float32 ``x[rows, cols]`` (cols % 128 == 0) in 1x128 tiles.

    Returns (q uint8[rows, cols], s float32[cols // 128, rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, cols = x.shape
    assert cols % 128 == 0
    xt = x.reshape(rows, cols // 128, 128)
    amax = np.abs(xt).max(axis=2)                              # [rows, cols/128]
    s = _scale_from_amax(amax)
    v = (xt / s[:, :, None]).astype(np.float32)                # float32 division
    q = e4m3_encode(v).reshape(rows, cols)
    return q, np.ascontiguousarray(s.T)


def dequant_1x128(q, s):
    """x_hat[r, c] = s[c // 128, r] * decode(q[r, c]) in float64."""
    rows, cols = q.shape
    return e4m3_decode(q) * np.repeat(s.T.astype(np.float64), 128, axis=1)[:, :cols]


def quant_128x128(w):
    """Quantise float32 ``w[rows, cols]`` (both % 128 == 0) in 128x128 blocks.

    Returns (q uint8[rows, cols], s float32[rows // 128, cols // 128]).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    wb = w.reshape(rows // 128, 128, cols // 128, 128)
    amax = np.abs(wb).max(axis=(1, 3))                         # [rb, cb]
    s = _scale_from_amax(amax)
    v = (wb / s[:, None, :, None]).astype(np.float32)
    q = e4m3_encode(v).reshape(rows, cols)
    return q, s


def dequant_128x128(q, s):
    """w_hat[r, c] = s[r // 128, c // 128] * decode(q[r, c]) in float64."""
    full = np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)
    return e4m3_decode(q) * full
