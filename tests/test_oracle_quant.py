"""Pins of the oracle's 1x128 / 128x128 quantisation: scale layout, the max element
mapping to 448, the half-ulp error bound, the pages' byte counts and block-size trend,
and the codec step against torch's float8_e4m3fn cast."""

import json
import os

import numpy as np
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats_and_counts.json")))


def _x(rows, cols, seed=0):
    return np.random.default_rng(seed).standard_normal((rows, cols)).astype(np.float32)


def test_layout_each_scale_belongs_to_its_tile():
    rows, cols = 5, 384
    x = np.zeros((rows, cols), np.float32)
    for r in range(rows):
        for cb in range(cols // 128):
            x[r, cb * 128 + (r * 7 + cb) % 128] = 2.0 ** (r + 4 * cb)   # tile max, powers of 2
    q, s = oracle.quant_1x128(x)
    assert s.shape == (cols // 128, rows)
    for r in range(rows):
        for cb in range(cols // 128):
            assert s[cb, r] == np.float32(2.0 ** (r + 4 * cb)) / np.float32(448)
            assert q[r, cb * 128 + (r * 7 + cb) % 128] == 0x7E


def test_tiles_are_independent():
    x = _x(8, 512)
    q0, s0 = oracle.quant_1x128(x)
    x2 = x.copy()
    x2[3, 256:384] *= 1000.0
    q1, s1 = oracle.quant_1x128(x2)
    changed = np.zeros_like(s0, bool)
    changed[2, 3] = True
    assert (s1[changed] != s0[changed]).all() and (s1[~changed] == s0[~changed]).all()
    mask = np.zeros_like(q0, bool)
    mask[3, 256:384] = True
    assert (q1[~mask] == q0[~mask]).all()


def test_max_maps_to_448_and_error_within_half_ulp():
    x = _x(64, 1024, seed=1) * np.exp(np.random.default_rng(2).uniform(-8, 8, (64, 1))).astype(np.float32)
    q, s = oracle.quant_1x128(x)
    xt = x.reshape(64, 8, 128)
    dec = oracle.e4m3_decode(q).reshape(64, 8, 128)
    assert np.abs(dec).max() <= 448
    arg = np.abs(xt).argmax(axis=2)
    assert (np.abs(np.take_along_axis(dec, arg[..., None], 2)) == 448).all()
    st = s.T[:, :, None].astype(np.float64)
    err = np.abs(xt - st * dec)
    # half an E4M3 quantum at the value's binade (3 fraction bits), never below the
    # subnormal half-quantum 2^-10
    v = np.abs(xt / st)
    binade = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    bound = st * np.exp2(binade - 4) * (1 + 1e-6)
    assert (err <= bound).all()


def test_zero_tile_has_unit_scale():
    x = _x(2, 256)
    x[1, 128:] = 0
    q, s = oracle.quant_1x128(x)
    assert s[1, 1] == 1.0 and (q[1, 128:] == 0).all()


def test_codec_step_matches_torch_cast():
    x = _x(32, 768, seed=4) * 3
    q, s = oracle.quant_1x128(x)
    v = torch.from_numpy(x.reshape(32, 6, 128) / s.T[:, :, None])       # float32 division
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).reshape(32, 768).numpy()
    assert (q == ref).all()


def test_weight_blocks():
    w = _x(256, 384, seed=5) * 0.02
    w[128:, 256:] *= 50
    q, s = oracle.quant_128x128(w)
    assert s.shape == (2, 3)
    for rb in range(2):
        for cb in range(3):
            blk = w[rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
            assert s[rb, cb] == np.abs(blk).max() / np.float32(448)
    deq = oracle.dequant_128x128(q, s)
    assert np.abs(deq - w).max() <= s.max() * 16


def test_activation_tile_bytes_from_page():
    g = GOLD["activation_tile_bytes"]
    T, d = g["T"], g["d"]
    q, s = oracle.quant_1x128(np.ones((1, d), np.float32))   # one row: per-row byte cost
    per_row = q.nbytes + s.nbytes
    assert round(T * per_row / 1e6, 2) == g["fp8_with_scales_mb"]
    assert round(T * d * 2 / 1e6, 2) == g["bf16_mb"]
    m = GOLD["scale_metadata_overhead"]
    assert round(100 * s.nbytes / q.nbytes, 3) == m["activation_pct"]
    qw, sw = oracle.quant_128x128(np.ones((128, 128), np.float32))
    assert round(100 * sw.nbytes / qw.nbytes, 4) == m["weight_pct"]


def test_block_size_trend_from_page():
    """Smaller blocks isolate outliers: fewer quiet values die and the quiet-value error
    drops from the per-4096 block to the per-32 block (qualitative; the page's NumPy
    simulation has no subnormals, so its absolute numbers are larger than ours)."""
    g = GOLD["block_size_trend"]
    errs, dead = [], []
    for seed in range(4):
        rng = np.random.default_rng(seed)
        x = rng.standard_normal(4096).astype(np.float32)
        pos = rng.choice(4096, 4, replace=False)
        x[pos] = 3000
        quiet = np.ones(4096, bool)
        quiet[pos] = False
        e_row, d_row = [], []
        for b in g["blocks"]:
            xb = x.reshape(-1, b)
            amax = np.abs(xb).max(axis=1)
            s = (amax / np.float32(448)).astype(np.float32)
            xh = (oracle.e4m3_round((xb / s[:, None]).astype(np.float32)) * s[:, None]).reshape(-1)
            e_row.append(np.linalg.norm(xh[quiet] - x[quiet]) / np.linalg.norm(x[quiet]))
            d_row.append(int(((xh == 0) & quiet).sum()))
        errs.append(e_row)
        dead.append(d_row)
    errs, dead = np.mean(errs, 0), np.mean(dead, 0)
    assert errs[-1] < errs[0] and errs[2] < errs[0]
    assert dead[0] > dead[2] >= dead[3]
    assert g["dead"][0] > g["dead"][2] > g["dead"][3]


# ---- power-of-two scales (the MX-native variant) ---------------------------------------

def _blocks_with_amax(amaxes, seed=0):
    """One 1x128 tile per amax value, random contents scaled so the tile's max-abs is it."""
    rng = np.random.default_rng(seed)
    x = rng.uniform(-1, 1, (len(amaxes), 128)).astype(np.float64)
    x[:, 0] = 1.0
    return (x * np.asarray(amaxes, np.float64)[:, None]).astype(np.float32)


def test_pow2_scale_is_the_smallest_power_of_two_that_fits():
    amaxes = [3.0, 448.0, 448.0 * 2 ** -20, 1e-30, 12345.0, 0.5, 224.0, 224.0001, 1.0]
    x = _blocks_with_amax(amaxes)
    q, s = oracle.quant_1x128_pow2(x)
    s = s[0].astype(np.float64)
    amax = np.abs(x.astype(np.float64)).max(axis=1)
    mant, _ = np.frexp(s)
    assert (mant == 0.5).all()                                # powers of two
    assert (amax / s <= 448).all() and (amax / s > 224).all()  # the smallest that fits
    dec = oracle.e4m3_decode(q)
    assert np.abs(dec).max() <= 448                           # never saturates


def test_pow2_closed_form_and_zero_tile():
    # amax 3 -> 448 * 2^-8 = 1.75 < 3 <= 448 * 2^-7 = 3.5, so s = 2^-7 and 3 / s = 384,
    # which E4M3 holds exactly (1.5 * 2^8)
    x = np.zeros((2, 128), np.float32)
    x[0, 5] = 3.0
    x[0, 6] = -1.5
    q, s = oracle.quant_1x128_pow2(x)
    assert s[0, 0] == 2.0 ** -7 and s[0, 1] == 1.0
    dec = oracle.e4m3_decode(q)
    assert dec[0, 5] == 384.0 and dec[0, 6] == -192.0
    assert (q[1] == 0).all()


def test_pow2_equals_fp32_scales_when_amax_over_448_is_a_power_of_two():
    amaxes = [448.0 * 2.0 ** k for k in range(-12, 6)]
    x = _blocks_with_amax(amaxes, seed=3)
    q2, s2 = oracle.quant_1x128_pow2(x)
    q1, s1 = oracle.quant_1x128(x)
    assert np.array_equal(s1, s2) and np.array_equal(q1, q2)


def test_pow2_reconstruction_error_bound_and_weight_blocks():
    rng = np.random.default_rng(8)
    w = (rng.standard_normal((256, 384)) * np.exp(rng.uniform(-6, 6, (256, 1)))).astype(np.float32)
    q, s = oracle.quant_128x128_pow2(w)
    assert s.shape == (2, 3)
    assert (np.frexp(s.astype(np.float64))[0] == 0.5).all()
    w_hat = oracle.dequant_128x128(q, s)
    full = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    # half an E4M3 ulp (3 fraction bits) relative, or half the subnormal unit 2^-9
    assert (np.abs(w_hat - w) <= 2.0 ** -4 * np.abs(w) + full * 2.0 ** -10).all()


def test_dequant_1x128_layout_distinct_scales():
    """Each element is its code's E4M3 value (decoded by torch's float8_e4m3fn cast, a
    library routine) times the scale of its own (K block, row): s[c // 128][r], the
    K-block-major activation-scale layout.  Checked element by element in plain Python,
    with a different power-of-two-free scale for every (row, K block) so a transposed or
    shifted scale index cannot pass."""
    import torch
    rows, cols = 3, 384
    rng = np.random.default_rng(11)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    q = finite[rng.integers(0, finite.size, (rows, cols))]
    s = np.array([[1.0 + r + 10.0 * kb + 0.125 for r in range(rows)] for kb in range(cols // 128)],
                 np.float32)                                     # [cols/128][rows]
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.dequant_1x128(q, s)
    assert got.shape == (rows, cols)
    for r in range(rows):
        for c in range(cols):
            assert got[r, c] == dec[r, c] * float(s[c // 128, r]), (r, c)
