"""Pins of the oracle's E4M3 and BF16 rounding against the pages' constants, the bit
definition of the format, and library casts (torch.float8_e4m3fn, torch.bfloat16)."""

import json
import os

import numpy as np
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats_and_counts.json")))


def test_e4m3_constants_from_page():
    g = GOLD["e4m3"]
    t = oracle.e4m3_decode_table()
    finite = t[~np.isnan(t)]
    assert finite.max() == g["max_finite"] == oracle.E4M3_MAX
    normals = finite[finite >= oracle.E4M3_MIN_NORMAL]
    assert abs(normals.min() - g["min_normal"]) < 5e-6
    # 8 steps per octave: every full binade [2^e, 2^(e+1)) holds 2**man_bits codes
    for e in range(-6, 8):
        n = np.sum((finite >= 2.0 ** e) & (finite < 2.0 ** (e + 1)))
        assert n == g["steps_per_octave"] == 2 ** g["man_bits"]
    # fn convention: exactly two NaN codes and no infinity
    assert np.isnan(t).sum() == 2 and np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert not np.isinf(t).any()
    # subnormals: exponent field 0 with unit 2^-9
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9 and t[0x08] == 2.0 ** -6


def test_e4m3_roundtrip_all_codes():
    t = oracle.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    assert (oracle.e4m3_encode(t[codes].astype(np.float32)) == codes).all()


def test_e4m3_midpoints_round_to_even():
    t = oracle.e4m3_decode_table()
    pos = np.array(sorted(v for v in t[:0x7F] if not np.isnan(v)))      # 0 .. 448
    codes = oracle.e4m3_encode(pos.astype(np.float32))
    for i in range(len(pos) - 1):
        mid = (pos[i] + pos[i + 1]) / 2
        got = oracle.e4m3_encode(np.float32(mid))
        even = codes[i] if codes[i] % 2 == 0 else codes[i + 1]           # even mantissa
        assert got == even, (pos[i], pos[i + 1])
        above = np.nextafter(np.float32(mid), np.float32(np.inf))
        below = np.nextafter(np.float32(mid), np.float32(0))
        assert oracle.e4m3_encode(above) == codes[i + 1]
        assert oracle.e4m3_encode(below) == codes[i]


def test_e4m3_saturation_and_specials():
    v = np.array([448, 463.9, 464, 465, 1e6, np.inf, -449, -np.inf], dtype=np.float32)
    assert list(oracle.e4m3_encode(v)) == [0x7E] * 6 + [0xFE] * 2
    assert oracle.e4m3_encode(np.float32(np.nan)) == 0x7F
    assert oracle.e4m3_encode(np.float32(-0.0)) == 0x80
    assert oracle.e4m3_encode(np.float32(-2.0 ** -11)) == 0x80       # rounds to -0


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(200000) * s for s in (1e-3, 0.05, 1.0, 40.0)])
    v = np.clip(v, -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (oracle.e4m3_encode(v) == ref).all()
    codes = np.arange(256, dtype=np.uint8)
    ref_dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ours = oracle.e4m3_decode(codes)
    same = (ours == ref_dec) | (np.isnan(ours) & np.isnan(ref_dec))
    assert same.all()


def test_e4m3_direct_cast_statistics_from_page():
    g = GOLD["direct_cast_gradients"]
    x = np.random.default_rng(1).standard_normal(g["n"]) * g["std"]
    q = oracle.e4m3_round(x.astype(np.float32))
    assert (q == 0).sum() == g["zeros"]
    assert np.linalg.norm(q - x) / np.linalg.norm(x) == g["rel_l2"]
    a = GOLD["direct_cast_activation"]
    x = np.random.default_rng(2).standard_normal(1 << 16) * a["std"]
    err = np.linalg.norm(oracle.e4m3_round(x.astype(np.float32)) - x) / np.linalg.norm(x)
    assert abs(err - a["rel_l2"]) < 0.1 * a["rel_l2"]      # teaching-simulation number


def test_bf16_round_matches_torch_and_rounds_from_double():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert (oracle.bf16_round(v) == ref).all()
    # a float64 just above a BF16 midpoint must round up, although float32 would collapse
    # it onto the midpoint first (double rounding)
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_round(np.float64(v)) == np.float32(1.0 + 2.0 ** -7)
    assert oracle.bf16_round(np.float64(1.0 + 2.0 ** -8)) == np.float32(1.0)   # tie -> even
    assert np.isinf(oracle.bf16_round(np.float64(3.5e38)))
