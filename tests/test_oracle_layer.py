"""Pins of the oracle's whole-layer forward: the pages' FLOP and weight counts, an
unquantised float64 MoE written with torch ops (same routing) that the FP8 layer must
track within quantisation error, and agreement of the per-token variant with the whole
layer."""

import json
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "formats_and_counts.json")))


def test_flop_and_weight_counts_from_pages():
    g = GOLD["flops"]
    cfg = workloads.V3
    assert (cfg.d, cfg.f, cfg.K) == (g["d_model"], g["d_ffn"], g["k"])
    per_expert = 3 * 2 * cfg.d * cfg.f
    assert round(cfg.K * per_expert / 1e6, 1) == g["routed_mflop_per_token"]
    assert round(g["tokens"] * cfg.K * per_expert / 1e12, 2) == g["batch_tflop"]
    assert round(3 * cfg.d * cfg.f / 1e6, 2) == g["weights_per_expert_millions"]
    assert round(cfg.flops() / cfg.T / 1e6, 2) == g["nine_experts_mflop"]
    assert round(257 * per_expert / 1e9, 2) == g["all_257_gflop"]


def _tiny_inputs(pow2=False):
    cfg = workloads.TINY
    x = workloads.gen_x(cfg).float().numpy()
    cen = workloads.gen_centroids(cfg).numpy()
    bias = workloads.gen_bias(cfg).numpy()
    w32 = [tuple(w.numpy() for w in workloads.gen_expert_f32(cfg, e)) for e in range(cfg.E + 1)]
    qw = oracle.quant_128x128_pow2 if pow2 else oracle.quant_128x128
    experts = [tuple(a for w in ws for a in qw(w)) for ws in w32]
    return cfg, x, cen, bias, w32, experts


def _unquantised_error(out, cfg, x, w32):
    """MAE / RMS of the layer output against an unquantised float64 MoE (torch ops) that
    uses the oracle's routing decisions."""
    xt = torch.from_numpy(x).double()
    ref = torch.zeros_like(xt)
    for e in range(cfg.E + 1):
        w1, w3, w2 = (torch.from_numpy(w).double() for w in w32[e])
        yexp = (F.silu(xt @ w1.T) * (xt @ w3.T)) @ w2.T
        if e == cfg.E:
            ref += yexp
        else:
            wgt = torch.from_numpy(np.where(out["idx"] == e, out["gate"], 0).sum(1)).double()
            ref += wgt[:, None] * yexp
    ref = ref.numpy()
    return np.abs(out["y"] - ref).mean() / np.sqrt((ref ** 2).mean())


def test_power_of_two_variant_tracks_the_unquantised_moe_like_the_fp32_scales():
    """The MX-native variant (power-of-two scales for x, weights and h) is as close to the
    unquantised MoE as the FP32-scale recipe; its scales are powers of two."""
    errs = {}
    for pow2 in (False, True):
        cfg, x, cen, bias, w32, experts = _tiny_inputs(pow2)
        out = oracle.moe_layer(x, cen, bias, experts, cfg.n_groups, cfg.topk_groups, cfg.K,
                               pow2=pow2)
        errs[pow2] = _unquantised_error(out, cfg, x, w32)
        if pow2:
            for sc in (out["sx"], out["sh"]):
                assert (np.frexp(sc.astype(np.float64))[0] == 0.5).all()
            toks = [3, 200]
            part = oracle.moe_layer_tokens(toks, x[toks], cen, bias, lambda e: w32[e],
                                           cfg.n_groups, cfg.topk_groups, cfg.K, pow2=True)
            assert (part["y"] == out["y"][toks]).all()
    assert errs[True] < 0.05 and errs[True] <= 1.5 * errs[False], errs


def test_tiny_layer_tracks_unquantised_float64_moe():
    cfg, x, cen, bias, w32, experts = _tiny_inputs()
    out = oracle.moe_layer(x, cen, bias, experts, cfg.n_groups, cfg.topk_groups, cfg.K)
    # unquantised reference with the oracle's routing decisions
    xt = torch.from_numpy(x).double()
    ref = torch.zeros_like(xt)
    for e in range(cfg.E + 1):
        w1, w3, w2 = (torch.from_numpy(w).double() for w in w32[e])
        yexp = (F.silu(xt @ w1.T) * (xt @ w3.T)) @ w2.T
        if e == cfg.E:
            ref += yexp
        else:
            wgt = torch.from_numpy(np.where(out["idx"] == e, out["gate"], 0).sum(1)).double()
            ref += wgt[:, None] * yexp
    ref = ref.numpy()
    rms = np.sqrt((ref ** 2).mean())
    err = np.abs(out["y"] - ref)
    assert err.mean() / rms < 0.05, err.mean() / rms
    # structure checks: each token's routed experts are distinct and in <= M groups
    gs = cfg.E // cfg.n_groups
    assert all(len({e // gs for e in r}) <= cfg.topk_groups for r in out["idx"])
    assert out["Y"].shape == (cfg.rows, cfg.d)
    # dropping the shared expert is visible
    y_noshared = oracle.combine(out["Y"], out["row_of"], out["gate"], shared_row_base=-1)
    assert np.abs(y_noshared - ref).mean() / rms > 0.2


def test_per_token_variant_matches_whole_layer():
    cfg, x, cen, bias, w32, experts = _tiny_inputs()
    out = oracle.moe_layer(x, cen, bias, experts, cfg.n_groups, cfg.topk_groups, cfg.K)
    toks = [0, 17, 255]
    part = oracle.moe_layer_tokens(toks, x[toks], cen, bias, lambda e: w32[e],
                                   cfg.n_groups, cfg.topk_groups, cfg.K)
    assert (part["idx"] == out["idx"][toks]).all()
    assert (part["gate"] == out["gate"][toks]).all()
    assert (part["y"] == out["y"][toks]).all()
    # pre-quantised experts given by the caller take the same path
    part2 = oracle.moe_layer_tokens(toks, x[toks], cen, bias, None, cfg.n_groups,
                                    cfg.topk_groups, cfg.K, expert_quantised=experts.__getitem__)
    assert (part2["y"] == part["y"]).all() and (part2["idx"] == part["idx"]).all()
