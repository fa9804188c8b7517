"""Floating-point comparison used by the parity tests.

Layer outputs and GEMM outputs must satisfy, element by element,
    |y - y_ref| / max(|y_ref|, RMS(y_ref)) <= 2e-2      (max relative error, floored by
                                                        the RMS so near-zeros do not explode)
and, over the tensor,
    mean|y - y_ref| / RMS(y_ref) <= 1e-3.
"""

import numpy as np

MAX_REL = 2e-2
MAE_REL = 1e-3


def rel_errors(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    if rms == 0.0:
        rms = 1.0
    err = np.abs(y - ref)
    max_rel = float((err / np.maximum(np.abs(ref), rms)).max()) if ref.size else 0.0
    mae = float(err.mean() / rms) if ref.size else 0.0
    return max_rel, mae


def assert_close(y, ref, max_rel=MAX_REL, mae=MAE_REL, what=""):
    mr, ma = rel_errors(y, ref)
    assert np.isfinite(np.asarray(y, np.float64)).all(), f"{what}: non-finite values"
    assert mr <= max_rel and ma <= mae, f"{what}: max_rel={mr:.3e} (<= {max_rel}), mae/rms={ma:.3e} (<= {mae})"
    return mr, ma


def bf16_to_f32(t):
    """torch BF16 tensor (any device) -> numpy float32."""
    return t.float().cpu().numpy()


def routing_margin(c_row, idx_row, n_groups, topk_groups, group_topn):
    """Smallest margin of one token's routing decisions (oracle scores c): between the
    last chosen and the best unchosen allowed expert, and between the last kept and the
    best dropped group score."""
    E = c_row.shape[0]
    gs = E // n_groups
    gsc = np.array([np.sort(c_row[g * gs:(g + 1) * gs])[::-1][:group_topn].sum(dtype=np.float64)
                    for g in range(n_groups)])
    srt = np.sort(gsc)[::-1]
    gap_g = srt[topk_groups - 1] - srt[topk_groups] if topk_groups < n_groups else np.inf
    kept = np.argsort(-gsc, kind="stable")[:topk_groups]
    allowed = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in kept])
    rest = np.setdiff1d(allowed, idx_row)
    gap_e = float(c_row[idx_row].min()) - float(c_row[rest].max()) if rest.size else np.inf
    return min(gap_g, gap_e)


def assert_fp8_decoded_close(got, ref, scale, what="", max_diff_frac=0.01, mae=MAE_REL):
    """Decoded FP8 tensors from two computations whose inputs differ in their last FP32
    bits: a value may land on the other side of an E4M3 rounding boundary, so each element
    may differ by one E4M3 step (1/8 of the value for normal codes, scale * 2^-9 in the
    subnormal range); few codes differ (beyond group scales an FP32 ulp apart), and the
    mean error stays within `mae` of the RMS.  `scale`: each element's group scale (broadcastable)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.broadcast_to(np.asarray(scale, np.float64), ref.shape)
    err = np.abs(got - ref)
    bound = 0.125 * np.abs(ref) + scale * 2.0 ** -9
    assert (err <= bound * (1 + 1e-6)).all(), f"{what}: an element moved by more than one E4M3 step"
    # a code change moves a value by >= 1/16 of it; a scale an FP32 ulp apart by ~1e-7
    moved = (err > 1e-4 * np.abs(ref) + scale * 2.0 ** -12).mean()
    assert moved <= max_diff_frac, f"{what}: {moved:.3%} of the codes differ"
    rms = np.sqrt(np.mean(ref ** 2)) or 1.0
    assert err.mean() / rms <= mae, f"{what}: mae/rms={err.mean() / rms:.3e}"
