"""GPU parity of the whole MoE layer forward against the oracle.

Tiny shape: every intermediate and the output, routed from identical logits (routing
bit-exact) and from the GPU's own router logits.  V3, decode and skewed shapes: the
router decisions of every token, and the outputs of sampled tokens computed one by one
by the oracle from the same synthetic weights."""

import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from fp8_block_scaled_bias_b300 import MoELayer, make_weights, ops
from tolerance import assert_close, bf16_to_f32, routing_margin

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_experts(cfg, pow2=False):
    qw = oracle.quant_128x128_pow2 if pow2 else oracle.quant_128x128
    ex = []
    for e in range(cfg.E + 1):
        w = [t.cpu().numpy() for t in workloads.gen_expert_f32(cfg, e, device="cuda")]
        ex.append(tuple(a for m in w for a in qw(m)))
    return ex


@pytest.fixture(scope="module")
def tiny():
    cfg = workloads.TINY
    w = make_weights(cfg, DEV)
    x = workloads.gen_x(cfg)
    return cfg, w, x, _oracle_experts(cfg)


def test_tiny_weights_quantised_like_oracle(tiny):
    cfg, w, x, ex = tiny
    for e in (0, 7, cfg.E):
        q1, s1, q3, s3, q2, s2 = ex[e]
        from fp8_block_scaled_bias_b300 import interleave_gate_up
        w13, s13 = interleave_gate_up(torch.from_numpy(q1), torch.from_numpy(s1),
                                      torch.from_numpy(q3), torch.from_numpy(s3))
        assert np.array_equal(w.w13[e].cpu().numpy(), w13.numpy())
        assert np.array_equal(w.s13[e].cpu().numpy(), s13.numpy())
        assert np.array_equal(w.w2[e].cpu().numpy(), q2)
        assert np.array_equal(w.s2[e].cpu().numpy(), s2)


def _compare_tiny(cfg, layer, ref, x, gate_tol=None):
    """gate_tol None: identical logits on both sides, gates within 16 float32 ulps;
    else an absolute tolerance (the GPU routed from its own logits)."""
    T, K = cfg.T, cfg.K
    for name in ("idx", "counts", "offsets", "row_token", "row_of"):
        got = getattr(layer, name).cpu().numpy()
        assert np.array_equal(got, ref[name]), name
    # the quantised activations, already in segment order
    tok = ref["row_token"]
    assert np.array_equal(layer.xq_rows.cpu().numpy(), ref["xq"][tok])
    assert np.array_equal(layer.sx_rows.cpu().numpy(), ref["sx"][:, tok])
    # from logits the GPU sigmoid uses expf: gates agree to a few float32 ulps
    g = layer.gate.cpu().numpy()
    if gate_tol is None:
        assert (np.abs(g - ref["gate"]) <= 16 * 2.0 ** -24 * ref["gate"] + 1e-12).all()
    else:
        assert np.abs(g - ref["gate"]).max() <= gate_tol
    # h is requantised from FP32 partial sums: decoded values agree to FP8 rounding
    hq = oracle.dequant_1x128(layer.hq.cpu().numpy(), layer.sh.cpu().numpy())
    hr = oracle.dequant_1x128(ref["hq"], ref["sh"])
    assert_close(hq, hr, max_rel=0.07, mae=5e-3, what="h")
    assert_close(bf16_to_f32(layer.y_rows), ref["Y"], what="expert rows")
    assert_close(bf16_to_f32(layer.y), ref["y"], what="layer output")


def test_tiny_layer_from_identical_logits(tiny):
    cfg, w, x, ex = tiny
    g = torch.Generator().manual_seed(5)
    logits = (torch.randn(cfg.T, cfg.E, generator=g) * 1.5).float()
    layer = MoELayer(cfg, w)
    layer.forward(x.to(DEV), logits=logits.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    ref = oracle.moe_layer(x.float().numpy(), w.centroids.cpu().numpy(), w.bias.cpu().numpy(),
                           ex, cfg.n_groups, cfg.topk_groups, cfg.K, logits=logits.numpy())
    _compare_tiny(cfg, layer, ref, x)
    # quantise-in-gather (the layer's path) equals quantise, then gather: identical bits
    xq, sx = ops.quant_1x128(x.to(DEV))
    xq_rows, sx_rows = ops.gather_rows(xq, sx, layer.row_token, layer.seg_end, layer.status)
    torch.cuda.synchronize()
    assert torch.equal(xq_rows, layer.xq_rows) and torch.equal(sx_rows, layer.sx_rows)
    # the one-call expert entry point runs the same kernels: identical bits
    hq, sh, y_rows = ops.swiglu_fwd(xq, sx, layer.row_token, layer.offsets,
                                    layer.rows, w.w13, w.s13, w.w2, w.s2, layer.status)
    torch.cuda.synchronize()
    assert torch.equal(hq, layer.hq) and torch.equal(sh, layer.sh)
    assert torch.equal(y_rows, layer.y_rows)


def test_tiny_layer_full_path(tiny):
    cfg, w, x, ex = tiny
    layer = MoELayer(cfg, w)
    layer.forward(x.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    ref = oracle.moe_layer(x.float().numpy(), w.centroids.cpu().numpy(), w.bias.cpu().numpy(),
                           ex, cfg.n_groups, cfg.topk_groups, cfg.K)
    z = layer.z.cpu().numpy()
    assert np.abs(z - ref["z"]).max() <= 1e-4 * np.abs(ref["z"]).max()
    if np.array_equal(layer.idx.cpu().numpy(), ref["idx"]):
        _compare_tiny(cfg, layer, ref, x, gate_tol=5e-4)
    else:                                     # a near-tie flipped: compare unaffected tokens
        same = (layer.idx.cpu().numpy() == ref["idx"]).all(1)
        assert same.mean() > 0.99
        assert_close(bf16_to_f32(layer.y)[same], ref["y"][same], what="layer output")


def test_tiny_layer_on_swapped_tiling(tiny, lib):
    """The tiny layer with both expert GEMMs on the swapped-operand tiling (weight rows on
    the MMA's M side, including its SwiGLU epilogue), every intermediate against the
    oracle from identical logits."""
    cfg, w, x, ex = tiny
    g = torch.Generator().manual_seed(5)
    logits = (torch.randn(cfg.T, cfg.E, generator=g) * 1.5).float()
    L = lib.load()
    try:
        L.moe_set_gemm_tiling(3)
        layer = MoELayer(cfg, w)
        layer.forward(x.to(DEV), logits=logits.to(DEV))
        torch.cuda.synchronize()
        layer.check_status()
    finally:
        L.moe_set_gemm_tiling(0)
    ref = oracle.moe_layer(x.float().numpy(), w.centroids.cpu().numpy(), w.bias.cpu().numpy(),
                           ex, cfg.n_groups, cfg.topk_groups, cfg.K, logits=logits.numpy())
    _compare_tiny(cfg, layer, ref, x)


def test_layer_is_deterministic(tiny):
    cfg, w, x, _ = tiny
    layer = MoELayer(cfg, w)
    xd = x.to(DEV)
    first = layer.forward(xd).clone()
    for _ in range(3):
        assert torch.equal(layer.forward(xd), first)


def test_residual_flag(tiny):
    cfg, w, x, _ = tiny
    layer = MoELayer(cfg, w)
    xd = x.to(DEV)
    y = layer.forward(xd).clone()
    assert torch.equal(layer.forward(xd, residual=True), y + xd)


# ---- V3-shaped configurations: all routing decisions, sampled outputs -------------------

@pytest.fixture(scope="module")
def v3_weights():
    return make_weights(workloads.V3, DEV)


def _routing_agrees(cfg, layer, x, bias):
    """The oracle's router on the oracle's own logits (float64).  Every token whose GPU
    decision differs must sit on a near-tie of the oracle's scores no wider than that
    token's own logit difference allows: a different expert set needs a decision margin
    below it, a different order of the same set needs two chosen scores that close.
    Returns the tokens routed identically, and the oracle's idx."""
    z_ref = oracle.router_logits(x.float().numpy(), layer.w.centroids.cpu().numpy())
    z = layer.z.cpu().numpy()
    assert np.abs(z - z_ref).max() <= 2e-5 * np.abs(z_ref).max()
    i_ref, g_ref = oracle.route(z_ref, bias, cfg.n_groups, cfg.topk_groups, cfg.group_topn, cfg.K)
    idx = layer.idx.cpu().numpy()
    same = (idx == i_ref).all(1)
    c = (oracle.sigmoid_f32(z_ref) + bias[None]).astype(np.float32)
    dz = np.abs(z.astype(np.float64) - z_ref).max(axis=1)
    for t in np.nonzero(~same)[0]:
        tol = dz[t] + 1e-6          # |dc| <= |dz| / 4; group scores add two c, margins two sides
        if set(idx[t]) != set(i_ref[t]):
            assert routing_margin(c[t], i_ref[t], cfg.n_groups, cfg.topk_groups,
                                  cfg.group_topn) < tol, t
        else:
            cs = c[t][i_ref[t]].astype(np.float64)
            assert np.min(np.abs(np.subtract.outer(cs, cs)) + np.eye(cfg.K)) < tol, t
    assert same.mean() >= 0.995
    g = layer.gate.cpu().numpy()
    assert np.abs(g[same] - g_ref[same]).max() <= 5e-4     # gates follow the logits
    return same, i_ref


_POOL = None


def _pool():
    """Process pool for the oracle's weight quantisation (spawned, never forked)."""
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        _POOL = cf.ProcessPoolExecutor(max_workers=max(1, min(24, (os.cpu_count() or 2) - 1)),
                                       mp_context=mp.get_context("spawn"))
        import atexit
        atexit.register(_POOL.shutdown)
    return _POOL


def _sampled_outputs(cfg, layer, x, bias, tokens, i_ref, pow2=False):
    """Oracle outputs of the sampled tokens; the experts they use are generated from the
    same seeds and quantised by the oracle (in parallel worker processes)."""
    need = sorted(set(int(e) for t in tokens for e in i_ref[t]) | {cfg.E})
    mats = []
    for e in need:
        mats.extend(t.cpu().numpy() for t in workloads.gen_expert_f32(cfg, e, device="cuda"))
    qw = oracle.quant_128x128_pow2 if pow2 else oracle.quant_128x128
    quant = list(_pool().map(qw, mats))
    q = {e: tuple(a for j in range(3) for a in quant[3 * i + j]) for i, e in enumerate(need)}
    return oracle.moe_layer_tokens(tokens, x.float().numpy()[tokens],
                                   layer.w.centroids.cpu().numpy(), bias, None, cfg.n_groups,
                                   cfg.topk_groups, cfg.K, expert_quantised=q.__getitem__,
                                   pow2=pow2)


def _steered_tokens(cfg, layer, same, rng, n):
    """n tokens (routed identically on both sides) chosen where a GEMM tile edge can break:
    the last row of segments whose length is off the 128-row grid, the first and last rows
    of the busiest expert, the last token (the shared segment's last M tile, partly filled
    when T % 128 != 0) and tokens on 1-row segments; random tokens fill the rest."""
    counts = layer.counts.cpu().numpy()
    offs = layer.offsets.cpu().numpy()
    row_token = layer.row_token.cpu().numpy()
    picks = []
    ragged = [e for e in range(cfg.E) if counts[e] % 128 != 0]
    for e in rng.permutation(ragged)[:4]:
        picks.append(int(row_token[offs[e + 1] - 1]))
    hot = int(np.argmax(counts))
    picks += [int(row_token[offs[hot]]), int(row_token[offs[hot + 1] - 1])]
    picks.append(cfg.T - 1)
    for e in [e for e in range(cfg.E) if counts[e] == 1][:2]:
        picks.append(int(row_token[offs[e]]))
    picks = [t for t in dict.fromkeys(picks) if same[t]]
    rest = np.setdiff1d(np.nonzero(same)[0], picks)
    picks += rng.choice(rest, max(0, n - len(picks)), replace=False).tolist()
    return sorted(picks[:max(n, len(picks))])


def _check_config(cfg, w, n_sample, mx=False):
    x = workloads.gen_x(cfg)
    layer = MoELayer(cfg, w, mx=mx)
    layer.forward(x.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    bias = w.bias.cpu().numpy()
    same, i_ref = _routing_agrees(cfg, layer, x, bias)
    # permutation invariants on the GPU's own routing
    counts = layer.counts.cpu().numpy()
    assert counts.sum() == cfg.T * cfg.K
    assert np.array_equal(counts, np.bincount(layer.idx.cpu().numpy().ravel(), minlength=cfg.E))
    if same.all():
        ref = oracle.permute(i_ref, cfg.E)
        for got, want in zip((layer.counts, layer.offsets, layer.row_token, layer.row_of), ref):
            assert np.array_equal(got.cpu().numpy(), want)
    rng = np.random.default_rng(cfg.T)
    tokens = _steered_tokens(cfg, layer, same, rng, n_sample)
    part = _sampled_outputs(cfg, layer, x, bias, tokens, i_ref, pow2=mx)
    y = bf16_to_f32(layer.y)[tokens]
    assert_close(y, part["y"], what=f"{cfg.name} sampled tokens" + (" (MX)" if mx else ""))
    return layer


def test_v3_layer(v3_weights):
    _check_config(workloads.V3, v3_weights, n_sample=16)


def test_decode_layer(v3_weights):
    _check_config(workloads.DECODE, v3_weights, n_sample=16)


def test_skewed_layer_and_bias_update(v3_weights):
    cfg = workloads.SKEWED
    w = v3_weights
    saved = w.bias.clone()
    try:
        w.bias.copy_(workloads.gen_bias(cfg).to(DEV))
        layer = _check_config(cfg, w, n_sample=16)
        counts = layer.counts.cpu().numpy()
        # the workload's calibrated skew (10x on the oracle's routing; near-ties may move
        # a few pairs on the GPU's own logits)
        assert 9.0 <= counts.max() / counts.mean() <= 11.0
        before = w.bias.cpu().numpy().copy()
        layer.bias_update(0.001)
        assert np.array_equal(w.bias.cpu().numpy(),
                              oracle.bias_update(before, counts, cfg.T, cfg.K, 0.001))
        x = workloads.gen_x(cfg).to(DEV)
        layer.forward(x)
        torch.cuda.synchronize()
        layer.check_status()
        c2 = layer.counts.cpu().numpy()
        over = counts * cfg.E > cfg.T * cfg.K
        assert c2[over].sum() <= counts[over].sum()      # overloaded experts lose load
    finally:
        w.bias.copy_(saved)


# ---- the MX-native variant (power-of-two scales applied by the tensor core) -------------

def test_tiny_mx_layer_from_identical_logits():
    cfg = workloads.TINY
    w = make_weights(cfg, DEV, pow2=True)
    ex = _oracle_experts(cfg, pow2=True)
    x = workloads.gen_x(cfg)
    g = torch.Generator().manual_seed(5)
    logits = (torch.randn(cfg.T, cfg.E, generator=g) * 1.5).float()
    layer = MoELayer(cfg, w, mx=True)
    layer.forward(x.to(DEV), logits=logits.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    ref = oracle.moe_layer(x.float().numpy(), w.centroids.cpu().numpy(), w.bias.cpu().numpy(),
                           ex, cfg.n_groups, cfg.topk_groups, cfg.K, logits=logits.numpy(),
                           pow2=True)
    for name in ("idx", "counts", "offsets", "row_token", "row_of"):
        assert np.array_equal(getattr(layer, name).cpu().numpy(), ref[name]), name
    tok = ref["row_token"]
    assert np.array_equal(layer.xq_rows.cpu().numpy(), ref["xq"][tok])
    assert np.array_equal(layer.sx_rows.cpu().numpy(), ref["sx"][:, tok])
    sh = layer.sh.cpu().numpy()
    assert (np.frexp(sh.astype(np.float64))[0] == 0.5).all()        # powers of two
    hq = oracle.dequant_1x128(layer.hq.cpu().numpy(), sh)
    assert_close(hq, oracle.dequant_1x128(ref["hq"], ref["sh"]), max_rel=0.07, mae=5e-3,
                 what="h (MX)")
    assert_close(bf16_to_f32(layer.y_rows), ref["Y"], what="expert rows (MX)")
    assert_close(bf16_to_f32(layer.y), ref["y"], what="layer output (MX)")


def test_v3_and_decode_mx_layer_sampled_tokens():
    """The MX-native layer at the V3 shape (the block-scaled tensor-core GEMMs) and on the
    decode batch (short segments: the swapped-operand kernel with power-of-two scales)."""
    w = make_weights(workloads.V3, DEV, pow2=True)
    try:
        _check_config(workloads.V3, w, n_sample=16, mx=True)
        _check_config(workloads.DECODE, w, n_sample=16, mx=True)
    finally:
        del w
        torch.cuda.empty_cache()
