"""GPU parity of the expert backward (training) against the oracle's FP8 backward
("DeepSeek-V3" book, ch. 17 "One linear layer creates three GEMMs", "SwiGLU
recomputation"; ch. 16 "Why transposition is not trivial").

Bit-exact: the transposed weights, the combine's row gradients, the padded offsets and
the 128x1 power-of-two regrouping (codes and scales).  Within the R12 tolerances: the
Wgrad GEMM (exact per-block products, FP32 accumulation), the SwiGLU backward's outputs
(FP32 with expf against float64) and the whole tiny layer backward."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from fp8_block_scaled_bias_b300 import MoELayer, make_weights, ops
from tolerance import assert_close, assert_fp8_decoded_close, bf16_to_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _seg(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def test_weight_transposes_bit_exact():
    rng = np.random.default_rng(0)
    G, R, C = 3, 512, 384
    w = torch.from_numpy(rng.integers(0, 256, (G, R, C), dtype=np.uint8))
    s = torch.from_numpy(rng.uniform(0.5, 2.0, (G, R // 128, C // 128)).astype(np.float32))
    wT, sT = ops.transpose_128x128(w.to(DEV), s.to(DEV))
    assert np.array_equal(wT.cpu().numpy(), w.numpy().transpose(0, 2, 1))
    assert np.array_equal(sT.cpu().numpy(), s.numpy().transpose(0, 2, 1))
    # gate/up interleaved in 64-row blocks -> [gate; up]^T
    wT, sT = ops.transpose_128x128(w.to(DEV), s.to(DEV), gate_up_interleaved=True)
    wn = w.numpy().reshape(G, R // 128, 2, 64, C)
    cat = np.concatenate([wn[:, :, 0].reshape(G, R // 2, C), wn[:, :, 1].reshape(G, R // 2, C)], 1)
    sn = s.numpy().reshape(G, R // 256, 2, C // 128)
    scat = np.concatenate([sn[:, :, 0], sn[:, :, 1]], 1)
    assert np.array_equal(wT.cpu().numpy(), cat.transpose(0, 2, 1))
    assert np.array_equal(sT.cpu().numpy(), scat.transpose(0, 2, 1))


def test_combine_bwd_rows_bit_exact():
    rng = np.random.default_rng(1)
    T, K, d = 37, 4, 256
    row_of = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    gate = rng.uniform(0.01, 1.0, (T, K)).astype(np.float32)
    dy = torch.tensor(rng.standard_normal((T, d)), dtype=torch.float32).to(torch.bfloat16)
    st = ops.new_status(DEV)
    got = ops.combine_bwd_rows(dy.to(DEV), torch.from_numpy(gate).to(DEV),
                               torch.from_numpy(row_of).to(DEV), T * K, T * K + T, status=st)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    ref = oracle.combine_backward_rows(dy.float().numpy(), gate, row_of, T * K, T * K + T)
    assert np.array_equal(bf16_to_f32(got), ref)


@pytest.mark.parametrize("gather", [False, True])
def test_regroup_128x1_bit_exact(gather):
    rng = np.random.default_rng(2)
    counts = [130, 0, 1, 256, 77, 0, 128, 300]
    seg = _seg(counts)
    R, C, G = int(seg[-1]), 384, len(counts)
    src_rows = 500 if gather else R
    x = torch.tensor(rng.standard_normal((src_rows, C)) *
                     np.exp(rng.uniform(-4, 4, (1, C))), dtype=torch.float32).to(torch.bfloat16)
    rows = rng.integers(0, src_rows, R).astype(np.int32) if gather else None
    offsets = torch.from_numpy(seg).to(DEV)
    st = ops.new_status(DEV)
    pad = ops.segment_pad_offsets(offsets, G, status=st)
    kcap = ops.padded_rows_cap(R, G)
    qT, sT = ops.quant_128x1_pow2(x.to(DEV), offsets, pad, kcap, status=st,
                                  rows=None if rows is None else torch.from_numpy(rows).to(DEV))
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    xr = x.float().numpy()[rows] if gather else x.float().numpy()
    q_ref, s_ref, pad_ref = oracle.quant_128x1_pow2_segments(xr, seg)
    P = int(pad_ref[-1])
    assert np.array_equal(pad.cpu().numpy(), pad_ref)
    assert np.array_equal(qT.cpu().numpy()[:, :P], q_ref)
    assert np.array_equal(sT.cpu().numpy()[:P // 128], s_ref)


def _pow2(shape, rng, lo=-8, hi=2):
    return np.exp2(rng.integers(lo, hi + 1, shape)).astype(np.float32)


@pytest.mark.parametrize("I,J", [(256, 384), (128, 640)])
def test_wgrad_gemm_ragged_experts(I, J):
    rng = np.random.default_rng(3)
    counts = [200, 0, 5, 128, 0, 513, 1]
    seg = _seg(counts)
    pad = oracle.padded_offsets(seg).astype(np.int32)
    G, kcap = len(counts), int(pad[-1]) + 256          # slack past the last block
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    aT = finite[rng.integers(0, finite.size, (I, kcap))]
    bT = finite[rng.integers(0, finite.size, (J, kcap))]
    saT = _pow2((kcap // 128, I), rng)
    sbT = _pow2((kcap // 128, J), rng)
    st = ops.new_status(DEV)
    dW = ops.wgrad(*(torch.from_numpy(a).to(DEV) for a in (aT, saT, bT, sbT, pad)), status=st)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    ref = oracle.wgrad(aT, saT, bT, sbT, pad)
    got = dW.cpu().numpy()
    for e in range(G):
        if counts[e] == 0:
            assert (got[e] == 0).all(), e
        else:
            assert_close(got[e], ref[e], what=f"wgrad expert {e}")
            # FP32 accumulation of exact block products: within a few FP32 ulps of the sum
            # of magnitudes
            assert np.abs(got[e] - ref[e]).max() <= 1e-5 * np.abs(ref[e]).max()


def test_wgrad_reports_bad_pad_table():
    aT = torch.zeros(128, 256, dtype=torch.uint8, device=DEV)
    s = torch.ones(2, 128, device=DEV)
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384]):
        st = ops.new_status(DEV)
        ops.wgrad(aT, s, aT, s, torch.tensor(bad, dtype=torch.int32, device=DEV), status=st)
        torch.cuda.synchronize()
        assert ops.status_value(st) == -6, bad


@pytest.mark.parametrize("counts,f", [
    ([130, 0, 77, 256, 1], 256),
    # more tiles than SMs: each persistent block streams several tiles through its two
    # shared-memory input buffers
    ([1300, 0, 777, 2560, 1, 129], 1024),
])
def test_swiglu_bwd_against_oracle(counts, f):
    rng = np.random.default_rng(4)
    seg = _seg(counts)
    R, G = int(seg[-1]), len(counts)
    g = (rng.standard_normal((R, f)) * 3).astype(np.float32)
    u = rng.standard_normal((R, f)).astype(np.float32)
    gq, sg = oracle.quant_1x128(g)
    uq, su = oracle.quant_1x128(u)
    guq = np.concatenate([gq, uq], 1)
    sgu = np.concatenate([sg, su], 0)
    dh = torch.tensor(rng.standard_normal((R, f)), dtype=torch.float32).to(torch.bfloat16)
    offsets = torch.from_numpy(seg).to(DEV)
    pad = ops.segment_pad_offsets(offsets, G)
    kcap = ops.padded_rows_cap(R, G)
    dguq, sdgu, hT, shT, dguT, sdguT = ops.swiglu_bwd(
        torch.from_numpy(guq).to(DEV), torch.from_numpy(sgu).to(DEV), dh.to(DEV), offsets, pad,
        kcap)
    torch.cuda.synchronize()
    gd = oracle.dequant_rows_1x128_f32(guq, sgu)
    h, dg, du = oracle.swiglu_backward(gd[:, :f], gd[:, f:], dh.float().numpy())
    P = int(oracle.padded_offsets(seg)[-1])
    # the 1x128 gradient rows, decoded
    sd = sdgu.cpu().numpy()
    got = oracle.dequant_1x128(dguq.cpu().numpy(), sd)
    dgu = np.concatenate([dg, du], 1)
    ref = oracle.dequant_1x128(*oracle.quant_1x128(dgu))
    assert_fp8_decoded_close(got, ref, np.repeat(sd.T, 128, 1), what="dG|dU 1x128")
    # the 128x1 tiles, decoded, against the oracle's regrouping of its own values
    for name, qT, sT, val in (("h^T", hT, shT, h), ("[dG|dU]^T", dguT, sdguT, dgu)):
        q_ref, s_ref, _ = oracle.quant_128x1_pow2_segments(val, seg)
        qg, sgot = qT.cpu().numpy()[:, :P], sT.cpu().numpy()[:P // 128]
        # scales agree except where FP32 and float64 put a column max on two sides of a
        # power of two
        assert (sgot == s_ref).mean() > 0.99, name
        sc = np.repeat(sgot.T.astype(np.float64), 128, 1)
        dec = oracle.e4m3_decode(qg) * sc
        dec_ref = oracle.e4m3_decode(q_ref) * np.repeat(s_ref.T.astype(np.float64), 128, 1)
        assert_fp8_decoded_close(dec, dec_ref, np.maximum(sc, np.repeat(s_ref.T, 128, 1)),
                                 what=name)


@pytest.fixture(scope="module")
def tiny_train():
    cfg = workloads.TINY
    w = make_weights(cfg, DEV)
    x = workloads.gen_x(cfg)
    layer = MoELayer(cfg, w, train=True)
    layer.forward(x.to(DEV))
    g = torch.Generator().manual_seed(11)
    dy = (torch.randn(cfg.T, cfg.d, generator=g) * 0.1).to(torch.bfloat16)
    out = layer.backward(dy.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    ex = []
    for e in range(cfg.E + 1):
        wf = [t.cpu().numpy() for t in workloads.gen_expert_f32(cfg, e, device="cuda")]
        ex.append(tuple(a for m in wf for a in oracle.quant_128x128(m)))
    return cfg, w, x, dy, layer, out, ex


def test_tiny_training_cache_against_oracle(tiny_train):
    cfg, w, x, dy, layer, out, ex = tiny_train
    seg = layer.offsets.cpu().numpy()
    xq = layer.xq_rows.cpu().numpy()
    sx = layer.sx_rows.cpu().numpy()
    guq, sgu = layer.guq.cpu().numpy(), layer.sgu.cpu().numpy()
    got = oracle.dequant_rows_1x128_f32(guq, sgu)
    for e in range(cfg.E + 1):
        r0, r1 = seg[e], seg[e + 1]
        if r1 == r0:
            continue
        gq, sg = oracle.swiglu_cache(xq[r0:r1], sx[:, r0:r1], ex[e][0], ex[e][1], ex[e][2],
                                     ex[e][3])
        ref = oracle.dequant_rows_1x128_f32(gq, sg)
        sc = np.maximum(np.repeat(sgu[:, r0:r1].T, 128, 1), np.repeat(sg.T, 128, 1))
        assert_fp8_decoded_close(got[r0:r1], ref, sc, what=f"g|u cache expert {e}")


def test_tiny_layer_backward_against_oracle(tiny_train):
    """The whole expert backward of the tiny layer: the oracle takes the GPU's own forward
    cache and row gradients (each checked separately) and recomputes every step."""
    cfg, w, x, dy, layer, out, ex = tiny_train
    T, K = cfg.T, cfg.K
    seg = layer.offsets.cpu().numpy()
    row_of = layer.row_of.cpu().numpy()
    gate = layer.gate.cpu().numpy()
    dy_rows = oracle.combine_backward_rows(dy.float().numpy(), gate, row_of, T * K, layer.rows)
    assert np.array_equal(bf16_to_f32(out["dy_rows"]), dy_rows)
    x_rows = x.float().numpy()[layer.row_token.cpu().numpy()]
    ref = oracle.expert_backward(seg, x_rows, dy_rows, layer.guq.cpu().numpy(),
                                 layer.sgu.cpu().numpy(), ex)
    assert np.array_equal(out["pad"].cpu().numpy(), ref["pad"])
    P = int(ref["pad"][-1])
    # the regrouped dY and X are bit-exact (same BF16 inputs, exact power-of-two division)
    assert np.array_equal(out["dyT"].cpu().numpy()[:, :P], ref["dyT"])
    assert np.array_equal(out["xT"].cpu().numpy()[:, :P], ref["xT"])
    assert np.array_equal(out["sxT"].cpu().numpy()[:P // 128], ref["sxT"])
    assert_close(bf16_to_f32(out["dh"]), ref["dh"], what="dh (down Dgrad)")
    assert_close(bf16_to_f32(out["dx_rows"]), ref["dx"], what="dX rows (gate/up Dgrad)")
    # the token gradient: the rows of each token summed (the combine with unit gates)
    dx_ref = oracle.combine(ref["dx"], row_of, np.ones((T, K), np.float32), T * K)
    assert_close(bf16_to_f32(out["dx"]), dx_ref, what="dx")
    dw13 = out["dw13"].cpu().numpy()
    dw2 = out["dw2"].cpu().numpy()
    for e in range(cfg.E + 1):
        if seg[e + 1] == seg[e]:
            assert (dw13[e] == 0).all() and (dw2[e] == 0).all()
            continue
        f = cfg.f
        assert_close(dw13[e, :f], ref["dw1"][e], what=f"dW1 expert {e}")
        assert_close(dw13[e, f:], ref["dw3"][e], what=f"dW3 expert {e}")
        assert_close(dw2[e], ref["dw2"][e], what=f"dW2 expert {e}")


def test_v3_width_backward_sampled(lib):
    """The backward at V3 width (d=7168, f=2048; 32 experts + the shared one, T=512, top-8):
    the row gradients bit-exact; the regrouped dY and X of two experts bit-exact; sampled
    rows of both Dgrads, sampled output rows of both Wgrads (from the GPU's own regrouped
    operands) and sampled tokens of dx against the oracle."""
    cfg = workloads.V3_E32
    T, K, d, f = cfg.T, cfg.K, cfg.d, cfg.f
    w = make_weights(cfg, DEV)
    x = workloads.gen_x(cfg)
    layer = MoELayer(cfg, w, train=True)
    layer.forward(x.to(DEV))
    g = torch.Generator().manual_seed(13)
    dy = (torch.randn(T, d, generator=g) * 0.1).to(torch.bfloat16)
    out = layer.backward(dy.to(DEV))
    torch.cuda.synchronize()
    layer.check_status()
    seg = layer.offsets.cpu().numpy()
    row_of, gate = layer.row_of.cpu().numpy(), layer.gate.cpu().numpy()
    dy_rows = oracle.combine_backward_rows(dy.float().numpy(), gate, row_of, T * K, layer.rows)
    assert np.array_equal(bf16_to_f32(out["dy_rows"]), dy_rows)
    pad = oracle.padded_offsets(seg)
    assert np.array_equal(out["pad"].cpu().numpy(), pad)
    counts = np.diff(seg)
    experts = [int(np.argmax(counts[:cfg.E])), cfg.E]        # the busiest and the shared one
    x_rows = x.float().numpy()[layer.row_token.cpu().numpy()]
    rng = np.random.default_rng(3)
    for e in experts:
        r0, r1, p0, p1 = seg[e], seg[e + 1], pad[e], pad[e + 1]
        sub = np.array([0, r1 - r0])
        q_ref, s_ref, _ = oracle.quant_128x1_pow2_segments(dy_rows[r0:r1], sub)
        assert np.array_equal(out["dyT"].cpu().numpy()[:, p0:p1], q_ref)
        assert np.array_equal(out["sdyT"].cpu().numpy()[p0 // 128:p1 // 128], s_ref)
        q_ref, s_ref, _ = oracle.quant_128x1_pow2_segments(x_rows[r0:r1], sub)
        assert np.array_equal(out["xT"].cpu().numpy()[:, p0:p1], q_ref)
        assert np.array_equal(out["sxT"].cpu().numpy()[p0 // 128:p1 // 128], s_ref)
        # Wgrad on sampled output rows, from the GPU's own 128x1 operands
        wq = [t.cpu().numpy() for t in workloads.gen_expert_f32(cfg, e, device="cuda")]
        rows_i = np.sort(rng.choice(d, 24, replace=False))
        ref = oracle.wgrad(out["dyT"].cpu().numpy()[rows_i][:, p0:p1],
                           out["sdyT"].cpu().numpy()[p0 // 128:p1 // 128][:, rows_i],
                           out["hT"].cpu().numpy()[:, p0:p1],
                           out["shT"].cpu().numpy()[p0 // 128:p1 // 128],
                           np.array([0, p1 - p0]))[0]
        assert_close(out["dw2"][e].cpu().numpy()[rows_i], ref, what=f"dW2 rows, expert {e}")
        rows_c = np.sort(rng.choice(2 * f, 24, replace=False))
        ref = oracle.wgrad(out["dguT"].cpu().numpy()[rows_c][:, p0:p1],
                           out["sdguT"].cpu().numpy()[p0 // 128:p1 // 128][:, rows_c],
                           out["xT"].cpu().numpy()[:, p0:p1],
                           out["sxT"].cpu().numpy()[p0 // 128:p1 // 128],
                           np.array([0, p1 - p0]))[0]
        assert_close(out["dw13"][e].cpu().numpy()[rows_c], ref, what=f"dW13 rows, expert {e}")
        # Dgrads of sampled rows of this expert
        w1q, s1 = oracle.quant_128x128(wq[0])
        w3q, s3 = oracle.quant_128x128(wq[1])
        w2q, s2 = oracle.quant_128x128(wq[2])
        rr = np.sort(rng.choice(np.arange(r0, r1), min(8, r1 - r0), replace=False))
        dyq, sdy = oracle.quant_1x128(dy_rows[rr])
        dh_ref = oracle.bf16_round(oracle.blockscaled_gemm(dyq, sdy, np.ascontiguousarray(w2q.T),
                                                           np.ascontiguousarray(s2.T)))
        assert_close(bf16_to_f32(out["dh"])[rr], dh_ref, what=f"dh rows, expert {e}")
        wcat_t = np.ascontiguousarray(np.concatenate([w1q, w3q], 0).T)
        scat_t = np.ascontiguousarray(np.concatenate([s1, s3], 0).T)
        dx_ref = oracle.bf16_round(oracle.blockscaled_gemm(
            out["dguq"].cpu().numpy()[rr], out["sdgu"].cpu().numpy()[:, rr], wcat_t, scat_t))
        assert_close(bf16_to_f32(out["dx_rows"])[rr], dx_ref, what=f"dX rows, expert {e}")
    # dx of sampled tokens: the sum of their rows' dX (unit gates), from the GPU's rows
    toks = np.sort(rng.choice(T, 16, replace=False))
    dxr = bf16_to_f32(out["dx_rows"])
    ref = oracle.combine(np.concatenate([dxr[row_of[toks].ravel()], dxr[T * K + toks]]),
                         np.arange(16 * K, dtype=np.int32).reshape(16, K),
                         np.ones((16, K), np.float32), 16 * K)
    assert_close(bf16_to_f32(out["dx"])[toks], ref, what="dx tokens")
