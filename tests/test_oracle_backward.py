"""Pins of the oracle's expert backward (DeepSeek-V3 book, ch. 17 "One linear layer
creates three GEMMs", "SwiGLU recomputation"; ch. 16 "Why transposition is not trivial").

Each piece is held to something other than itself: the SwiGLU derivative to torch
autograd in float64; the 128x1 regrouping to the (pinned) forward power-of-two quantiser
run on the transposed matrix, to the power-of-two rule's closed form and to segment
isolation; the Wgrad GEMM to a float64 matmul of dequantised operands and to closed
forms (segment lengths, empty experts); the whole expert backward to float64 autograd of
the unquantised expert, within FP8 quantisation error."""

import numpy as np
import torch

import oracle
import workloads


def _rng(seed):
    return np.random.default_rng(seed)


def test_swiglu_backward_matches_autograd():
    rng = _rng(0)
    g = (rng.standard_normal(4096) * 4).astype(np.float32)
    g[:5] = [0.0, -30.0, 30.0, 1e-3, -1e-3]
    u = rng.standard_normal(4096).astype(np.float32)
    dh = rng.standard_normal(4096).astype(np.float32)
    gt = torch.tensor(g, dtype=torch.float64, requires_grad=True)
    ut = torch.tensor(u, dtype=torch.float64, requires_grad=True)
    h_t = torch.nn.functional.silu(gt) * ut
    h_t.backward(torch.tensor(dh, dtype=torch.float64))
    h, dg, du = oracle.swiglu_backward(g, u, dh)
    for got, ref in ((h, h_t.detach()), (dg, gt.grad), (du, ut.grad)):
        ref = ref.numpy()
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        assert (np.abs(got.astype(np.float64) - ref) <= ulp + 1e-300).all()
    # dG and dU are not interchangeable, and the gate (not the up value) enters silu
    assert not np.allclose(dg, du)


def test_regroup_128x1_single_segment_is_pow2_1x128_of_transpose():
    rng = _rng(1)
    x = (rng.standard_normal((256, 384)) * np.exp(rng.uniform(-6, 6, (1, 384)))).astype(np.float32)
    qT, sT, pad = oracle.quant_128x1_pow2_segments(x, [0, 256])
    q_ref, s_ref = oracle.quant_1x128_pow2(np.ascontiguousarray(x.T))      # [384, 256]
    assert pad.tolist() == [0, 256]
    assert np.array_equal(qT, q_ref)
    assert np.array_equal(sT, s_ref)                                      # [2, 384]


def test_regroup_128x1_segments_padding_and_isolation():
    rng = _rng(2)
    counts = [130, 0, 1, 127]
    seg = np.concatenate([[0], np.cumsum(counts)])
    R, C = int(seg[-1]), 256
    x = rng.standard_normal((R, C)).astype(np.float32)
    x[130:131] *= 1e4                      # expert 2's single row is huge
    qT, sT, pad = oracle.quant_128x1_pow2_segments(x, seg)
    assert pad.tolist() == [0, 256, 256, 384, 512]
    assert qT.shape == (C, 512) and sT.shape == (4, C)
    # padded rows hold code 0
    dec = oracle.e4m3_decode(qT)
    assert (qT[:, 130:256] == 0).all() and (qT[:, 257:384] == 0).all() and (qT[:, 511] == 0).all()
    # scales: smallest power of two with 448 s >= amax over the block's own rows only
    for rb, (r0, r1) in enumerate([(0, 128), (128, 130), (130, 131), (131, 258)]):
        amax = np.abs(x[r0:r1]).max(axis=0).astype(np.float64)
        s = sT[rb].astype(np.float64)
        assert (np.log2(s) == np.round(np.log2(s))).all()
        assert (448 * s >= amax).all() and (448 * s / 2 < amax).all()
    # the huge row did not leak into its neighbours' scales
    assert sT[3].max() < 1.0 and sT[1].max() < 1.0
    # reconstruction within half an E4M3 step of the group scale
    for rb, (r0, r1, p0) in enumerate([(0, 128, 0), (128, 130, 128), (130, 131, 256),
                                       (131, 258, 384)]):
        rec = dec[:, p0:p0 + (r1 - r0)].T * sT[rb][None, :].astype(np.float64)
        assert (np.abs(rec - x[r0:r1]) <= sT[rb][None, :] * 16.0 + 1e-30).all()


def test_wgrad_equals_dequantised_matmul_per_segment():
    rng = _rng(3)
    counts = [200, 0, 5, 128]
    seg = np.concatenate([[0], np.cumsum(counts)])
    R = int(seg[-1])
    a = rng.standard_normal((R, 256)).astype(np.float32)
    b = rng.standard_normal((R, 384)).astype(np.float32)
    aT, saT, pad = oracle.quant_128x1_pow2_segments(a, seg)
    bT, sbT, _ = oracle.quant_128x1_pow2_segments(b, seg)
    got = oracle.wgrad(aT, saT, bT, sbT, pad)
    ad = oracle.e4m3_decode(aT) * np.repeat(saT.T.astype(np.float64), 128, axis=1)
    bd = oracle.e4m3_decode(bT) * np.repeat(sbT.T.astype(np.float64), 128, axis=1)
    for e in range(4):
        p0, p1 = pad[e], pad[e + 1]
        ref = ad[:, p0:p1] @ bd[:, p0:p1].T
        assert np.allclose(got[e], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max(initial=1.0))
    assert (got[1] == 0).all()
    # against the unquantised product: FP8 error only
    ref = a[:200].astype(np.float64).T @ b[:200].astype(np.float64)
    assert np.abs(got[0] - ref).mean() / np.sqrt((ref ** 2).mean()) < 0.05


def test_wgrad_closed_form_counts_rows():
    counts = [130, 0, 1, 256]
    seg = np.concatenate([[0], np.cumsum(counts)])
    R = int(seg[-1])
    ones = np.ones((R, 128), np.float32)
    aT, saT, pad = oracle.quant_128x1_pow2_segments(ones, seg)
    bT, sbT, _ = oracle.quant_128x1_pow2_segments(2 * ones, seg)
    got = oracle.wgrad(aT, saT, bT, sbT, pad)
    for e, n in enumerate(counts):
        assert (got[e] == 2.0 * n).all()


def _expert_fixture(seed=4, d=256, f=256, counts=(150, 0, 40, 129)):
    rng = _rng(seed)
    seg = np.concatenate([[0], np.cumsum(counts)])
    R = int(seg[-1])
    x = torch.tensor(rng.standard_normal((R, d)), dtype=torch.float32).to(torch.bfloat16)
    dy = torch.tensor(rng.standard_normal((R, d)) * 0.1, dtype=torch.float32).to(torch.bfloat16)
    x, dy = x.float().numpy(), dy.float().numpy()
    experts = []
    for e in range(len(counts)):
        w1 = (rng.standard_normal((f, d)) * 0.05).astype(np.float32)
        w3 = (rng.standard_normal((f, d)) * 0.05).astype(np.float32)
        w2 = (rng.standard_normal((d, f)) * 0.05).astype(np.float32)
        experts.append(tuple(a for w in (w1, w3, w2) for a in oracle.quant_128x128(w)))
    return seg, x, dy, experts


def test_expert_backward_against_float64_autograd():
    """The unquantised expert y = (silu(x W1^T) * (x W3^T)) W2^T on the dequantised
    weights and the same x, differentiated by autograd in float64: the FP8 backward
    matches it within FP8 quantisation error, for every input and weight gradient."""
    seg, x, dy, experts = _expert_fixture()
    xq, sx = oracle.quant_1x128(x)
    guq = np.zeros((x.shape[0], 512), np.uint8)
    sgu = np.ones((4, x.shape[0]), np.float32)
    for e in range(4):
        r0, r1 = seg[e], seg[e + 1]
        if r1 > r0:
            w1q, s1, w3q, s3 = experts[e][:4]
            guq[r0:r1], sgu[:, r0:r1] = oracle.swiglu_cache(xq[r0:r1], sx[:, r0:r1], w1q, s1,
                                                            w3q, s3)
    out = oracle.expert_backward(seg, x, dy, guq, sgu, experts)

    def rel(a, b):
        return np.abs(a - b).mean() / np.sqrt((b ** 2).mean())

    for e in range(4):
        r0, r1 = seg[e], seg[e + 1]
        w = [torch.tensor(oracle.dequant_128x128(experts[e][2 * i], experts[e][2 * i + 1]),
                          dtype=torch.float64, requires_grad=True) for i in range(3)]
        if r1 == r0:
            assert (out["dw1"][e] == 0).all() and (out["dw2"][e] == 0).all()
            continue
        xt = torch.tensor(x[r0:r1], dtype=torch.float64, requires_grad=True)
        y = (torch.nn.functional.silu(xt @ w[0].T) * (xt @ w[1].T)) @ w[2].T
        y.backward(torch.tensor(dy[r0:r1], dtype=torch.float64))
        assert rel(out["dx"][r0:r1], xt.grad.numpy()) < 0.06
        assert rel(out["dw1"][e], w[0].grad.numpy()) < 0.06
        assert rel(out["dw3"][e], w[1].grad.numpy()) < 0.06
        assert rel(out["dw2"][e], w[2].grad.numpy()) < 0.06


def test_expert_backward_zero_gradient_is_zero():
    seg, x, dy, experts = _expert_fixture(seed=5, counts=(130, 3))
    R = x.shape[0]
    guq = workloads.gen_fp8_codes(R, 512).numpy()
    sgu = np.ones((4, R), np.float32)
    out = oracle.expert_backward(seg, x, np.zeros_like(dy), guq, sgu, experts)
    for k in ("dh", "dg", "du", "dx", "dw1", "dw3", "dw2"):
        assert (out[k] == 0).all(), k


def test_combine_backward_rows_matches_autograd():
    """The rows' gradient of the combine, from torch autograd of the combine itself (float64),
    rounded to BF16 the way the expert backward takes it."""
    rng = _rng(6)
    T, K, d = 7, 3, 16
    row_of = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    gate = rng.uniform(0.05, 1.0, (T, K)).astype(np.float32)
    dy = torch.tensor(rng.standard_normal((T, d)), dtype=torch.float32).to(torch.bfloat16)
    Y = torch.zeros(T * K + T, d, dtype=torch.float64, requires_grad=True)
    y = Y[T * K:T * K + T] + sum(torch.tensor(gate[:, k], dtype=torch.float64)[:, None] *
                                 Y[torch.tensor(row_of[:, k], dtype=torch.long)] for k in range(K))
    y.backward(dy.double())
    got = oracle.combine_backward_rows(dy.float().numpy(), gate, row_of, T * K, T * K + T)
    ref = Y.grad.numpy()
    assert np.array_equal(got[T * K:], dy.float().numpy())        # the shared rows: dy itself
    # the routed rows: the exact product rounded once to BF16 (at most half a BF16 ulp)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30).all()
    assert np.array_equal(got, oracle.bf16_round(got))
