"""Pins of the oracle permutation (numpy's stable argsort, conservation, inverse maps)
and of the block-scaled GEMM / SwiGLU / combine (closed forms, and the definitional
identity with a float64 matmul of operands decoded by torch's float8 type)."""

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import workloads


def test_permute_is_stable_argsort_and_conserves_pairs():
    rng = np.random.default_rng(0)
    T, K, E = 300, 4, 16
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, row_token, row_of = oracle.permute(idx, E, include_shared=True)
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")                         # library routine
    assert (row_token[:T * K] == order // K).all()
    assert (counts == np.bincount(flat, minlength=E)).all() and counts.sum() == T * K
    assert offsets[0] == 0 and offsets[E] == T * K and offsets[E + 1] == T * K + T
    assert (np.diff(offsets[:E + 1]) == counts).all()
    assert (row_token[row_of] == np.arange(T)[:, None]).all()
    assert sorted(row_of.reshape(-1)) == list(range(T * K))          # nothing dropped
    for e in range(E):
        seg = row_token[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()                             # token order
        assert (idx[seg] == e).any(axis=1).all()
    assert (row_token[T * K:] == np.arange(T)).all()
    c2, o2, rt2, ro2 = oracle.permute(idx, E, include_shared=False)
    assert o2[E + 1] == T * K and len(rt2) == T * K and (ro2 == row_of).all()


def _decode_torch(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()


def test_gemm_equals_float64_matmul_of_dequantised_operands():
    M, N, K = 70, 256, 512
    qa = workloads.gen_fp8_codes(M, K, sub_seed=11).numpy()
    qb = workloads.gen_fp8_codes(N, K, sub_seed=12).numpy()
    sa = workloads.gen_scales((K // 128, M), sub_seed=13).numpy()
    sb = workloads.gen_scales((N // 128, K // 128), sub_seed=14).numpy()
    C = oracle.blockscaled_gemm(qa, sa, qb, sb)
    A = _decode_torch(qa) * torch.from_numpy(sa).double().T.repeat_interleave(128, 1)
    B = _decode_torch(qb) * torch.from_numpy(sb).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
    ref = (A @ B.T).numpy()
    assert np.allclose(C, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_gemm_closed_forms():
    M, N, K = 3, 128, 384
    one = np.full((M, K), 0x38, np.uint8)                          # E4M3 1.0
    assert oracle.e4m3_decode(np.uint8(0x38)) == 1.0
    C = oracle.blockscaled_gemm(one, np.ones((3, M), np.float32),
                                np.full((N, K), 0x38, np.uint8), np.ones((1, 3), np.float32))
    assert (C == K).all()
    # only K-block 1 is non-zero: C = sa[1, m] * sb[0, 1] * 128
    qa = np.zeros((M, K), np.uint8)
    qa[:, 128:256] = 0x38
    sa = np.array([[5, 5, 5], [2, 3, 4], [7, 7, 7]], np.float32)
    sb = np.array([[9, 0.5, 9]], np.float32)
    C = oracle.blockscaled_gemm(qa, sa, np.full((N, K), 0x38, np.uint8), sb)
    assert (C == (np.array([2, 3, 4])[:, None] * 0.5 * 128)).all()


def test_gemm_partial_sums_are_exact():
    """Largest-magnitude operands: 128 products of 448*448 sum exactly in float64."""
    qa = np.full((1, 128), 0x7E, np.uint8)
    qb = np.full((128, 128), 0x7E, np.uint8)
    qb[1] = 0x01                                                    # smallest subnormal
    C = oracle.blockscaled_gemm(qa, np.ones((1, 1), np.float32), qb, np.ones((1, 1), np.float32))
    assert C[0, 0] == 128 * 448.0 * 448.0
    assert C[0, 1] == 128 * 448.0 * 2.0 ** -9


def _swiglu_inputs(m=20, d=256, f=256, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, d)).astype(np.float32)
    w1, w3 = (rng.standard_normal((f, d)) * 0.05).astype(np.float32), (rng.standard_normal((f, d)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((d, f)) * 0.05).astype(np.float32)
    return x, w1, w3, w2


def test_swiglu_structure_against_torch_float64():
    x, w1, w3, w2 = _swiglu_inputs()
    xq, sx = oracle.quant_1x128(x)
    W = [oracle.quant_128x128(w) for w in (w1, w3, w2)]
    hq, sh, Y = oracle.swiglu_expert(xq, sx, *W[0], *W[1], *W[2])
    xt = _decode_torch(xq) * torch.from_numpy(sx).double().T.repeat_interleave(128, 1)
    wt = [_decode_torch(q) * torch.from_numpy(s).double().repeat_interleave(128, 0).repeat_interleave(128, 1)
          for q, s in W]
    h = F.silu(xt @ wt[0].T) * (xt @ wt[1].T)
    ref = (h @ wt[2].T).numpy()
    rms = np.sqrt((ref ** 2).mean())
    err = np.abs(Y - ref)
    assert err.mean() / rms < 0.02 and err.max() / rms < 0.2       # only h's FP8 + BF16 rounding
    swapped = oracle.swiglu_expert(xq, sx, *W[1], *W[0], *W[2])[2]  # gate/up exchanged
    assert np.abs(swapped - ref).mean() / rms > 0.2


def test_swiglu_zero_gate_or_up_gives_zero():
    x, w1, w3, w2 = _swiglu_inputs(seed=1)
    xq, sx = oracle.quant_1x128(x)
    z = oracle.quant_128x128(np.zeros_like(w1))
    W1, W3, W2 = (oracle.quant_128x128(w) for w in (w1, w3, w2))
    for a, b in ((z, W3), (W1, z)):
        hq, sh, Y = oracle.swiglu_expert(xq, sx, *a, *b, *W2)
        assert (oracle.e4m3_decode(hq) == 0).all() and (Y == 0).all() and (sh == 1).all()


def test_combine_closed_form():
    T, K, d = 6, 3, 16
    Y = np.ones((T * K + T, d), np.float32)
    Y[T * K:] = 0
    gate = np.full((T, K), np.float32(1) / np.float32(3))
    row_of = np.arange(T * K, dtype=np.int32).reshape(T, K)
    y = oracle.combine(Y, row_of, gate, shared_row_base=T * K)
    assert (y == 1.0).all()
    Y[T * K:] = 2.0
    y = oracle.combine(Y, row_of, gate, shared_row_base=T * K)
    assert (y == 3.0).all()
    assert (oracle.combine(Y, row_of, gate, shared_row_base=-1) == 1.0).all()
