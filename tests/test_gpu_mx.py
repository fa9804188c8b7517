"""GPU parity of the MX-native variant (power-of-two scales applied by the tensor core,
tcgen05.mma kind::mxf8f6f4) against the oracle: the power-of-two quantisers bit-exact,
the GEMM against the exact block-scaled definition.  Short segments (decode batches) take
the swapped-operand kernel, whose power-of-two promotion is exact; both paths are
covered."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from fp8_block_scaled_bias_b300 import ops
from tolerance import assert_close, bf16_to_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pow2_scales(shape, seed, lo=-8, hi=2):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.exp2(rng.integers(lo, hi + 1, shape)).astype(np.float32))


def _run(A, sA, B, sB, seg, M, expect_status=0):
    st = ops.new_status(DEV)
    C = ops.mx_grouped_gemm(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV),
                            torch.tensor(seg, dtype=torch.int32, device=DEV), M, status=st)
    torch.cuda.synchronize()
    assert ops.status_value(st) == expect_status
    return bf16_to_f32(C)


def _ref(A, sA, B, sB, seg):
    A, sA, B, sB = (t.numpy() for t in (A, sA, B, sB))
    out = np.zeros((seg[-1], B.shape[1]), np.float64)
    for g in range(len(seg) - 1):
        r0, r1 = seg[g], seg[g + 1]
        if r1 > r0:
            out[r0:r1] = oracle.blockscaled_gemm(A[r0:r1], sA[:, r0:r1], B[g], sB[g])
    return oracle.bf16_round(out)


def test_scale_factor_placement_closed_form():
    """All codes 1.0, K = 128: C[r][n] = 128 * sA[r] * sB[n / 128] exactly, with a different
    power of two for every row residue and every N block, so each row's and each
    column's scale must land where the tensor core reads it."""
    M, N, K = 256, 512, 128
    one = 0x38                                              # E4M3 1.0
    A = torch.full((M, K), one, dtype=torch.uint8)
    B = torch.full((1, N, K), one, dtype=torch.uint8)
    r = np.arange(M)
    sA = torch.from_numpy(np.exp2((r % 37) - 18).astype(np.float32))[None, :]
    sB = torch.from_numpy(np.exp2(np.arange(N // 128) - 2).astype(np.float32))[None, :, None]
    C = _run(A, sA, B, sB, [0, M], M)
    want = 128.0 * sA.numpy()[0][:, None] * np.repeat(sB.numpy()[0, :, 0], 128)[None, :]
    bad = np.argwhere(C != want)
    assert bad.size == 0, f"{len(bad)} wrong; first (row, col, got, want): " + str(
        [(int(i), int(j), float(C[i, j]), float(want[i, j])) for i, j in bad[:6]])


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (128, 256, 128), (200, 256, 512),
                                   (300, 512, 1024), (129, 384, 256), (512, 1024, 7168)])
def test_dense_mx_gemm(M, N, K):
    A = workloads.gen_fp8_codes(M, K, sub_seed=M + K)
    B = workloads.gen_fp8_codes(N, K, sub_seed=N + 7)[None]
    sA = _pow2_scales((K // 128, M), M)
    sB = _pow2_scales((1, N // 128, K // 128), N)
    C = _run(A, sA, B, sB, [0, M], M)
    assert_close(C, _ref(A, sA, B, sB, [0, M]), what=f"mx dense {M}x{N}x{K}")


def test_grouped_ragged_mx_gemm():
    seg = [0, 5, 5, 300, 301, 560]                          # an empty segment, ragged tails
    G, N, K = len(seg) - 1, 384, 512
    M = seg[-1]
    A = workloads.gen_fp8_codes(M, K, sub_seed=3)
    B = torch.stack([workloads.gen_fp8_codes(N, K, sub_seed=10 + g) for g in range(G)])
    sA = _pow2_scales((K // 128, M), 4)
    sB = _pow2_scales((G, N // 128, K // 128), 5)
    C = _run(A, sA, B, sB, seg, M)
    assert_close(C, _ref(A, sA, B, sB, seg), what="mx grouped")


@pytest.mark.parametrize("N", [384, 1152])
def test_grouped_ragged_mx_gemm_paired_tile(N):
    """M >= 256 * G selects the paired 256-row tile (two 128-row accumulators sharing each
    224-column B tile).  Empty segments, lengths off the 128- and 256-row grids, and N not
    a multiple of 224, so 224-column tiles straddle the 128-column weight-scale blocks
    and the last tile is partly filled."""
    counts = [0, 905, 1, 257, 0, 383, 511, 1]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    G, K = len(counts), 384
    M = seg[-1]
    assert M >= 256 * G
    A = workloads.gen_fp8_codes(M, K, sub_seed=61)
    B = torch.stack([workloads.gen_fp8_codes(N, K, sub_seed=70 + g) for g in range(G)])
    sA = _pow2_scales((K // 128, M), 62)
    sB = _pow2_scales((G, N // 128, K // 128), 63)
    C = _run(A, sA, B, sB, seg, M)
    assert_close(C, _ref(A, sA, B, sB, seg), what=f"mx grouped paired N={N}")


def test_mx_short_segments_on_swapped_operands():
    """Decode-like segments (M <= 16 G, N % 256 == 0) take the swapped-operand kernel with
    exact power-of-two promotion; against the oracle."""
    rng = np.random.default_rng(23)
    counts = rng.integers(0, 9, 40)
    counts[[1, 5]] = 0
    counts[[8, 9]] = [1, 37]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    G, N, K = len(counts), 512, 384
    M = seg[-1]
    assert M <= 16 * G
    A = workloads.gen_fp8_codes(M, K, sub_seed=81)
    B = torch.stack([workloads.gen_fp8_codes(N, K, sub_seed=90 + g) for g in range(G)])
    sA = _pow2_scales((K // 128, M), 82)
    sB = _pow2_scales((G, N // 128, K // 128), 83)
    C = _run(A, sA, B, sB, seg, M)
    assert_close(C, _ref(A, sA, B, sB, seg), what="mx short segments")


def test_pow2_quantisers_bit_exact():
    x = workloads.gen_x(workloads.V3)[:512]
    q, s = ops.quant_1x128(x.to(DEV), pow2=True)
    q_ref, s_ref = oracle.quant_1x128_pow2(x.float().numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref) and np.array_equal(q.cpu().numpy(), q_ref)
    g = torch.Generator().manual_seed(2)
    w = torch.randn(256, 512, generator=g) * 0.006
    w[:128, :128] *= 1e4
    w[128:, 128:256] = 0
    q, s = ops.quant_128x128(w.to(DEV), pow2=True)
    q_ref, s_ref = oracle.quant_128x128_pow2(w.numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref) and np.array_equal(q.cpu().numpy(), q_ref)


def test_mx_gemm_on_quantised_v3_activations_and_weights():
    """The variant end to end on a V3-shaped expert: x rows and N(0, 0.006) weights
    quantised with power-of-two scales, then the MX GEMM against the oracle."""
    cfg = workloads.V3
    x = workloads.gen_x(cfg)[:384].to(DEV)
    g = torch.Generator(device=DEV).manual_seed(9)
    w = torch.randn(512, cfg.d, generator=g, device=DEV) * cfg.w_std
    xq, sx = ops.quant_1x128(x, pow2=True)
    wq, sw = ops.quant_128x128(w, pow2=True)
    C = _run(xq.cpu(), sx.cpu(), wq.cpu()[None], sw.cpu()[None], [0, 384], 384)
    ref = _ref(xq.cpu(), sx.cpu(), wq.cpu()[None], sw.cpu()[None], [0, 384])
    assert_close(C, ref, what="mx V3 expert")


def test_non_power_of_two_scale_is_reported():
    M, N, K = 128, 256, 128
    A = workloads.gen_fp8_codes(M, K, sub_seed=1)
    B = workloads.gen_fp8_codes(N, K, sub_seed=2)[None]
    sA = _pow2_scales((1, M), 1)
    sA[0, 7] = 0.3
    sB = _pow2_scales((1, N // 128, 1), 2)
    _run(A, sA, B, sB, [0, M], M, expect_status=-6)


@pytest.mark.parametrize("case", ["normal", "v3_expert"])
def test_accuracy_against_the_fp32_scale_path(case):
    """A/B: both recipes against the exact product of the unquantised inputs.  Power-of-
    two scales put a group's max-abs in (224, 448] instead of at 448: the same 3-bit
    mantissa for normal values, so the error should stay close to the FP32-scale one."""
    g = torch.Generator(device=DEV).manual_seed(21)
    M, N, K = 256, 512, 2048
    if case == "normal":
        a = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
        b = torch.randn(N, K, generator=g, device=DEV)
    else:
        a = workloads.gen_x(workloads.V3)[:M, :K].to(DEV)
        b = torch.randn(N, K, generator=g, device=DEV) * workloads.V3.w_std
    exact = a.double() @ b.double().T
    seg = torch.tensor([0, M], dtype=torch.int32, device=DEV)
    errs = {}
    for pow2 in (False, True):
        qa, sa = ops.quant_1x128(a, pow2=pow2)
        qb, sb = ops.quant_128x128(b, pow2=pow2)
        gemm = ops.mx_grouped_gemm if pow2 else ops.grouped_gemm
        C = gemm(qa, sa, qb[None], sb[None], seg, M).double()
        rms = exact.pow(2).mean().sqrt()
        errs[pow2] = float((C - exact).abs().mean() / rms)
    assert errs[False] < 0.05 and errs[True] < 0.05, errs
    assert errs[True] <= 1.5 * errs[False], errs


@pytest.mark.parametrize("mx", [False, True], ids=["fp32_scales", "mx"])
def test_gate_up_with_distinct_gate_and_up_block_scales(mx):
    """Gate and up weight blocks with different scales (the 64-row interleave must pair
    every B row with its own block's scale) over ragged segments: h against the oracle's
    SwiGLU of the exact block-scaled products."""
    from fp8_block_scaled_bias_b300 import interleave_gate_up
    seg = [0, 100, 100, 300]
    S, d, f = len(seg) - 1, 512, 256
    M = seg[-1]
    rng = np.random.default_rng(17)
    A = workloads.gen_fp8_codes(M, d, sub_seed=41)
    sA = _pow2_scales((d // 128, M), 42, -3, 0)
    w1 = [workloads.gen_fp8_codes(f, d, sub_seed=50 + e) for e in range(S)]
    w3 = [workloads.gen_fp8_codes(f, d, sub_seed=60 + e) for e in range(S)]
    s1 = [torch.from_numpy(np.exp2(rng.integers(-12, -9, (f // 128, d // 128))).astype(np.float32))
          for _ in range(S)]
    s3 = [torch.from_numpy(np.exp2(rng.integers(-6, -3, (f // 128, d // 128))).astype(np.float32))
          for _ in range(S)]
    if not mx:                                   # any positive scales for the FP32 path
        s1 = [s * 1.37 for s in s1]
    pairs = [interleave_gate_up(w1[e], s1[e], w3[e], s3[e]) for e in range(S)]
    w13 = torch.stack([p[0] for p in pairs]).to(DEV)
    s13 = torch.stack([p[1] for p in pairs]).to(DEV)
    st = ops.new_status(DEV)
    hq, sh = ops.gate_up(A.to(DEV), sA.to(DEV), torch.tensor(seg, dtype=torch.int32, device=DEV),
                         w13, s13, st, mx=mx)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    got = oracle.dequant_1x128(hq.cpu().numpy(), sh.cpu().numpy())
    quant = oracle.quant_1x128_pow2 if mx else oracle.quant_1x128
    ref = np.zeros((M, f))
    for e in range(S):
        r0, r1 = seg[e], seg[e + 1]
        if r1 == r0:
            continue
        a, sa = A.numpy()[r0:r1], sA.numpy()[:, r0:r1]
        g = oracle.blockscaled_gemm(a, sa, w1[e].numpy(), s1[e].numpy()).astype(np.float32)
        u = oracle.blockscaled_gemm(a, sa, w3[e].numpy(), s3[e].numpy()).astype(np.float32)
        gd = g.astype(np.float64)
        h = (gd / (1 + np.exp(-gd)) * u).astype(np.float32)
        ref[r0:r1] = oracle.dequant_1x128(*quant(h))
    assert_close(got, ref, max_rel=0.07, mae=5e-3, what="h")
