"""GPU parity of the tcgen05 block-scaled grouped GEMM (through the C-ABI) against the
oracle's exact definition: dense and grouped, ragged and empty segments, a half-width
last N tile, gathered A rows, and the five full-size sweep shapes on sampled rows.  The
small cases run under every tiling (one CTA per 128-row tile; CTA pairs sharing one
cta_group::2 MMA per 256-row tile; swapped operands with weight rows on the MMA's M side,
which falls back to the first when N % 256 != 0).  The failure path of the bounded waits is exercised
by a launch whose MMA-issuing thread waits on a barrier nothing arrives on."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from fp8_block_scaled_bias_b300 import ops
from tolerance import assert_close, bf16_to_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(params=[1, 2, 3], ids=["single", "pair", "swap"])
def tiling(request, lib):
    L = lib.load()
    assert L.moe_set_gemm_tiling(request.param) == 0
    yield request.param
    L.moe_set_gemm_tiling(0)


def _codes(rows, cols, seed):
    return workloads.gen_fp8_codes(rows, cols, sub_seed=seed)


def _run(A, sA, B, sB, seg, M, a_rows=None):
    st = ops.new_status(DEV)
    C = ops.grouped_gemm(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV),
                         torch.tensor(seg, dtype=torch.int32, device=DEV), M,
                         a_rows=None if a_rows is None else torch.tensor(a_rows, dtype=torch.int32,
                                                                         device=DEV),
                         status=st)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    return bf16_to_f32(C)


def _ref(A, sA, B, sB, seg, a_rows=None):
    """The oracle's GEMM per segment, rounded to BF16 like the kernel's output."""
    A, sA, B, sB = (t.numpy() for t in (A, sA, B, sB))
    M = seg[-1]
    out = np.zeros((M, B.shape[1]), np.float64)
    for g in range(len(seg) - 1):
        r0, r1 = seg[g], seg[g + 1]
        if r1 == r0:
            continue
        rows = np.arange(r0, r1) if a_rows is None else np.asarray(a_rows[r0:r1])
        out[r0:r1] = oracle.blockscaled_gemm(A[rows], sA[:, rows], B[g], sB[g])
    return oracle.bf16_round(out)


def _check(C, ref, what):
    """R12 tolerance, and BF16 results equal or one BF16 ulp apart (FP32 accumulation
    against the exact sum changes at most the last rounding)."""
    assert_close(C, ref, what=what)
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
    assert (np.abs(C - ref) <= np.maximum(ulp, 1e-3 * rms)).all(), what
    assert (C == ref).mean() > 0.9, what


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (128, 256, 128), (200, 256, 512),
                                   (300, 512, 1024), (129, 384, 256), (513, 384, 640)])
def test_dense_gemm(M, N, K, tiling):
    A, B = _codes(M, K, 1), _codes(N, K, 2)
    sA = workloads.gen_scales((K // 128, M), sub_seed=3)
    sB = workloads.gen_scales((1, N // 128, K // 128), sub_seed=4)
    C = _run(A, sA, B[None], sB, [0, M], M)
    _check(C, _ref(A, sA, B[None], sB, [0, M]), f"dense {M}x{N}x{K}")


def test_grouped_ragged_segments(tiling):
    counts = [0, 130, 1, 256, 77, 0, 128]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    M, N, K, G = seg[-1], 384, 256, len(counts)
    A = _codes(M, K, 5)
    sA = workloads.gen_scales((K // 128, M), sub_seed=6)
    B = _codes(G * N, K, 7).view(G, N, K)
    sB = workloads.gen_scales((G, N // 128, K // 128), sub_seed=8)
    C = _run(A, sA, B, sB, seg, M)
    _check(C, _ref(A, sA, B, sB, seg), "grouped")


def test_grouped_rows_past_last_segment_untouched(tiling):
    seg = [0, 100, 100, 150]
    M, N, K = 300, 256, 128
    A = _codes(M, K, 9)
    sA = workloads.gen_scales((K // 128, M), sub_seed=10)
    B = _codes(3 * N, K, 11).view(3, N, K)
    sB = workloads.gen_scales((3, N // 128, K // 128), sub_seed=12)
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    ops.grouped_gemm(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV),
                     torch.tensor(seg, dtype=torch.int32, device=DEV), M, out=C)
    C = bf16_to_f32(C)
    assert (C[150:] == 7.0).all()
    _check(C[:150], _ref(A, sA, B, sB, seg), "prefix rows")


def test_grouped_with_gathered_rows(tiling):
    T, K, N = 90, 256, 256
    rng = np.random.default_rng(0)
    a_rows = np.concatenate([rng.permutation(T)[:50], rng.permutation(T)[:70], np.arange(T)])
    seg = [0, 50, 120, 120 + T]
    A = _codes(T, K, 13)
    sA = workloads.gen_scales((K // 128, T), sub_seed=14)
    B = _codes(3 * N, K, 15).view(3, N, K)
    sB = workloads.gen_scales((3, N // 128, K // 128), sub_seed=16)
    C = _run(A, sA, B, sB, seg, len(a_rows), a_rows=a_rows)
    _check(C, _ref(A, sA, B, sB, seg, a_rows), "gathered")


def test_grouped_strided_output(tiling):
    """C as a column window of a wider buffer: a row pitch and base that are 16- but not
    32-byte aligned (the epilogue's 16-byte store path); the columns around it stay."""
    counts = [70, 0, 200, 33]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    M, N, K, G = seg[-1], 384, 384, len(counts)
    A = _codes(M, K, 41)
    sA = workloads.gen_scales((K // 128, M), sub_seed=42)
    B = _codes(G * N, K, 43).view(G, N, K)
    sB = workloads.gen_scales((G, N // 128, K // 128), sub_seed=44)
    buf = torch.full((M, N + 24), 7.0, dtype=torch.bfloat16, device=DEV)
    C = buf[:, 8:8 + N]
    assert (C.stride(0) * 2) % 32 == 16 and C.data_ptr() % 32 == 16
    st = ops.new_status(DEV)
    ops.grouped_gemm(A.to(DEV), sA.to(DEV), B.to(DEV), sB.to(DEV),
                     torch.tensor(seg, dtype=torch.int32, device=DEV), M, status=st, out=C)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    full = bf16_to_f32(buf)
    assert (full[:, :8] == 7.0).all() and (full[:, 8 + N:] == 7.0).all()
    _check(full[:, 8:8 + N], _ref(A, sA, B, sB, seg), "strided C")


def test_bad_segment_table_is_reported(tiling):
    A = torch.zeros(64, 128, dtype=torch.uint8, device=DEV)
    sA = torch.ones(1, 64, device=DEV)
    B = torch.zeros(2, 256, 128, dtype=torch.uint8, device=DEV)
    sB = torch.ones(2, 2, 1, device=DEV)
    st = ops.new_status(DEV)
    ops.grouped_gemm(A, sA, B, sB, torch.tensor([0, 40, 30], dtype=torch.int32, device=DEV), 64,
                     status=st)
    assert ops.status_value(st) == -6
    st = ops.new_status(DEV)
    ops.grouped_gemm(A, sA, B, sB, torch.tensor([0, 40, 65], dtype=torch.int32, device=DEV), 64,
                     status=st)
    assert ops.status_value(st) == -6


def test_closed_form_all_ones(tiling):
    M, N, K = 256, 256, 1024
    A = torch.full((M, K), 0x38, dtype=torch.uint8)          # E4M3 1.0
    B = torch.full((1, N, K), 0x38, dtype=torch.uint8)
    C = _run(A, torch.ones(K // 128, M), B, torch.ones(1, N // 128, K // 128), [0, M], M)
    assert (C == K).all()


@pytest.mark.parametrize("M,N,K", workloads.GEMM_SWEEP)
def test_sweep_shape_sampled_rows(M, N, K):
    """Full-size sweep shape, same launch as the bench; 128 seeded rows checked against
    the oracle over every column."""
    A = _codes(M, K, 21)
    B = _codes(N, K, 22)
    sA = workloads.gen_scales((K // 128, M), sub_seed=23)
    sB = workloads.gen_scales((1, N // 128, K // 128), sub_seed=24)
    C = _run(A, sA, B[None], sB, [0, M], M)
    rows = np.sort(np.random.default_rng(M + N + K).choice(M, 128, replace=False))
    rows[0], rows[-1] = 0, M - 1
    ref = oracle.bf16_round(oracle.blockscaled_gemm(A.numpy()[rows], sA.numpy()[:, rows],
                                                    B.numpy(), sB.numpy()[0]))
    _check(C[rows], ref, f"sweep {M}x{N}x{K}")


def test_sweep_recipe_normal_operands():
    """The sweep's own recipe: A, B ~ N(0,1), each side quantises them itself."""
    M, N, K = 4096, 7168, 2048
    a = workloads.gen_normal(M, K, sub_seed=31)
    b = workloads.gen_normal(N, K, sub_seed=32)
    qa, sa = ops.quant_1x128(a.to(torch.bfloat16).to(DEV))
    qb, sb = ops.quant_128x128(b.to(DEV))
    C = bf16_to_f32(ops.grouped_gemm(qa, sa, qb[None], sb[None],
                                     torch.tensor([0, M], dtype=torch.int32, device=DEV), M))
    rows = np.random.default_rng(1).choice(M, 64, replace=False)
    qa_r, sa_r = oracle.quant_1x128(a.to(torch.bfloat16).float().numpy()[rows])
    qb_r, sb_r = oracle.quant_128x128(b.numpy())
    ref = oracle.bf16_round(oracle.blockscaled_gemm(qa_r, sa_r, qb_r, sb_r))
    _check(C[rows], ref, "N(0,1) recipe")
    exact = a.to(torch.bfloat16).double().numpy()[rows] @ b.double().numpy().T
    # FP8 quantisation error against the unquantised product: a few percent of RMS
    assert np.abs(C[rows] - exact).mean() / np.sqrt((exact ** 2).mean()) < 0.05


def test_grouped_many_ragged_segments_both_tilings_equal(lib):
    """40 segments of 0..300 rows (empty ones, 1-row ones, ends on and off the 128- and
    256-row grids), N with a half-filled last tile: both tilings give the oracle's result
    and the same bits."""
    rng = np.random.default_rng(17)
    counts = rng.integers(0, 300, 40)
    counts[[3, 9, 20]] = 0
    counts[[5, 6]] = 1
    counts[[11, 12]] = [128, 256]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    M, N, K, G = seg[-1], 640, 384, len(counts)
    A = _codes(M, K, 41)
    sA = workloads.gen_scales((K // 128, M), sub_seed=42)
    B = _codes(G * N, K, 43).view(G, N, K)
    sB = workloads.gen_scales((G, N // 128, K // 128), sub_seed=44)
    L = lib.load()
    outs = []
    try:
        for mode in (1, 2, 3):
            L.moe_set_gemm_tiling(mode)
            outs.append(_run(A, sA, B, sB, seg, M))
    finally:
        L.moe_set_gemm_tiling(0)
    assert np.array_equal(outs[0], outs[1])
    ref = _ref(A, sA, B, sB, seg)
    _check(outs[1], ref, "40 ragged segments")
    # N = 640 is not a multiple of 256: the swapped tiling falls back to the single one
    assert np.array_equal(outs[2], outs[0])


def test_swapped_tiling_short_segments(lib):
    """Decode-like segments (0 to 40 rows, many of 1-8) on the swapped-operand tiling,
    N a multiple of 256, against the oracle."""
    rng = np.random.default_rng(19)
    counts = rng.integers(0, 9, 60)
    counts[[2, 7]] = 0
    counts[[10, 11, 12]] = [1, 32, 40]
    seg = np.concatenate([[0], np.cumsum(counts)]).tolist()
    M, N, K, G = seg[-1], 768, 512, len(counts)
    assert M <= 16 * G                         # the automatic choice picks it too
    A = _codes(M, K, 51)
    sA = workloads.gen_scales((K // 128, M), sub_seed=52)
    B = _codes(G * N, K, 53).view(G, N, K)
    sB = workloads.gen_scales((G, N // 128, K // 128), sub_seed=54)
    L = lib.load()
    try:
        L.moe_set_gemm_tiling(3)
        C3 = _run(A, sA, B, sB, seg, M)
        L.moe_set_gemm_tiling(1)
        C1 = _run(A, sA, B, sB, seg, M)
    finally:
        L.moe_set_gemm_tiling(0)
    _check(C3, _ref(A, sA, B, sB, seg), "swapped short segments")
    assert np.abs(C3 - C1).max() <= np.abs(C1).max() * 2.0 ** -7


@pytest.mark.parametrize("mode", [1, 2], ids=["single", "pair"])
def test_bounded_wait_expiry_reports_and_recovers(lib, mode):
    """Failure detection without a GPU fault: the MMA issuer waits on a barrier nothing
    arrives on, with every wait limited to 1 ms.  The kernel must report
    MOE_ERR_DEVICE_TIMEOUT, drain, free its TMEM and return within milliseconds, and the
    next (normal) launch on the same GPU must be correct."""
    import time
    from fp8_block_scaled_bias_b300._lib import call
    L = lib.load()
    M, N, K = 512, 512, 1024
    A = torch.full((M, K), 0x38, dtype=torch.uint8, device=DEV)     # E4M3 1.0
    B = torch.full((2, N, K), 0x38, dtype=torch.uint8, device=DEV)
    sA = torch.ones(K // 128, M, device=DEV)
    sB = torch.ones(2, N // 128, K // 128, device=DEV)
    seg = torch.tensor([0, 200, M], dtype=torch.int32, device=DEV)
    C = torch.zeros(M, N, dtype=torch.bfloat16, device=DEV)
    try:
        L.moe_set_gemm_tiling(mode)
        st = ops.new_status(DEV)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        call("moe_test_gemm_wait_expiry", A.data_ptr(), sA.data_ptr(), B.data_ptr(),
             sB.data_ptr(), seg.data_ptr(), 2, M, N, K, C.data_ptr(), N, st.data_ptr(),
             1_000_000, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert ops.status_value(st) == -4                 # MOE_ERR_DEVICE_TIMEOUT
        assert dt < 1.0, dt
        # the same GEMM without the stall: the context is healthy and the result exact
        st = ops.new_status(DEV)
        ops.grouped_gemm(A, sA, B, sB, seg, M, status=st, out=C)
        torch.cuda.synchronize()
        assert ops.status_value(st) == 0
        assert (bf16_to_f32(C) == K).all()
    finally:
        L.moe_set_gemm_tiling(0)
