"""GPU parity of the memory-bound kernels against the CPU oracle, through the C-ABI:
1x128 / 128x128 quantisation and the router (bit-exact given identical inputs),
permutation (bit-exact, deterministic), combine and bias update."""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from fp8_block_scaled_bias_b300 import ops
from tolerance import assert_close, bf16_to_f32, routing_margin

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def _wide_range_bf16(rows, cols, seed):
    """BF16 values whose 1x128 tiles span many binades, with zero tiles, subnormal-scale
    tiles and repeated maxima."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g)
    tile_scale = torch.exp2(torch.randint(-40, 40, (rows, cols // 128), generator=g).float())
    x = x * tile_scale.repeat_interleave(128, dim=1)
    if rows > 2 and cols >= 256:
        x[1, 128:256] = 0.0
        x[2, :128] = 3.0                      # every element is the max
        x[0, :128] *= 1e-30                   # deep subnormal E4M3 after scaling
    return x.to(torch.bfloat16)


# ---- quantisation --------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(1, 128), (3, 384), (257, 512), (256, 512), (33, 7168)])
def test_quant_1x128_bit_exact(rows, cols):
    x = _wide_range_bf16(rows, cols, seed=rows * 7 + cols)
    q, s = ops.quant_1x128(x.to(DEV))
    q_ref, s_ref = oracle.quant_1x128(x.float().numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quant_1x128_v3_activations_bit_exact():
    x = workloads.gen_x(workloads.V3)                  # [4096, 7168] with 72 outlier channels
    q, s = ops.quant_1x128(x.to(DEV))
    q_ref, s_ref = oracle.quant_1x128(x.float().numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quant_1x128_strided_input():
    x = _wide_range_bf16(9, 640, seed=3).to(DEV)
    view = x[:, 128:512]                               # ldx = 640, cols = 384
    q = torch.empty(9, 384, dtype=torch.uint8, device=DEV)
    s = torch.empty(3, 9, dtype=torch.float32, device=DEV)
    from fp8_block_scaled_bias_b300._lib import call
    call("fp8_quant_1x128", view.data_ptr(), 9, 384, 640, q.data_ptr(), s.data_ptr(),
         torch.cuda.current_stream().cuda_stream)
    q_ref, s_ref = oracle.quant_1x128(view.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(s.cpu().numpy(), s_ref)


@pytest.mark.parametrize("T,K,cols,shared", [(5, 3, 384, True), (300, 8, 512, True),
                                              (257, 1, 128, False), (1, 4, 7168, True)])
def test_quant_scatter_bit_exact(T, K, cols, shared):
    """Every row a token is dispatched to holds the oracle's 1x128 quantisation of that
    token; rows nobody is dispatched to are left untouched."""
    x = _wide_range_bf16(T, cols, seed=T + K)
    rng = np.random.default_rng(T)
    n_rows = T * K + (T if shared else 0) + 3                   # 3 rows nobody writes
    row_of = rng.permutation(T * K).astype(np.int32).reshape(T, K)
    q = torch.full((n_rows, cols), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((cols // 128, n_rows), -1.0, dtype=torch.float32, device=DEV)
    status = ops.new_status(DEV)
    ops.quant_scatter_1x128(x.to(DEV), torch.from_numpy(row_of).to(DEV), n_rows,
                            T * K if shared else None, status, out=(q, sc))
    assert ops.status_value(status) == 0
    q_ref, s_ref = oracle.quant_1x128(x.float().numpy())
    qg, sg = q.cpu().numpy(), sc.cpu().numpy()
    for t in range(T):
        for r in list(row_of[t]) + ([T * K + t] if shared else []):
            assert np.array_equal(qg[r], q_ref[t]) and np.array_equal(sg[:, r], s_ref[:, t])
    used = T * K + (T if shared else 0)
    assert (qg[used:] == 0xAB).all() and (sg[:, used:] == -1.0).all()


def test_quant_scatter_v3_matches_quant_then_gather():
    cfg = workloads.V3
    x = workloads.gen_x(cfg).to(DEV)
    g = torch.Generator().manual_seed(4)
    idx = torch.stack([torch.randperm(cfg.E, generator=g)[:cfg.K] for _ in range(cfg.T)])
    counts, offsets, row_token, row_of = ops.permute(idx.int().to(DEV), cfg.E, True)
    q, s = ops.quant_1x128(x)
    want = ops.gather_rows(q, s, row_token)
    got = ops.quant_scatter_1x128(x, row_of, cfg.rows, cfg.T * cfg.K)
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])


def test_quant_scatter_bad_row_sets_status():
    x = _wide_range_bf16(2, 256, seed=1).to(DEV)
    row_of = torch.tensor([[0, 9], [3, -1]], dtype=torch.int32, device=DEV)
    q = torch.zeros(4, 256, dtype=torch.uint8, device=DEV)
    sc = torch.zeros(2, 4, dtype=torch.float32, device=DEV)
    status = ops.new_status(DEV)
    ops.quant_scatter_1x128(x, row_of, 4, None, status, out=(q, sc))
    assert ops.status_value(status) == -6
    q_ref, s_ref = oracle.quant_1x128(x.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy()[[0, 3]], q_ref)
    assert (q.cpu().numpy()[[1, 2]] == 0).all() and (sc.cpu().numpy()[:, [1, 2]] == 0).all()


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 512), (2048, 7168)])
def test_quant_128x128_bit_exact(rows, cols):
    g = torch.Generator().manual_seed(rows + cols)
    w = torch.randn(rows, cols, generator=g) * 0.006
    w[:128, :128] *= 1e4
    if cols > 128:
        w[:128, 128:256] = 0
    q, s = ops.quant_128x128(w.to(DEV))
    q_ref, s_ref = oracle.quant_128x128(w.numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


# ---- router --------------------------------------------------------------------------

def test_route_worked_example_from_page():
    g = GOLD["bias_selection"]
    s = torch.tensor([g["affinity"]], dtype=torch.float32, device=DEV)
    b = torch.tensor(g["bias"], dtype=torch.float32, device=DEV)
    idx, gate = ops.route(s, b, 1, 1, g["k"], group_topn=g["k"], affinities=True)
    assert sorted((idx[0].cpu().numpy() + 1).tolist()) == g["chosen_one_based"]
    assert list(np.round(gate[0].cpu().numpy(), g["gate_decimals"])) == g["gates_approx"]
    i_ref, g_ref = oracle.route(s.cpu().numpy(), b.cpu().numpy(), 1, 1, g["k"], g["k"],
                                scores_are_affinities=True)
    assert np.array_equal(idx.cpu().numpy(), i_ref) and np.array_equal(gate.cpu().numpy(), g_ref)


def _affinities_with_ties(T, E, seed):
    rng = np.random.default_rng(seed)
    s = rng.uniform(0, 1, (T, E)).astype(np.float32)
    s[rng.random((T, E)) < 0.01] = 1.0                 # saturated sigmoid: exact ties
    s[:, 5] = s[:, 3]                                  # duplicated columns
    s = np.round(s * 64) / 64 if seed % 2 else s       # coarse grid: many ties
    return s.astype(np.float32)


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.V3], ids=["tiny", "v3"])
@pytest.mark.parametrize("T", [1, 37, 4096])
def test_route_affinities_bit_exact(cfg, T):
    for seed in (0, 1):
        s = _affinities_with_ties(T, cfg.E, seed + T)
        b = workloads.gen_bias(cfg).numpy()
        idx, gate = ops.route(torch.from_numpy(s).to(DEV), torch.from_numpy(b).to(DEV),
                              cfg.n_groups, cfg.topk_groups, cfg.K, affinities=True)
        i_ref, g_ref = oracle.route(s, b, cfg.n_groups, cfg.topk_groups, cfg.group_topn, cfg.K,
                                    scores_are_affinities=True)
        assert np.array_equal(idx.cpu().numpy(), i_ref)
        assert np.array_equal(gate.cpu().numpy(), g_ref)


def test_route_other_shapes_and_route_scale():
    for (E, G, M, K, n) in [(64, 8, 3, 6, 2), (32, 1, 1, 5, 5), (1024, 32, 4, 32, 8), (48, 4, 4, 4, 3),
                           (512, 16, 4, 8, 2), (288, 9, 3, 8, 2)]:
        rng = np.random.default_rng(E + K)
        s = rng.uniform(0, 1, (300, E)).astype(np.float32)
        b = rng.uniform(-0.05, 0.05, E).astype(np.float32)
        for rs in (1.0, 2.5):
            idx, gate = ops.route(torch.from_numpy(s).to(DEV), torch.from_numpy(b).to(DEV), G, M,
                                  K, group_topn=n, route_scale=rs, affinities=True)
            i_ref, g_ref = oracle.route(s, b, G, M, n, K, route_scale=rs,
                                        scores_are_affinities=True)
            assert np.array_equal(idx.cpu().numpy(), i_ref), (E, G, M, K)
            assert np.array_equal(gate.cpu().numpy(), g_ref), (E, G, M, K)


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.V3], ids=["tiny", "v3"])
@pytest.mark.parametrize("group_topn", ["all", 1])
def test_route_group_score_variants(cfg, group_topn):
    """Group scored by the sum over all its members (group_topn = E / n_groups) or by its
    best member alone, bit-exact against the oracle."""
    n = cfg.E // cfg.n_groups if group_topn == "all" else group_topn
    s = _affinities_with_ties(1024, cfg.E, 11)
    b = workloads.gen_bias(cfg).numpy()
    idx, gate = ops.route(torch.from_numpy(s).to(DEV), torch.from_numpy(b).to(DEV),
                          cfg.n_groups, cfg.topk_groups, cfg.K, group_topn=n, affinities=True)
    i_ref, g_ref = oracle.route(s, b, cfg.n_groups, cfg.topk_groups, n, cfg.K,
                                scores_are_affinities=True)
    assert np.array_equal(idx.cpu().numpy(), i_ref)
    assert np.array_equal(gate.cpu().numpy(), g_ref)


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.V3], ids=["tiny", "v3"])
def test_route_from_logits(cfg):
    """From logits the GPU sigmoid uses expf: decisions match the oracle except where the
    oracle's own margin is within a few float32 ulps; gates stay within 4 ulps."""
    T = 2048
    g = torch.Generator().manual_seed(11)
    z = (torch.randn(T, cfg.E, generator=g) * 5.4).float()    # V3-like logit spread
    z[::97, :3] = 40.0                                         # saturated affinities
    b = workloads.gen_bias(cfg)
    idx, gate = ops.route(z.to(DEV), b.to(DEV), cfg.n_groups, cfg.topk_groups, cfg.K)
    i_ref, g_ref = oracle.route(z.numpy(), b.numpy(), cfg.n_groups, cfg.topk_groups,
                                cfg.group_topn, cfg.K)
    idx, gate = idx.cpu().numpy(), gate.cpu().numpy()
    s = oracle.sigmoid_f32(z.numpy())
    c = (s + b.numpy()[None]).astype(np.float32)
    bad = np.nonzero((idx != i_ref).any(1))[0]
    for t in bad:
        assert routing_margin(c[t], i_ref[t], cfg.n_groups, cfg.topk_groups, cfg.group_topn) < 1e-6
    assert len(bad) <= max(2, T // 500)
    ok = np.setdiff1d(np.arange(T), bad)
    assert (np.abs(gate[ok] - g_ref[ok]) <= 16 * 2.0 ** -24 * g_ref[ok] + 1e-12).all()


def test_bias_update_bit_exact():
    rng = np.random.default_rng(0)
    for (T, K, E) in [(10, 4, 8), (4096, 8, 256), (16384, 8, 256), (3, 3, 9)]:
        counts = rng.multinomial(T * K, np.ones(E) / E).astype(np.int32)
        counts[0] = (T * K) // E if (T * K) % E == 0 else counts[0]
        b = rng.uniform(-1, 1, E).astype(np.float32)
        b[-1] = 1e8
        bt = torch.from_numpy(b).to(DEV)
        ops.bias_update(bt, torch.from_numpy(counts).to(DEV), T, K, 0.001)
        assert np.array_equal(bt.cpu().numpy(), oracle.bias_update(b, counts, T, K, 0.001))


# ---- permutation ---------------------------------------------------------------------

def _random_idx(T, K, E, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    p = np.ones(E) if skew == 0 else 1.0 / np.arange(1, E + 1) ** skew
    p = p / p.sum()
    return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,K,E,skew", [(1, 4, 16, 0), (127, 4, 16, 0), (128, 8, 256, 0),
                                        (129, 8, 256, 1.1), (4096, 8, 256, 0),
                                        (1000, 32, 1024, 1.1), (300, 3, 5, 0)])
@pytest.mark.parametrize("shared", [True, False])
def test_permute_bit_exact(T, K, E, skew, shared):
    idx = _random_idx(T, K, E, seed=T + K, skew=skew)
    st = ops.new_status(DEV)
    out = ops.permute(torch.from_numpy(idx).to(DEV), E, shared, st)
    ref = oracle.permute(idx, E, include_shared=shared)
    for got, want, name in zip(out, ref, ("counts", "offsets", "row_token", "row_of")):
        assert np.array_equal(got.cpu().numpy(), want), name
    assert ops.status_value(st) == 0


def test_permute_deterministic_and_hot_expert():
    T, K, E = 4096, 8, 256
    idx = np.tile(np.arange(K, dtype=np.int32), (T, 1))   # every token -> experts 0..7
    idx[::3] = np.arange(K, 2 * K)
    it = torch.from_numpy(idx).to(DEV)
    first = [t.cpu().numpy() for t in ops.permute(it, E)]
    for _ in range(5):
        again = [t.cpu().numpy() for t in ops.permute(it, E)]
        assert all(np.array_equal(a, b) for a, b in zip(first, again))
    ref = oracle.permute(idx, E)
    assert all(np.array_equal(a, b) for a, b in zip(first, ref))


def test_permute_reports_bad_index():
    idx = torch.tensor([[0, 1], [2, 16]], dtype=torch.int32, device=DEV)
    st = ops.new_status(DEV)
    ops.permute(idx, 16, True, st)
    assert ops.status_value(st) == -6


# ---- combine -------------------------------------------------------------------------

@pytest.mark.parametrize("T,K,d,shared", [(1, 4, 512, True), (255, 4, 512, True),
                                          (64, 8, 7168, True), (33, 8, 136, False)])
def test_combine_matches_oracle(T, K, d, shared):
    rng = np.random.default_rng(T + d)
    rows = T * K + (T if shared else 0)
    Y = torch.from_numpy(rng.standard_normal((rows, d)).astype(np.float32)).to(torch.bfloat16)
    row_of = np.stack([rng.permutation(T * K)[:K] for _ in range(T)]).astype(np.int32)
    gate = rng.uniform(0, 1, (T, K)).astype(np.float32)
    gate /= gate.sum(1, keepdims=True)
    y = ops.combine(Y.to(DEV), torch.from_numpy(row_of).to(DEV), torch.from_numpy(gate).to(DEV),
                    T * K if shared else -1)
    ref = oracle.combine(Y.float().numpy(), row_of, gate, T * K if shared else -1)
    y = bf16_to_f32(y)
    assert_close(y, ref, what="combine")
    # FP32 accumulation vs float64: the BF16 results differ by at most one BF16 ulp
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    assert (np.abs(y - ref) <= ulp).all()


def test_combine_v3_shape_sampled_tokens():
    """The V3 launch (T=4096, K=8, d=7168, 36,864 BF16 expert rows, shared rows last):
    64 seeded tokens checked against the oracle, the others by the same FP32 rule's
    invariants (finite, one BF16 ulp of the float64 sum on the sampled ones)."""
    cfg = workloads.V3
    T, K, d = cfg.T, cfg.K, cfg.d
    rng = np.random.default_rng(77)
    rows = T * K + T
    Y = torch.randn(rows, d, generator=torch.Generator().manual_seed(77)).to(torch.bfloat16)
    row_of = rng.permutation(T * K).reshape(T, K).astype(np.int32)
    gate = rng.uniform(0, 1, (T, K)).astype(np.float32)
    gate /= gate.sum(1, keepdims=True)
    st = ops.new_status(DEV)
    y = ops.combine(Y.to(DEV), torch.from_numpy(row_of).to(DEV), torch.from_numpy(gate).to(DEV),
                    T * K, st)
    torch.cuda.synchronize()
    assert ops.status_value(st) == 0
    y = bf16_to_f32(y)
    assert np.isfinite(y).all()
    toks = np.sort(rng.choice(T, 64, replace=False))
    toks[-1] = T - 1
    Yn = Y.float().numpy()
    ref = oracle.combine(np.concatenate([Yn[row_of[toks].ravel()], Yn[T * K + toks]]),
                         np.arange(len(toks) * K, dtype=np.int32).reshape(len(toks), K),
                         gate[toks], len(toks) * K)
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    assert (np.abs(y[toks] - ref) <= ulp).all()


def test_combine_page_toy_mixture():
    g = GOLD["toy_mixture"]
    Y = torch.zeros(2, 8, dtype=torch.bfloat16)
    Y[0], Y[1] = g["expert_outputs"][0], g["expert_outputs"][1]
    s = torch.tensor([g["affinity"]], dtype=torch.float32, device=DEV)
    idx, gate = ops.route(s, torch.zeros(4, device=DEV), 1, 1, 2, group_topn=2, affinities=True)
    row_of = torch.tensor([[0, 1]], dtype=torch.int32, device=DEV)
    y = ops.combine(Y.to(DEV), row_of, gate, -1)
    assert abs(float(y[0, 0]) - g["routed_contribution_approx"]) < 0.02


def test_combine_reports_bad_row():
    Y = torch.zeros(4, 8, dtype=torch.bfloat16, device=DEV)
    row_of = torch.tensor([[0, 9]], dtype=torch.int32, device=DEV)
    gate = torch.ones(1, 2, device=DEV)
    st = ops.new_status(DEV)
    ops.combine(Y, row_of, gate, -1, st)
    assert ops.status_value(st) == -6


# ---- router logits -------------------------------------------------------------------

@pytest.mark.parametrize("T,d,E", [(1, 128, 16), (130, 512, 16), (256, 512, 48), (300, 384, 80),
                                   (128, 7168, 256), (4096, 7168, 256)])
def test_router_logits_against_oracle(T, d, E):
    """z on BF16 tensor cores from the hi/lo split: within 2^-14 of sum_k |x_k e_k| of the
    exact product (dropping the lo plane would miss by about 2^-9 of it).  The small-T
    shapes run with the K loop split across CTAs (partials summed in split order), and
    the split result must repeat bit for bit."""
    g = torch.Generator().manual_seed(T + d + E)
    x = torch.randn(T, d, generator=g)
    x[:, :4] *= 30.0                                   # outlier channels
    x = x.to(torch.bfloat16)
    cen = (torch.randn(E, d, generator=g) * 0.02).float()
    hilo = ops.router_split_bf16(cen.to(DEV))
    st = ops.new_status(DEV)
    z = ops.router_logits(x.to(DEV), hilo, st).cpu().numpy()
    assert ops.status_value(st) == 0
    xf = x.float().numpy().astype(np.float64)
    z_ref = xf @ cen.numpy().astype(np.float64).T
    bound = 2.0 ** -14 * (np.abs(xf) @ np.abs(cen.numpy().astype(np.float64)).T) + 1e-30
    assert (np.abs(z - z_ref) <= bound).all()
    assert np.array_equal(oracle.router_logits(x.float().numpy(), cen.numpy()),
                          z_ref.astype(np.float32))
    z2 = ops.router_logits(x.to(DEV), hilo, st).cpu().numpy()
    assert np.array_equal(z, z2)


def test_router_split_planes():
    w = torch.tensor([[1.0, 1.0 + 2 ** -10, -3.14159265, 1e-30, 0.0, 65504.0, -2.0 ** -130, 7.0]],
                     dtype=torch.float32).repeat(1, 16)
    hl = ops.router_split_bf16(w.to(DEV)).cpu()
    hi, lo = hl[0].float(), hl[1].float()
    assert torch.equal(hi, w.to(torch.bfloat16).float())
    assert torch.equal(lo, (w - hi).to(torch.bfloat16).float())
    assert ((hi + lo - w).abs() <= 2.0 ** -16 * w.abs() + 1e-38).all()
