"""Workload shapes and seeded synthetic inputs for the MoE FFN forward.

This module only draws random numbers and shapes them; it holds none of the method's
arithmetic (no quantisation, routing or GEMM).  Both the CUDA path (tests, bench) and
the CPU oracle consume what it produces, and it is the only code they share.

Recipe (all inputs synthetic, seeded, base seed 0; sub-seeds per tensor):
  x         N(0, 1) float32 -> a seeded set of outlier channels is multiplied by the
            outlier factor -> cast to BF16 (RNE).                       sub-seed 0 / 5
  centroids N(0, 0.02) float32 [E, d]                                    sub-seed 1
  bias      U(-0.01, 0.01) float32 [E]; the skewed workload adds a Zipf-shaped
            preference  -beta * s * ln(rank_i)  with ranks from a seeded permutation
                                                                         sub-seed 2 / 6
  experts   N(0, w_std) float32, one generator per (expert, matrix), so any single
            expert can be regenerated on its own                         sub-seed 3
  FP8 GEMM operands  random finite E4M3 codes and positive float32 scales 2**U(-8, 2),
            or N(0, 1) float32 matrices for the quantise-then-multiply path   sub-seed 7
"""

from dataclasses import dataclass, replace
import math

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int              # tokens
    d: int              # model width
    E: int              # routed experts
    n_groups: int       # expert groups (nodes)
    topk_groups: int    # M, groups a token may use
    K: int              # experts per token
    f: int              # expert hidden width (routed and shared)
    n_outlier: int      # outlier channels in x
    outlier_scale: float
    w_std: float        # expert weight std before quantisation
    router_std: float = 0.02
    bias_range: float = 0.01
    zipf_s: float = 0.0     # > 0: skewed-popularity bias
    zipf_beta: float = 0.0

    @property
    def group_topn(self):
        return self.K // self.topk_groups

    @property
    def rows(self):
        """Rows of the permuted activation buffer: routed pairs plus one shared row per token."""
        return self.T * self.K + self.T

    def flops(self):
        """Algorithmic FP8 GEMM FLOPs of one forward: T * (K + 1) * 3 matrices * 2 * d * f."""
        return self.T * (self.K + 1) * 6 * self.d * self.f


TINY = MoEConfig("tiny", T=256, d=512, E=16, n_groups=4, topk_groups=2, K=4, f=256,
                 n_outlier=4, outlier_scale=20.0, w_std=0.02)
V3 = MoEConfig("v3", T=4096, d=7168, E=256, n_groups=8, topk_groups=4, K=8, f=2048,
               n_outlier=72, outlier_scale=30.0, w_std=0.006)
# beta: bisected on the oracle router over this workload's own x, centroids and bias so
# that the busiest expert takes 10x the mean load (the workload's "up to ~10x mean load on
# hot experts"); tests/test_workloads.py checks the ratio
SKEWED = replace(V3, name="skewed", T=16384, zipf_s=1.1, zipf_beta=0.0176)
DECODE = replace(V3, name="decode", T=128)
# V3 shapes with 32 experts and 512 tokens (about 128 rows per expert, like V3): a small
# case for profiler captures (1.4 GB of expert weights).
V3_E32 = replace(V3, name="v3_e32", T=512, E=32)
# its decode-shaped counterpart (16 tokens: segments of 0-8 rows) for GEMM captures
DECODE_E32 = replace(V3, name="decode_e32", T=16, E=32)
CONFIGS = {c.name: c for c in (TINY, V3, SKEWED, DECODE, V3_E32, DECODE_E32)}

# Standalone FP8 block-scaled GEMM sweep, (M, N, K).
GEMM_SWEEP = [(4096, 7168, 2048), (4096, 4096, 7168), (8192, 18432, 7168),
              (8192, 7168, 18432), (16384, 24576, 1536)]

SEED_X, SEED_ROUTER, SEED_BIAS, SEED_EXPERT, SEED_OUTLIER, SEED_ZIPF, SEED_GEMM = range(7)


def _gen(sub_seed, base_seed=0, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(base_seed * 1_000_003 + sub_seed)
    return g


def gen_x(cfg, base_seed=0, T=None):
    """BF16 [T, d] activations with outlier channels (CPU tensor)."""
    T = cfg.T if T is None else T
    x = torch.randn(T, cfg.d, generator=_gen(SEED_X, base_seed))
    chans = torch.randperm(cfg.d, generator=_gen(SEED_OUTLIER, base_seed))[:cfg.n_outlier]
    x[:, chans] *= cfg.outlier_scale
    return x.to(torch.bfloat16)


def gen_centroids(cfg, base_seed=0):
    """float32 [E, d] router centroids (CPU tensor)."""
    return torch.randn(cfg.E, cfg.d, generator=_gen(SEED_ROUTER, base_seed)) * cfg.router_std


def gen_bias(cfg, base_seed=0):
    """float32 [E] selection bias (CPU tensor)."""
    b = (torch.rand(cfg.E, generator=_gen(SEED_BIAS, base_seed)) * 2 - 1) * cfg.bias_range
    if cfg.zipf_s > 0:
        rank = torch.randperm(cfg.E, generator=_gen(SEED_ZIPF, base_seed)).double() + 1.0
        b = b + (-cfg.zipf_beta * cfg.zipf_s * torch.log(rank)).float()
    return b.float()


def gen_expert_f32(cfg, e, device="cpu", base_seed=0):
    """float32 (w1 [f, d], w3 [f, d], w2 [d, f]) of expert e (e == E: the shared expert).

    One generator per (expert, matrix): the same call on the same device type always
    returns the same values, whatever else was generated before.
    """
    out = []
    for j, shape in enumerate(((cfg.f, cfg.d), (cfg.f, cfg.d), (cfg.d, cfg.f))):
        g = _gen(SEED_EXPERT * 100_000_000 + e * 3 + j, base_seed, device)
        out.append(torch.randn(*shape, generator=g, device=device) * cfg.w_std)
    return tuple(out)


# Finite E4M3 codes: every byte except the two NaN encodings 0x7F and 0xFF.
_FINITE_CODES = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)


def gen_fp8_codes(rows, cols, sub_seed=SEED_GEMM, base_seed=0):
    """uint8 [rows, cols] random finite E4M3 codes (CPU tensor)."""
    g = _gen(sub_seed, base_seed)
    pick = torch.randint(0, _FINITE_CODES.numel(), (rows, cols), generator=g)
    return _FINITE_CODES[pick]


def gen_scales(shape, sub_seed=SEED_GEMM + 100, base_seed=0):
    """float32 positive scales 2**U(-8, 2) (CPU tensor)."""
    g = _gen(sub_seed, base_seed)
    return torch.exp2(torch.rand(*shape, generator=g) * 10 - 8).float()


def gen_normal(rows, cols, sub_seed, base_seed=0, device="cpu"):
    """float32 N(0, 1) [rows, cols]."""
    return torch.randn(rows, cols, generator=_gen(sub_seed, base_seed, device), device=device)


def zipf_load_note(cfg):
    """Human-readable description of the skewed-bias recipe (for bench/config output)."""
    if cfg.zipf_s <= 0:
        return "uniform bias U(-0.01, 0.01)"
    return (f"bias U(-0.01,0.01) - {cfg.zipf_beta} * {cfg.zipf_s} * ln(rank), "
            f"ranks a seeded permutation of 1..{cfg.E}")


def ceil_div(a, b):
    return -(-a // b)


def log2_ceil(n):
    return 0 if n <= 1 else math.ceil(math.log2(n))
