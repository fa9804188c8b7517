"""GPU parity of the sequence-wise balance statistics (moe_seq_balance_stats) with the
oracle ("DeepSeek-V3" book, ch. 8, "The complementary sequence loss")."""

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_bias_b300 import ops
from fp8_block_scaled_bias_b300._lib import MoEError

pytestmark = pytest.mark.gpu
DEV = "cuda"

# f: both sides take the same integer counts and one correctly rounded FP32 division.
# P: FP32 sums over at most a few thousand terms against float64; loss likewise.
P_RTOL, P_ATOL, LOSS_RTOL = 1e-5, 1e-9, 1e-5


def _topk_margin(s, k):
    """Smallest gap between the k-th and (k+1)-th largest affinity over all tokens."""
    srt = -np.sort(-s.astype(np.float64), axis=1)
    return float((srt[:, k - 1] - srt[:, k]).min()) if s.shape[1] > k else np.inf


def _check(scores, K, L, aff, alpha=1e-4):
    f, P, loss = ops.seq_balance_stats(torch.from_numpy(scores).to(DEV), K, L, alpha=alpha,
                                       affinities=aff)
    f_ref, P_ref, l_ref = oracle.seq_balance_stats(scores, K, L, alpha=alpha,
                                                   scores_are_affinities=aff)
    assert np.array_equal(f.cpu().numpy(), f_ref)
    np.testing.assert_allclose(P.cpu().numpy(), P_ref, rtol=P_RTOL, atol=P_ATOL)
    np.testing.assert_allclose(loss.cpu().numpy(), l_ref, rtol=LOSS_RTOL)


@pytest.mark.parametrize("T,E,K,L", [(64, 16, 4, 64), (300, 48, 6, 100), (130, 256, 8, 65),
                                     (4096, 256, 8, 4096), (4096, 256, 8, 1024), (7, 1024, 32, 1),
                                     (96, 8, 8, 32)])
def test_affinities_match_oracle(T, E, K, L):
    rng = np.random.default_rng(T + E)
    s = rng.integers(1, 64, (T, E)).astype(np.float32) / 64       # many exact ties
    _check(s, K, L, True)


@pytest.mark.parametrize("T,E,K,L", [(256, 16, 4, 128), (4096, 256, 8, 4096), (2048, 64, 6, 512)])
def test_logits_match_oracle(T, E, K, L):
    rng = np.random.default_rng(E + K)
    # the GPU's expf sigmoid may differ from the oracle's by an ulp or two: every token's
    # logits are a random permutation of a grid 0.02 apart (plus a per-token offset), so
    # affinities are at least ~5e-4 apart and the top-K is the same on both sides
    z = np.stack([(rng.permutation(E) - E / 2) * 0.02 + rng.uniform(-1, 1) for _ in range(T)])
    z = z.astype(np.float32)
    assert _topk_margin(oracle.sigmoid_f32(z), K) > 1e-6
    _check(z, K, L, False)


def test_uniform_usage_closed_form():
    E, K, L = 8, 2, 4
    s = np.full((L, E), 0.25, np.float32)
    for t in range(L):
        s[t, 2 * t:2 * t + 2] = 0.75
    f, P, loss = ops.seq_balance_stats(torch.from_numpy(s).to(DEV), K, L, affinities=True)
    assert (f.cpu().numpy() == 1.0).all()
    np.testing.assert_allclose(P.cpu().numpy(), 1.0 / E, rtol=1e-6)
    assert abs(float(loss[0]) - 1e-4) < 1e-10


def test_deterministic_and_argument_checks():
    rng = np.random.default_rng(9)
    z = torch.from_numpy((rng.standard_normal((1024, 256)) * 3).astype(np.float32)).to(DEV)
    a = ops.seq_balance_stats(z, 8, 256)
    b = ops.seq_balance_stats(z, 8, 256)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    with pytest.raises(MoEError) as e:
        ops.seq_balance_stats(z, 8, 300)                           # 300 does not divide 1024
    assert e.value.status == -1
    with pytest.raises(MoEError) as e:
        ops.seq_balance_stats(z, 257, 256)                         # K > E
    assert e.value.status == -1
