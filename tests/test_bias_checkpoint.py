"""CPU test of the bias checkpoint: the selection bias is the layer's only state that
training updates step by step, and it round-trips through .npy bit for bit."""

import numpy as np
import pytest
import torch

import workloads
from fp8_block_scaled_bias_b300 import load_bias, save_bias


def test_bias_round_trips_bit_for_bit(tmp_path):
    b = workloads.gen_bias(workloads.SKEWED)              # includes the Zipf term
    p = tmp_path / "bias.npy"
    save_bias(b, p)
    out = torch.full_like(b, float("nan"))
    load_bias(p, out)
    assert torch.equal(out.view(torch.int32), b.view(torch.int32))


def test_load_bias_rejects_a_different_expert_count(tmp_path):
    p = tmp_path / "bias.npy"
    save_bias(torch.zeros(16), p)
    with pytest.raises(ValueError):
        load_bias(p, torch.zeros(256))
    np.save(tmp_path / "f64.npy", np.zeros(16))
    with pytest.raises(ValueError):
        load_bias(tmp_path / "f64.npy", torch.zeros(16))
