"""GPU check of moe_permute_noalloc, the permutation entry point that allocates nothing.

Callers that cannot allocate device memory where they call the layer -- inside CUDA
graph capture, under a runtime that owns all device memory, or in a loop where an
allocation would stall the device -- use this entry point; its scratch is a static
device array inside the library.  This test calls it through the C-ABI and compares
every output with moe_permute (which takes caller workspace) on two calls in a row with
different inputs, so stale scratch contents from the first call cannot leak into the
second.  The file sorts last so that a stop-at-first-failure run has already run every
other test; it also passes when run on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

from fp8_block_scaled_bias_b300 import ops
from fp8_block_scaled_bias_b300._lib import call

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _idx(T, K, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _noalloc(idx, E, shared):
    T, K = idx.shape
    rows = T * K + (T if shared else 0)
    out = (torch.full((E,), -7, dtype=torch.int32, device=DEV),
           torch.full((E + 2,), -7, dtype=torch.int32, device=DEV),
           torch.full((rows,), -7, dtype=torch.int32, device=DEV),
           torch.full((T, K), -7, dtype=torch.int32, device=DEV))
    st = ops.new_status(DEV)
    call("moe_permute_noalloc", idx.data_ptr(), T, K, E, int(shared), out[0].data_ptr(),
         out[1].data_ptr(), out[2].data_ptr(), out[3].data_ptr(), st.data_ptr(),
         torch.cuda.current_stream().cuda_stream)
    return out, st


def test_noalloc_permute_matches_workspace_permute_twice():
    cases = [(4096, 8, 256, True, 1), (1000, 4, 16, False, 2)]      # two calls in a row
    for T, K, E, shared, seed in cases:
        idx = torch.from_numpy(_idx(T, K, E, seed)).to(DEV)
        got, st = _noalloc(idx, E, shared)
        want = ops.permute(idx, E, shared, ops.new_status(DEV))
        torch.cuda.synchronize()
        assert ops.status_value(st) == 0
        for g, w, name in zip(got, want, ("counts", "offsets", "row_token", "row_of")):
            assert torch.equal(g, w), name


def test_noalloc_permute_rejects_sizes_beyond_its_scratch():
    # ceil(T/128) * E int32 must fit in the 262144-entry static array
    T, K, E = 128 * 257, 2, 1024
    idx = torch.zeros(T, K, dtype=torch.int32, device=DEV)
    with pytest.raises(Exception) as e:
        _noalloc(idx, E, True)
    assert getattr(e.value, "status", None) == -2
