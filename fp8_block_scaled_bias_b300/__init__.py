"""B300-native forward of a DeepSeek-V3 MoE FFN layer with FP8 block-scaled experts.

The compute runs in libmoe_fp8.so (hand-written sm_103a CUDA; C-ABI in
include/moe_fp8.h).  This package is its thin Python binding: ``ops`` wraps each entry
point for torch tensors, ``layer`` chains them into one layer forward.
"""

from ._lib import LIB_PATH, MoEError, SIGNATURES, load
from . import ops
from .layer import (MoELayer, MoEWeights, make_weights, interleave_gate_up, quantise_expert,
                    save_bias, load_bias)

__all__ = ["LIB_PATH", "MoEError", "SIGNATURES", "load", "ops", "MoELayer", "MoEWeights",
           "make_weights", "interleave_gate_up", "quantise_expert", "save_bias", "load_bias"]
