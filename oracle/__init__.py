"""CPU oracle for the DeepSeek-V3 MoE FFN forward with FP8 block scaling.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The CUDA library never calls it and shares no code with it; the only thing both
sides consume is the seeded synthetic data made by ``workloads.py``.

Everything here is plain numpy in float64 (or exactly emulated float32 / E4M3 /
BF16 rounding where the method fixes a narrower type), written for a reader who
wants to check it against the pages by eye, not for speed.

Sources, cited by page title and section:

* "DeepSeek-V3: the recipe, and the interconnect that shaped it"
  (paperfordummies.in) -- sections "The one formula", "Auxiliary-loss-free
  balancing", "Node-limited routing: capping the fan-out", "FP8: the other half
  of the byte reduction".
* "DeepSeek-V3" (deepseek-2024.kryvik.com) -- "The core ideas" 1 (DeepSeekMoE,
  node-limited routing), 2 (auxiliary-loss-free load balancing), 6 (FP8 mixed
  precision, items (a)-(d)).
* The DeepSeek-V3 book (slop-6tp.pages.dev/papers-html/dsv3) -- ch. 2 "RMSNorm and
  SwiGLU", ch. 7 "Fine-grained and Shared Experts", ch. 8 "Routing and Load
  Balancing" (including "The complementary sequence loss"), ch. 15 "Moving Tokens to
  Experts", ch. 16 "Understanding FP8 Numbers", ch. 17 "The Actual Mixed-precision
  Pipeline".

Modules:
  formats  -- E4M3 (fn variant) codec and BF16 rounding
  quant    -- 1x128 activation and 128x128 weight quantisation
  router   -- router logits, sigmoid affinity, group-limited top-k, gates, bias update
  permute  -- stable grouping of (token, slot) pairs into expert segments
  gemm     -- block-scaled GEMM with per-128-K promotion, SwiGLU expert, combine
  layer    -- the whole layer forward, and a per-token variant for large shapes
  balance  -- sequence-wise balance statistics f_i, P_i and the complementary loss
  backward -- expert backward: Dgrad / Wgrad GEMMs, 128x1 regrouping, SwiGLU recompute

Parity pins live in ``tests/test_oracle_*.py``.  Functions without an independent
pin say "parity unpinned" in their docstring.
"""

from .formats import (E4M3_MAX, E4M3_MIN_NORMAL, e4m3_decode, e4m3_decode_table,
                      e4m3_encode, e4m3_round, bf16_round)
from .quant import (quant_1x128, quant_128x128, dequant_1x128, dequant_128x128,
                    quant_1x128_pow2, quant_128x128_pow2)
from .router import router_logits, sigmoid_f32, route, route_token, bias_update
from .permute import permute
from .gemm import blockscaled_gemm, swiglu_expert, combine
from .layer import moe_layer, moe_layer_tokens
from .balance import plain_topk, seq_balance_stats
from .backward import (combine_backward_rows, padded_offsets, quant_128x1_pow2_segments, wgrad, swiglu_backward,
                       dequant_rows_1x128_f32, swiglu_cache, expert_backward)

__all__ = [
    "E4M3_MAX", "E4M3_MIN_NORMAL", "e4m3_decode", "e4m3_decode_table", "e4m3_encode",
    "e4m3_round", "bf16_round", "quant_1x128", "quant_128x128", "dequant_1x128",
    "dequant_128x128", "quant_1x128_pow2", "quant_128x128_pow2", "router_logits", "sigmoid_f32", "route", "route_token",
    "bias_update", "permute", "blockscaled_gemm", "swiglu_expert", "combine",
    "moe_layer", "moe_layer_tokens", "plain_topk", "seq_balance_stats",
    "combine_backward_rows", "padded_offsets", "quant_128x1_pow2_segments", "wgrad", "swiglu_backward",
    "dequant_rows_1x128_f32", "swiglu_cache", "expert_backward",
]
