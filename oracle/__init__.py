"""CPU oracle of the sparse MoE expert-layer forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import or run this package.
The product (``moe_expert_layer_fwd_gb300``) never imports it, and this package
imports nothing from the product: the two share no code.  The only module both
sides use is ``moe_inputs`` (seeded inputs, none of the method's arithmetic).

What it computes, step by step, each function citing the passage it follows:

* ``gating``   -- top-k expert choice and weights (softmax, or sigmoid with a
  selection-only correction bias and a routed scaling factor, or the fused op's
  variant with the bias inside the sigmoid).
* ``routing``  -- init-routing: stable sort of token-expert pairs by expert,
  per-expert counts, offsets, the permutation and its inverse; and the same
  restricted to a local expert range (the expert-parallel form).
* ``ffn``      -- the expert FFN down(SiLU(gate(x)) * up(x)) over the
  concatenated [gate; up] weight, grouped per expert.
* ``layer``    -- finalize-routing (unpermute, weighted sum, shared-expert add),
  the whole layer, the routed part of the layer over a local expert range, and the
  layer on MXFP4 expert weights (for sampled tokens).
* ``frontend`` -- the step before gating: fused residual add + RMSNorm + cast
  (FP32 for the gate, BF16 for the experts) and the router gate GEMM.
* ``mx``       -- MXFP8 (E4M3 elements, E8M0 scale per 32) dynamic quantisation, and
  MXFP4 (E2M1 elements) expert weights.
* ``w4a8``     -- the W4A8 layer: MXFP8 hidden state times MXFP4 expert weights, the SwiGLU
  output quantised to MXFP8 before the down projection.

Precision: float64 everywhere, except the expert *selection*, which is an
integer decided by floating point and is therefore taken in float32 with the
same pinned operations the GPU uses (``gating.exp_f32_pinned``).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
brute force and library routines (no function is "parity unpinned").
"""
from .gating import exp_f32_pinned, sigmoid_f32_pinned, selection_keys, gating_topk
from .routing import init_routing, init_routing_range, expand_rows
from .ffn import swiglu, expert_ffn, grouped_gemm_swiglu, grouped_gemm, bf16_to_f64
from .frontend import add_rms_norm_cast, round_bf16, router_logits
from .mx import (mx_dequantize_e2m1, mx_dequantize_e4m3, mx_quantize_e2m1, mx_quantize_e4m3,
                 mxfp4_weights)
from .w4a8 import ffn_w4a8, moe_layer_forward_w4a8
from .layer import (finalize_routing, moe_layer_forward, moe_layer_forward_range, moe_layer_forward_tokens,
                    moe_layer_forward_tokens_mxfp4, shared_expert)

__all__ = [
    "exp_f32_pinned", "sigmoid_f32_pinned", "selection_keys", "gating_topk",
    "init_routing", "init_routing_range", "expand_rows",
    "swiglu", "expert_ffn", "grouped_gemm_swiglu", "grouped_gemm", "bf16_to_f64",
    "add_rms_norm_cast", "round_bf16", "router_logits", "mx_quantize_e4m3", "mx_dequantize_e4m3",
    "mx_quantize_e2m1", "mx_dequantize_e2m1", "mxfp4_weights",
    "finalize_routing", "moe_layer_forward", "moe_layer_forward_range", "moe_layer_forward_tokens",
    "moe_layer_forward_tokens_mxfp4", "shared_expert", "ffn_w4a8", "moe_layer_forward_w4a8",
]
