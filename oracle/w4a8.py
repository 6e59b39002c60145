"""The W4A8 expert layer (oracle): MXFP8 activations times MXFP4 expert weights.  Test
infrastructure only.

Sources:
* Qwen3-MoE low-latency inference practice (Atlas A3/950), MoE EP section, "computation
  decomposition (AllGather scheme, W4A8 quantisation)": the hidden state is quantised to MXFP8
  (npu_dynamic_mx_quant gives the MXFP8 data and its scale), the tokens are routed
  (init_routing_v2), the grouped matmuls (npu_grouped_matmul) run on that MXFP8 data with the
  experts' MXFP4 weights, and finalize-routing takes the weighted sum.
* Hy3 295B MoE practice, section 5.2: on the quantised path the SwiGLU is the fused
  SwiGLU + group quantisation (npu_swiglu_group_quant): the activation that enters the down
  projection is quantised as well.

Readings (the pages name the formats and the ops, not their arithmetic):
* x is given as MXFP8 (E4M3 codes, one E8M0 scale per 32 along H: ``mx.mx_quantize_e4m3``); the
  GEMMs see its exact values, codes times scales.
* The expert weights are the checkpoint's bf16 weights quantised to MXFP4 along their input
  dimension (``mx.mxfp4_weights``); the GEMMs see their exact values.
* Products are exact and sums are taken in float64 here (the GPU accumulates in fp32).
* act = SiLU(g) * u of the gate/up result, then quantised to MXFP8 along I with the same rule as x
  (blocks of 32 consecutive features of a row, E8M0 scale 2^(floor(log2 amax) - 8), E4M3
  round-half-to-even saturating at 448); the down projection sees the quantised act.  The
  quantisation of act is an integer decision the GPU takes on its fp32 act: where the fp32 and the
  float64 values fall on two sides of a rounding boundary the two act codes differ by one E4M3 step
  -- a difference far inside the layer tolerance, against which the GPU path is checked.
* The routing weight multiplies the down projection's result (the bf16 layer's order); the shared
  expert is the same quantised FFN with its own MXFP4 weights, weight 1.
"""
from __future__ import annotations

import numpy as np

from .gating import gating_topk
from .mx import mx_dequantize_e4m3, mx_quantize_e4m3, mxfp4_weights
from .routing import init_routing


def ffn_w4a8(x, w13, w2):
    """x [n,H] float64 (MXFP8 values), w13 [2I,H] and w2 [H,I] float64 (MXFP4 values) ->
    (out [n,H], act_codes [n,I], act_scales [n,I/32]): h = x . w13^T, act = SiLU(h[:, :I]) * h[:, I:],
    quantised to MXFP8 along I, out = dequant(act) . w2^T."""
    h = np.asarray(x, np.float64) @ np.asarray(w13, np.float64).T
    I = h.shape[1] // 2
    g, u = h[:, :I], h[:, I:]
    act = g / (1.0 + np.exp(-g)) * u
    codes, scales = mx_quantize_e4m3(act)
    out = mx_dequantize_e4m3(codes, scales) @ np.asarray(w2, np.float64).T
    return out, codes, scales


def moe_layer_forward_w4a8(x_codes, x_scales, logits, k, gate, w13, w2, bias=None, routed_scaling_factor=1.0,
                           eps=1e-20, w13_s=None, w2_s=None, tokens=None) -> dict:
    """The W4A8 layer.  x_codes [T,H] / x_scales [T,H/32]: MXFP8 hidden state; w13 [E,2I,H], w2
    [E,H,I] (and the shared expert's w13_s [2I_s,H], w2_s [H,I_s]): bf16 checkpoint weights, each
    needed expert quantised to MXFP4 here.  Routing for all tokens; y (float64) for ``tokens``
    (default: all), and for every pair of those tokens its act codes and scales (keyed by pair
    index p = t*k + j)."""
    x = mx_dequantize_e4m3(x_codes, x_scales)
    T, H = x.shape
    E = np.asarray(w13).shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, np.int64)
    topk_w, topk_idx = gating_topk(logits, k, gate, bias, routed_scaling_factor, eps)
    counts, offsets, sorted_pair, pair_pos = init_routing(topk_idx, E)
    y = np.zeros((tokens.size, H))
    act = {}
    sel_idx = topk_idx[tokens]
    sel_w = topk_w[tokens]
    for e in np.unique(sel_idx):
        rr, jj = np.nonzero(sel_idx == e)
        out, ac, asc = ffn_w4a8(x[tokens[rr]], mxfp4_weights(w13[e]), mxfp4_weights(w2[e]))
        y[rr] += sel_w[rr, jj][:, None] * out
        for n, (r, j) in enumerate(zip(rr, jj)):
            act[int(tokens[r]) * k + int(j)] = (ac[n], asc[n])
    shared = None
    if w13_s is not None:
        shared, sc, ss = ffn_w4a8(x[tokens], mxfp4_weights(w13_s), mxfp4_weights(w2_s))
        y += shared
    return dict(topk_w=topk_w, topk_idx=topk_idx, counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_pos=pair_pos, tokens=tokens, y=y, act=act, shared=shared, x=x)

