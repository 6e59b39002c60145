"""Finalize-routing and the whole MoE layer (oracle).  Test infrastructure only.

Sources:
* Qwen3-MoE low-latency inference practice, section "GMM enablement and
  routing optimisation": finalize-routing re-arranges the expert outputs back
  into token order and takes their weighted sum to give the final output.
* Hy3 295B MoE practice, sections 1.1-1.2 (one shared expert per MoE layer,
  gate/up 4096->1536, down 1536->4096, added to the routed output) and 8.1
  (the shared-expert term ``shared_expert_x`` belongs to the combine step).

Reading: the shared expert is an ungated FFN with weight 1 (the pages show no
shared-expert gate).  float64 throughout; y is not rounded.
"""
from __future__ import annotations

import numpy as np

from .ffn import _f64, expert_ffn, grouped_gemm, grouped_gemm_swiglu
from .gating import gating_topk
from .mx import mxfp4_weights
from .routing import expand_rows, init_routing, init_routing_range


def finalize_routing(y_perm, pair_pos, T: int, k: int, shared=None) -> np.ndarray:
    """y[t] = sum_j y_perm[pair_pos[t*k+j]] (+ shared[t]); y_perm rows already carry the routing weights.

    A pair with pair_pos = -1 was routed to experts outside the local range (expert-range routing)
    and adds nothing here.
    """
    y_perm = _f64(y_perm)
    pp = np.asarray(pair_pos, np.int64).reshape(T, k)
    rows = y_perm[np.maximum(pp, 0)] * (pp >= 0)[:, :, None]  # [T,k,H]
    y = rows.sum(axis=1)
    if shared is not None:
        y = y + _f64(shared)
    return y


def shared_expert(x, w13_s, w2_s) -> np.ndarray:
    """The shared expert: the same FFN applied to every token, weight 1."""
    return expert_ffn(x, w13_s, w2_s)


def moe_layer_forward(x, logits, k, gate, w13, w2, bias=None, routed_scaling_factor=1.0, eps=1e-20,
                      w13_s=None, w2_s=None) -> dict:
    """Whole layer on all tokens; returns every intermediate the GPU path exposes."""
    x = np.asarray(x)
    T = x.shape[0]
    E = np.asarray(w13).shape[0]
    topk_w, topk_idx = gating_topk(logits, k, gate, bias, routed_scaling_factor, eps)
    counts, offsets, sorted_pair, pair_pos = init_routing(topk_idx, E)
    x_exp = expand_rows(x, sorted_pair, k)
    act = grouped_gemm_swiglu(x_exp, w13, offsets)
    row_scale = topk_w.reshape(-1)[sorted_pair]
    y_perm = grouped_gemm(act, w2, offsets, row_scale)
    shared = shared_expert(x, w13_s, w2_s) if w13_s is not None else None
    y = finalize_routing(y_perm, pair_pos, T, k, shared)
    return dict(topk_w=topk_w, topk_idx=topk_idx, counts=counts, offsets=offsets,
                sorted_pair=sorted_pair, pair_pos=pair_pos, x_exp=x_exp, act=act,
                y_perm=y_perm, shared=shared, y=y)


def moe_layer_forward_tokens(tokens, x, logits, k, gate, w13, w2, bias=None, routed_scaling_factor=1.0,
                             eps=1e-20, w13_s=None, w2_s=None) -> dict:
    """Routing for all tokens, and y only for the listed tokens (for full-size workloads).

    y[t] = sum_j w[t,j] * FFN_{idx[t,j]}(x[t]) + shared(x[t]) for t in ``tokens``;
    each needed expert's weights are widened to float64 one expert at a time.
    """
    x = np.asarray(x)
    tokens = np.asarray(tokens, np.int64)
    E = np.asarray(w13).shape[0]
    topk_w, topk_idx = gating_topk(logits, k, gate, bias, routed_scaling_factor, eps)
    counts, offsets, sorted_pair, pair_pos = init_routing(topk_idx, E)
    H = x.shape[1]
    y = np.zeros((tokens.size, H))
    sel_idx = topk_idx[tokens]  # [n,k]
    sel_w = topk_w[tokens]
    for e in np.unique(sel_idx):
        rr, jj = np.nonzero(sel_idx == e)
        out = expert_ffn(x[tokens[rr]], w13[e], w2[e])
        y[rr] += sel_w[rr, jj][:, None] * out
    if w13_s is not None:
        y += expert_ffn(x[tokens], w13_s, w2_s)
    return dict(topk_w=topk_w, topk_idx=topk_idx, counts=counts, offsets=offsets,
                sorted_pair=sorted_pair, pair_pos=pair_pos, tokens=tokens, y=y)


def moe_layer_forward_range(x, logits, k, gate, w13, w2, e0: int, e1: int, bias=None, routed_scaling_factor=1.0,
                            eps=1e-20) -> dict:
    """The routed part of the layer restricted to the local experts [e0, e1) (Qwen3-MoE practice, MoE
    EP with AllGather + ReduceScatter: routing keeps the tokens of this rank's experts, the GMMs run
    on them and finalize-routing gives this rank's partial output, which the reduce-scatter sums).

    y_part[t] = sum over slots j with e0 <= idx[t,j] < e1 of w[t,j] * FFN_{idx[t,j]}(x[t]).
    """
    x = np.asarray(x)
    T = x.shape[0]
    E = np.asarray(w13).shape[0]
    topk_w, topk_idx = gating_topk(logits, k, gate, bias, routed_scaling_factor, eps)
    counts, offsets, sorted_pair, pair_pos = init_routing_range(topk_idx, E, e0, e1)
    x_exp = expand_rows(x, sorted_pair, k)
    act = grouped_gemm_swiglu(x_exp, w13[e0:e1], offsets)
    y_perm = grouped_gemm(act, w2[e0:e1], offsets, topk_w.reshape(-1)[sorted_pair])
    y = finalize_routing(y_perm, pair_pos, T, k)
    return dict(topk_w=topk_w, topk_idx=topk_idx, counts=counts, offsets=offsets, sorted_pair=sorted_pair,
                pair_pos=pair_pos, x_exp=x_exp, act=act, y_perm=y_perm, y=y)


def moe_layer_forward_tokens_mxfp4(tokens, x, logits, k, gate, w13, w2, bias=None, routed_scaling_factor=1.0,
                                   eps=1e-20) -> dict:
    """The layer with MXFP4 expert weights (Qwen3-MoE practice, W4A8 section: the experts' weights
    are MXFP4), for the listed tokens: every needed expert's w13 and w2 are quantised to MXFP4 along
    their input dimension and decoded (``mx.mxfp4_weights``), then the layer is the bf16 layer's
    definition on those weights.  Routing for all tokens, y for ``tokens``.
    """
    x = np.asarray(x)
    tokens = np.asarray(tokens, np.int64)
    E = np.asarray(w13).shape[0]
    topk_w, topk_idx = gating_topk(logits, k, gate, bias, routed_scaling_factor, eps)
    counts, offsets, sorted_pair, pair_pos = init_routing(topk_idx, E)
    y = np.zeros((tokens.size, x.shape[1]))
    sel_idx = topk_idx[tokens]
    sel_w = topk_w[tokens]
    for e in np.unique(sel_idx):
        rr, jj = np.nonzero(sel_idx == e)
        out = expert_ffn(x[tokens[rr]], mxfp4_weights(w13[e]), mxfp4_weights(w2[e]))
        y[rr] += sel_w[rr, jj][:, None] * out
    return dict(topk_w=topk_w, topk_idx=topk_idx, counts=counts, offsets=offsets,
                sorted_pair=sorted_pair, pair_pos=pair_pos, tokens=tokens, y=y)
