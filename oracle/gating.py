"""Gating top-k (oracle).  Test infrastructure only.

Sources:
* Qwen3-MoE low-latency inference practice (Atlas A3/950), section "GMM
  enablement and routing optimisation": the fused gating op replaces
  "top-k, then softmax" -- routing scores per token and its top-k experts.
* Hy3 295B MoE end-to-end inference practice, section 1.3 (sigmoid router:
  ``npu_moe_gating_top_k(router_logits, k, bias=e_score_correction_bias,
  norm_type=1, routed_scaling_factor, eps=1e-20)``; the seven small ops it
  replaces are sigmoid, top-k, gather, normalise, scale; top-k weights x2.826)
  and section 5.1 "P1 precision note" (in the model the correction bias is
  added AFTER the sigmoid and only affects which experts are chosen; the fused
  op adds it INSIDE the sigmoid -- gate "sigmoid_inner_bias" here).
* For the fused op's placement the pages say only that the bias sits inside
  the sigmoid; the reading taken: one sigmoid s_e = sigma(l_e + b_e) serves both
  the choice and the weights (normalised with eps, scaled like "sigmoid").

Readings (the pages are silent or garbled here):
* ties between equal selection keys go to the lower expert index, and keys
  compare as IEEE floats (-0 == +0);
* "eps1e-20" is the epsilon added to the denominator of the normalisation;
* the selection key is computed in float32 with pinned operations (below) on
  both sides, because a float decides an integer here;
* weights are computed in float64 from the exact definition.
"""
from __future__ import annotations

import numpy as np

# --- pinned float32 exp ---------------------------------------------------
# Cody-Waite reduction x = n*ln2 + r with ln2 = C1 + C2 (C1 = 355/512 holds 9
# bits so n*C1 is exact for |n| < 2^15), n = rint(x*log2(e)), then the degree-7
# Taylor polynomial of e^r (coefficients 1/m! rounded to float32) by Horner
# with separately rounded multiply and add, then scaling by the exact float
# 2^n.  Domain: x is clamped to [-87, 88] so that 2^n stays a normal float.
# Every step is one IEEE binary32 round-to-nearest operation, so any
# implementation that performs the same operations in the same order gets the
# same bits.
_LOG2E = np.float32(1.4426950408889634)
_C1 = np.float32(0.693359375)
_C2 = np.float32(-2.12194440e-4)
_COEF = [np.float32(1.0 / f) for f in (1.0, 1.0, 2.0, 6.0, 24.0, 120.0, 720.0, 5040.0)]
_LO = np.float32(-87.0)
_HI = np.float32(88.0)


def exp_f32_pinned(x) -> np.ndarray:
    """e^x in float32 by the pinned operation sequence described above."""
    x = np.minimum(np.maximum(np.asarray(x, np.float32), _LO), _HI)
    n = np.rint(x * _LOG2E)
    r = (x - n * _C1) - n * _C2
    p = np.full_like(r, _COEF[7])
    for c in _COEF[6::-1]:
        p = p * r + c
    scale = ((n.astype(np.int32) + 127) << 23).view(np.float32)
    return (p * scale).astype(np.float32)


def sigmoid_f32_pinned(l) -> np.ndarray:
    """1 / (1 + e^-l) in float32: pinned exp, then one RN add and one RN divide."""
    l = np.asarray(l, np.float32)
    e = exp_f32_pinned(-l)
    return (np.float32(1.0) / (np.float32(1.0) + e)).astype(np.float32)


def selection_keys(logits: np.ndarray, gate: str, bias=None) -> np.ndarray:
    """float32 keys whose top-k (descending, lower index on ties) are the chosen experts.

    softmax: softmax is strictly increasing in the logit, so the logit itself is
    the key (top-k of the probabilities == top-k of the logits).
    sigmoid: sigma(l) + bias, the bias added after the sigmoid (Hy3 section 5.1).
    sigmoid_inner_bias: sigma(l + bias), the sum rounded once to float32.
    """
    logits = np.asarray(logits, np.float32)
    if gate == "softmax":
        return logits.copy()
    if gate == "sigmoid":
        s = sigmoid_f32_pinned(logits)
        if bias is not None:
            s = (s + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
        return s
    if gate == "sigmoid_inner_bias":
        z = logits if bias is None else (logits + np.asarray(bias, np.float32)[None, :]).astype(np.float32)
        return sigmoid_f32_pinned(z)
    raise ValueError(f"unknown gate {gate!r}")


def gating_topk(logits, k: int, gate: str, bias=None, routed_scaling_factor: float = 1.0,
                eps: float = 1e-20):
    """Returns (topk_w float64 [T,k], topk_idx int32 [T,k]); slot j holds the j-th best expert.

    softmax: w_j = exp(l_j - l_max) / sum_j' exp(l_j' - l_max) over the k chosen
      logits ("top-k then softmax" equals softmax over all E renormalised over k).
    sigmoid: w_j = sigma_j / (sum_j' sigma_j' + eps) * routed_scaling_factor, with
      sigma the plain sigmoid of the logit (bias excluded).
    sigmoid_inner_bias: the same with sigma_j = sigmoid(l_j + b_j).
    """
    logits = np.asarray(logits, np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    keys = selection_keys(logits, gate, bias)
    eidx = np.broadcast_to(np.arange(E, dtype=np.int64), (T, E))
    # lexsort: last key is primary -> descending key, then ascending expert id
    order = np.lexsort((eidx, -keys), axis=-1)
    topk_idx = order[:, :k].astype(np.int32)
    l = np.take_along_axis(logits, topk_idx, axis=1).astype(np.float64)
    if gate == "softmax":
        z = np.exp(l - l.max(axis=1, keepdims=True))
        w = z / z.sum(axis=1, keepdims=True)
    else:
        if gate == "sigmoid_inner_bias" and bias is not None:
            l = l + np.asarray(bias, np.float64)[topk_idx]
        sig = 1.0 / (1.0 + np.exp(-l))
        rsf = float(np.float32(routed_scaling_factor))
        w = sig / (sig.sum(axis=1, keepdims=True) + float(np.float32(eps))) * rsf
    return w, topk_idx
