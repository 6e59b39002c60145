"""The MoE front end (oracle): fused residual add + RMSNorm + cast, and the router gate GEMM.
Test infrastructure only.

Source: Qwen3-MoE low-latency inference practice (Atlas A3/950), section "fused RMSNorm + Cast":
the normalisation before the MoE must give the hidden state in two precisions, FP32 for the gate
computation and BF16 for the expert computation, and one fused op does the residual add, the
RMSNorm and the dtype conversion: (hidden_fp32, hidden_bf16, _, residual) =
add_rms_norm_cast(hidden, residual, norm_weight, epsilon).  When there is no residual (the first
layer) the op is RMSNorm + cast alone.  The router gate GEMM then maps the FP32 hidden state to
router_logits[T, E].

Readings (the pages give no formulas):
* residual_out = round_bf16(hidden + residual), rounded once (round to nearest even); it is the
  residual stream the next layer reads, and the RMSNorm normalises this value (as the model's
  "h = h + residual; residual = h; h = norm(h)" does);
* RMSNorm(r) = r / sqrt(mean(r^2) + eps) * w, with w the norm weight (bf16, widened exactly);
* hidden_bf16 = round_bf16(hidden_fp32);
* router_logits = hidden_fp32 . w_gate^T with the bf16 gate weight widened exactly (FP32 gate).
float64 throughout; the bf16 roundings are taken from the exact float64 values.
"""
from __future__ import annotations

import numpy as np

from .ffn import _f64


def round_bf16(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 (8 significant bits), ties to even; returned as
    float64.  Normal range only (|v| >= 2^-126), which is all the inputs here produce."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                    # v = m * 2^e, 0.5 <= |m| < 1
    q = np.rint(m * 256.0)                # 8 significant bits; rint rounds halves to even
    return np.ldexp(q, e - 8)


def add_rms_norm_cast(hidden, residual, norm_weight, eps: float):
    """Returns (hidden_f64 [T,H] -- the FP32 output's exact value, hidden_bf16 [T,H] as float64,
    residual_out [T,H] as float64 (bf16 values)).  hidden, residual, norm_weight: bf16 bit patterns
    (uint16) or floats; residual may be None (first layer: no add, residual_out = hidden)."""
    h = _f64(hidden)
    r = h if residual is None else round_bf16(h + _f64(residual))
    w = _f64(norm_weight)
    ms = (r * r).mean(axis=1, keepdims=True)
    y = r / np.sqrt(ms + float(np.float32(eps))) * w[None, :]
    return y, round_bf16(y), r


def router_logits(hidden_f, w_gate) -> np.ndarray:
    """router_logits[T,E] = hidden . w_gate^T (w_gate [E,H], bf16 bit patterns or floats)."""
    return np.asarray(hidden_f, np.float64) @ _f64(w_gate).T
