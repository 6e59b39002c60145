"""Expert FFN and the grouped GEMMs (oracle).  Test infrastructure only.

Sources:
* Qwen3-MoE low-latency inference practice, section "MoE TP optimisation:
  computation decomposition": each expert computes x = down(SiLU(gate(x)) *
  up(x)); gate_proj and up_proj are concatenated into ``w13`` ([gate; up]),
  and the fused SwiGLU splits its input in two halves along the last axis and
  returns SiLU(x[0]) * x[1].
* Same page, "GMM enablement and routing optimisation": the grouped matmul
  computes all experts in one op instead of a per-expert loop.
* Hy3 295B MoE practice, section 6.2: the grouped matmul's group_list is the
  per-expert token count; expert weights keep the checkpoint layout
  [out_features, in_features] (used through a transposed view).

float64 throughout; bf16 inputs widen exactly.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(u) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    return bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def swiglu(h) -> np.ndarray:
    """chunk(h, 2, -1) -> (x0, x1); SiLU(x0) * x1 with SiLU(z) = z / (1 + e^-z)."""
    h = np.asarray(h, np.float64)
    x0, x1 = np.split(h, 2, axis=-1)
    return x0 / (1.0 + np.exp(-x0)) * x1


def expert_ffn(x_rows, w13_e, w2_e) -> np.ndarray:
    """down(SiLU(gate(x)) * up(x)) for rows x [n,H]; w13_e [2I,H] = [gate; up]; w2_e [H,I]."""
    h = _f64(x_rows) @ _f64(w13_e).T
    return swiglu(h) @ _f64(w2_e).T


def grouped_gemm_swiglu(x_rows, w13, offsets) -> np.ndarray:
    """act[pos] = SwiGLU(x_rows[pos] . w13[e]^T) for pos in expert e's segment [offsets[e], offsets[e+1])."""
    x_rows = _f64(x_rows)
    E = len(offsets) - 1
    I = np.asarray(w13).shape[1] // 2
    act = np.zeros((x_rows.shape[0], I))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            act[a:b] = swiglu(x_rows[a:b] @ _f64(w13[e]).T)
    return act


def grouped_gemm(a_rows, w, offsets, row_scale=None) -> np.ndarray:
    """out[pos] = row_scale[pos] * (a_rows[pos] . w[e]^T) over expert segments (scale 1 if None)."""
    a_rows = _f64(a_rows)
    E = len(offsets) - 1
    N = np.asarray(w).shape[1]
    out = np.zeros((a_rows.shape[0], N))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = a_rows[lo:hi] @ _f64(w[e]).T
    if row_scale is not None:
        out *= np.asarray(row_scale, np.float64)[:, None]
    return out
