"""Pins of the oracle's MoE front end (fused residual add + RMSNorm + cast; router gate GEMM).

Passage: Qwen3-MoE low-latency inference practice, "fused RMSNorm + Cast" (the norm before the
MoE gives FP32 for the gate and BF16 for the experts; one op does add + RMSNorm + cast).
Pinned by closed forms, by torch's bf16 conversion and rms_norm, and by torch's matmul.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.frontend import add_rms_norm_cast, round_bf16, router_logits


def _bits(a_f32):
    """fp32 values -> bf16 bit patterns via torch (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a_f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_round_bf16_closed_forms():
    # spacing at 1 is 2^-7 (8 significant bits); halves go to the even neighbour
    cases = {1.0: 1.0, 1 + 2 ** -7: 1 + 2 ** -7, 1 + 2 ** -8: 1.0, 1 + 3 * 2 ** -8: 1 + 2 ** -6,
             1 + 2 ** -8 + 2 ** -20: 1 + 2 ** -7, -(1 + 2 ** -8): -1.0, 0.0: 0.0, 3.0: 3.0,
             2 - 2 ** -9: 2.0, 1.5 * 2 ** -100: 1.5 * 2 ** -100}
    for v, ref in cases.items():
        assert round_bf16(np.float64(v)) == ref, v


def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    v = (rng.normal(size=20000) * np.exp(rng.uniform(-20, 20, size=20000))).astype(np.float32)
    ours = round_bf16(v.astype(np.float64))
    ref = oracle.bf16_to_f64(_bits(v))
    assert (ours == ref).all()


def _inputs(T, H, seed):
    rng = np.random.default_rng(seed)
    h = _bits(rng.normal(size=(T, H)).astype(np.float32))
    res = _bits(rng.normal(size=(T, H)).astype(np.float32) * 2)
    w = _bits((1 + 0.1 * rng.normal(size=H)).astype(np.float32))
    return h, res, w


def test_add_rms_norm_cast_vs_torch():
    h, res, w = _inputs(37, 256, 1)
    eps = 1e-6
    y, y16, r = add_rms_norm_cast(h, res, w, eps)
    hf, rf, wf = (oracle.bf16_to_f64(a) for a in (h, res, w))
    # residual: the bf16 rounding of the sum (exact in float32 for these operands), via torch
    r_ref = oracle.bf16_to_f64(_bits((hf + rf).astype(np.float32)))
    assert (r == r_ref).all()
    y_ref = torch.nn.functional.rms_norm(torch.from_numpy(r_ref), (256,), torch.from_numpy(wf),
                                         eps=float(np.float32(eps))).numpy()
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-14)
    assert (y16 == round_bf16(y)).all()


def test_rms_norm_closed_forms_and_first_layer():
    H = 64
    w = np.full(H, 1.0)
    c = 3.0
    y, _, r = add_rms_norm_cast(np.full((2, H), c), None, w, 0.0)
    assert (r == c).all()                       # no residual: the residual stream is the input
    np.testing.assert_allclose(y, 1.0, rtol=1e-15)
    # scale invariance (eps = 0) and the eps term: c / sqrt(c^2 + eps)
    h, _, w2 = _inputs(5, H, 2)
    a = add_rms_norm_cast(h, None, w2, 0.0)[0]
    b = add_rms_norm_cast(oracle.bf16_to_f64(h) * 4.0, None, w2, 0.0)[0]
    np.testing.assert_allclose(a, b, rtol=1e-14)
    y, _, _ = add_rms_norm_cast(np.full((1, H), 0.5), None, w, 0.25)
    np.testing.assert_allclose(y, 0.5 / np.sqrt(0.25 + float(np.float32(0.25))), rtol=1e-7)


def test_router_logits_vs_torch_and_hand():
    y = np.array([[1.0, 2.0, -1.0]])
    wg = np.array([[1.0, 0.0, 0.0], [0.5, 0.5, 2.0]])
    np.testing.assert_allclose(router_logits(y, wg), [[1.0, -0.5]], rtol=0)
    rng = np.random.default_rng(3)
    yf = rng.normal(size=(20, 128)).astype(np.float32)
    wg = _bits(rng.normal(size=(16, 128)).astype(np.float32) * 0.05)
    ref = torch.from_numpy(yf).double() @ torch.from_numpy(oracle.bf16_to_f64(wg)).T
    np.testing.assert_allclose(router_logits(yf, wg), ref.numpy(), rtol=1e-13)
