"""Pins of the oracle's gating top-k against closed forms, brute force and library routines.

Passages pinned: Qwen3-MoE practice, "GMM enablement and routing optimisation"
(fused gating replaces top-k then softmax); Hy3 practice section 1.3 (sigmoid
router, eps 1e-20, weights normalised then x2.826) and section 5.1 P1 note
(bias after the sigmoid, selection only; the fused op's bias inside the sigmoid).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _ulp32(v: float) -> float:
    m, e = math.frexp(abs(v))
    return math.ldexp(1.0, e - 24)


def test_pinned_exp_within_2ulp_of_double_exp():
    xs = np.concatenate([np.linspace(-87.0, 88.0, 400001, dtype=np.float32),
                         np.float32([0.0, -0.0, 1.0, -1.0, 0.5, 1e-8, -1e-8, 88.0, -87.0])])
    got = oracle.exp_f32_pinned(xs).astype(np.float64)
    worst = 0.0
    for x, g in zip(xs.astype(np.float64), got):
        ref = math.exp(x)
        if ref < 1.1754943508222875e-38:  # subnormal range: skip the ulp metric
            continue
        worst = max(worst, abs(g - ref) / _ulp32(ref))
    assert worst <= 2.0, worst


def test_pinned_exp_closed_forms():
    assert oracle.exp_f32_pinned(np.float32([0.0]))[0] == np.float32(1.0)
    assert oracle.exp_f32_pinned(np.float32([-0.0]))[0] == np.float32(1.0)
    # at the float32 nearest n*ln2 the result is 2^n times e^(x - n ln2), within 2 ulp
    for n in (-20, -3, 1, 5, 60, 126):
        xf = float(np.float32(n * math.log(2.0)))
        v = float(oracle.exp_f32_pinned(np.float32([xf]))[0])
        ref = 2.0 ** n * math.exp(xf - n * math.log(2.0))
        assert abs(v - ref) <= 2 * _ulp32(ref)


def test_pinned_sigmoid_closed_forms():
    s = oracle.sigmoid_f32_pinned(np.float32([0.0, 40.0, -40.0, 2.0]))
    assert s[0] == np.float32(0.5)
    assert s[1] == np.float32(1.0)
    assert 0.0 < s[2] < 1e-17
    assert abs(float(s[3]) - 1.0 / (1.0 + math.exp(-2.0))) < 1.2e-7
    l = np.linspace(-30, 30, 2001, dtype=np.float32)
    pair = oracle.sigmoid_f32_pinned(l).astype(np.float64) + oracle.sigmoid_f32_pinned(-l).astype(np.float64)
    assert np.max(np.abs(pair - 1.0)) < 2.5e-7


def _brute_select(keys_row, k):
    """Full sort of all E keys (descending, lower index first on equal keys)."""
    return [e for _, e in sorted(((-float(v), e) for e, v in enumerate(keys_row)))][:k]


@pytest.mark.parametrize("seed", range(6))
def test_softmax_selection_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 40, 12, 4
    logits = (np.round(rng.normal(size=(T, E)) * 4) / 4).astype(np.float32)  # 2^-2 grid: many ties
    logits[0, :] = 0.0
    logits[1, :5] = -0.0  # -0 == +0
    _, idx = oracle.gating_topk(logits, k, "softmax")
    for t in range(T):
        assert list(idx[t]) == _brute_select(logits[t], k)
    assert list(idx[0]) == [0, 1, 2, 3]


def test_sigmoid_selection_matches_double_precision_keys_away_from_ties():
    rng = np.random.default_rng(11)
    T, E, k = 200, 64, 8
    logits = (np.round(rng.normal(size=(T, E)) * 256) / 256).astype(np.float32)
    bias = rng.normal(0, 0.01, size=E).astype(np.float32)
    _, idx = oracle.gating_topk(logits, k, "sigmoid", bias, 2.826)
    checked = 0
    for t in range(T):
        keys = [1.0 / (1.0 + math.exp(-float(l))) + float(b) for l, b in zip(logits[t], bias)]
        srt = sorted(keys, reverse=True)
        if srt[k - 1] - srt[k] < 1e-6:
            continue  # near tie: float32 decides
        checked += 1
        assert list(idx[t]) == _brute_select(keys, k)
    assert checked > 150


def test_sigmoid_tie_break_and_bias_selects_only():
    logits = np.zeros((2, 6), np.float32)
    # equal keys -> lowest indices
    w, idx = oracle.gating_topk(logits, 3, "sigmoid", None, 2.826)
    assert list(idx[0]) == [0, 1, 2]
    # closed form: all sigma = 1/2 -> each weight = 0.5 / (1.5 + eps) * 2.826
    np.testing.assert_allclose(w[0], [2.826 / 3] * 3, rtol=1e-6)
    # a bias changes the choice but not the weight formula
    bias = np.float32([0, 0, 0, 0, 0, 5.0])
    w2, idx2 = oracle.gating_topk(logits, 3, "sigmoid", bias, 2.826)
    assert list(idx2[0]) == [5, 0, 1]
    np.testing.assert_allclose(w2[0], w[0], rtol=0, atol=1e-12)


def test_softmax_closed_form():
    logits = np.float32([[0.0, math.log(3.0)]])
    w, idx = oracle.gating_topk(logits, 2, "softmax")
    assert list(idx[0]) == [1, 0]
    np.testing.assert_allclose(w[0], [0.75, 0.25], rtol=1e-6)
    w1, idx1 = oracle.gating_topk(logits, 1, "softmax")
    assert w1[0, 0] == 1.0 and idx1[0, 0] == 1


def test_topk_then_softmax_equals_renormalised_full_softmax():
    """'top-k then softmax' == softmax over all E, gathered and renormalised (torch CPU)."""
    rng = np.random.default_rng(3)
    logits = (np.round(rng.normal(size=(64, 32)) * 256) / 256).astype(np.float32)
    w, idx = oracle.gating_topk(logits, 6, "softmax")
    p = torch.softmax(torch.from_numpy(logits).double(), dim=-1)
    g = torch.gather(p, 1, torch.from_numpy(idx).long())
    ref = (g / g.sum(-1, keepdim=True)).numpy()
    np.testing.assert_allclose(w, ref, rtol=1e-12)


@pytest.mark.parametrize("gate,target", [("softmax", 1.0), ("sigmoid", 2.826)])
def test_weight_invariants(gate, target):
    rng = np.random.default_rng(5)
    logits = (np.round(rng.normal(size=(300, 48)) * 256) / 256).astype(np.float32)
    bias = rng.normal(0, 0.01, size=48).astype(np.float32) if gate == "sigmoid" else None
    w, idx = oracle.gating_topk(logits, 8, gate, bias, target)
    np.testing.assert_allclose(w.sum(1), float(np.float32(target)), rtol=1e-6)
    assert (w >= 0).all()
    for t in range(idx.shape[0]):
        assert len(set(idx[t])) == 8
    if gate == "softmax":
        assert (np.diff(w, axis=1) <= 1e-15).all()
    else:
        # sigmoid weights use sigma of the logit only (no bias): closed form per row
        sig = 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx, 1).astype(np.float64)))
        np.testing.assert_allclose(w, sig / sig.sum(1, keepdims=True) * float(np.float32(2.826)), rtol=1e-12)


# ---------------------------------------------------------------- bias inside the sigmoid
def _golden_bias_placement():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "gating_bias_placement.json")) as f:
        return json.load(f)


def test_bias_placement_hand_example():
    g = _golden_bias_placement()
    logits = np.float32([g["logits"]])
    bias = np.float32(g["bias"])
    m = g["model_after_sigmoid"]
    w, idx = oracle.gating_topk(logits, m["k"], "sigmoid", bias, g["routed_scaling_factor"], g["eps"])
    assert list(idx[0]) == m["topk_idx"]
    np.testing.assert_allclose(w[0], m["topk_w"], rtol=1e-6)
    for case in g["fused_inside_sigmoid"]:
        w, idx = oracle.gating_topk(logits, case["k"], "sigmoid_inner_bias", bias, g["routed_scaling_factor"],
                                    g["eps"])
        assert list(idx[0]) == case["topk_idx"]
        np.testing.assert_allclose(w[0], case["topk_w"], rtol=1e-6)


def test_inner_bias_without_bias_is_the_plain_sigmoid_gate():
    rng = np.random.default_rng(21)
    logits = (np.round(rng.normal(size=(200, 40)) * 256) / 256).astype(np.float32)
    for bias in (None, np.zeros(40, np.float32)):
        w0, i0 = oracle.gating_topk(logits, 6, "sigmoid", None, 2.826)
        w1, i1 = oracle.gating_topk(logits, 6, "sigmoid_inner_bias", bias, 2.826)
        assert (i0 == i1).all()
        np.testing.assert_allclose(w1, w0, rtol=1e-12)


def test_inner_bias_selection_is_the_order_of_logit_plus_bias():
    """sigmoid is strictly increasing: away from float32 ties the choice is the top-k of l + b."""
    rng = np.random.default_rng(23)
    T, E, k = 200, 64, 8
    logits = (np.round(rng.normal(size=(T, E)) * 256) / 256).astype(np.float32)
    bias = rng.normal(0, 0.5, size=E).astype(np.float32)
    w, idx = oracle.gating_topk(logits, k, "sigmoid_inner_bias", bias, 2.826)
    checked = 0
    for t in range(T):
        z = [float(l) + float(b) for l, b in zip(logits[t], bias)]
        keys = [1.0 / (1.0 + math.exp(-v)) for v in z]
        srt = sorted(keys, reverse=True)
        if srt[k - 1] - srt[k] < 1e-6:
            continue
        checked += 1
        assert list(idx[t]) == _brute_select(z, k)
        sel = [keys[e] for e in idx[t]]
        np.testing.assert_allclose(w[t], np.array(sel) / sum(sel) * float(np.float32(2.826)), rtol=1e-9)
    assert checked > 150
    np.testing.assert_allclose(w.sum(1), float(np.float32(2.826)), rtol=1e-6)
