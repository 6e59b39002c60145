"""Pins of the oracle's finalize-routing and whole layer.

Passages pinned: Qwen3-MoE practice, "GMM enablement and routing optimisation"
(finalize-routing: back to token order, weighted sum); Hy3 practice sections
1.1-1.2 (one shared expert added to the routed output) and 8.1 (shared term
folded into combine).  The layer is checked against the dense definition of a
sparse MoE: y_t = sum over ALL experts e of m_{t,e} * FFN_e(x_t) + shared(x_t),
with m_{t,e} the routing weight if e was chosen and 0 otherwise.
"""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle


def _dense_brute(x, w13, w2, w, idx, w13_s=None, w2_s=None):
    """Plain loops over all experts with masked weights (no routing, no grouping)."""
    xf = oracle.bf16_to_f64(x) if x.dtype == np.uint16 else x
    T, H = xf.shape
    E = w13.shape[0]
    y = np.zeros((T, H))
    for t in range(T):
        for e in range(E):
            m = 0.0
            for j in range(idx.shape[1]):
                if idx[t, j] == e:
                    m = w[t, j]
            if m == 0.0:
                continue
            w13e = oracle.bf16_to_f64(w13[e])
            w2e = oracle.bf16_to_f64(w2[e])
            I = w13e.shape[0] // 2
            g = w13e[:I] @ xf[t]
            u = w13e[I:] @ xf[t]
            a = np.array([gi / (1.0 + math.exp(-gi)) for gi in g]) * u
            y[t] += m * (w2e @ a)
        if w13_s is not None:
            w13s = oracle.bf16_to_f64(w13_s)
            I_s = w13s.shape[0] // 2
            g = w13s[:I_s] @ xf[t]
            u = w13s[I_s:] @ xf[t]
            a = np.array([gi / (1.0 + math.exp(-gi)) for gi in g]) * u
            y[t] += oracle.bf16_to_f64(w2_s) @ a
    return y


def _small(name, **kw):
    return mi.CONFIGS[name].with_(**kw)


@pytest.mark.parametrize("cfg", [
    mi.CONFIGS["tiny"],
    _small("hy3_decode", T=6, H=64, E=10, k=3, I=64, I_s=64),
    _small("long_prefill", T=24, H=64, E=9, k=4, I=64, zipf_beta=0.3, n_dead=2),
])
def test_layer_dense_equivalence(cfg):
    inp = mi.generate(cfg)
    r = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                 cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)
    ref = _dense_brute(inp.x, inp.w13, inp.w2, r["topk_w"], r["topk_idx"], inp.w13_s, inp.w2_s)
    np.testing.assert_allclose(r["y"], ref, rtol=1e-10, atol=1e-12)
    # intermediate consistency: y_perm rows carry the weights of their pairs
    P = cfg.T * cfg.k
    assert r["y_perm"].shape == (P, cfg.H)


def test_layer_single_expert_is_dense_swiglu_mlp():
    """E = 1, k = 1 (softmax): every token's weight is exactly 1 -> a dense SwiGLU MLP (torch CPU)."""
    cfg = mi.CONFIGS["tiny"].with_(E=1, k=1)
    inp = mi.generate(cfg)
    r = oracle.moe_layer_forward(inp.x, inp.logits, 1, "softmax", inp.w13, inp.w2)
    assert (r["topk_w"] == 1.0).all()
    f = lambda u: torch.from_numpy(u.astype(np.int32) << 16).view(torch.float32).double()
    g, u = torch.chunk(torch.nn.functional.linear(f(inp.x), f(inp.w13[0])), 2, -1)
    ref = torch.nn.functional.linear(torch.nn.functional.silu(g) * u, f(inp.w2[0])).numpy()
    np.testing.assert_allclose(r["y"], ref, rtol=1e-11, atol=1e-13)


def test_layer_token_permutation_equivariance():
    cfg = mi.CONFIGS["hy3_decode"].with_(T=12, H=64, E=16, k=4, I=64, I_s=64)
    inp = mi.generate(cfg)
    perm = np.random.default_rng(0).permutation(cfg.T)
    a = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias, 2.826,
                                 1e-20, inp.w13_s, inp.w2_s)
    b = oracle.moe_layer_forward(inp.x[perm], inp.logits[perm], cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                 2.826, 1e-20, inp.w13_s, inp.w2_s)
    np.testing.assert_allclose(b["y"], a["y"][perm], rtol=1e-12, atol=1e-14)
    assert (b["topk_idx"] == a["topk_idx"][perm]).all()


def test_finalize_hand_example():
    # T=2, k=2: pairs p=0..3 at positions pair_pos; y_perm rows hold weighted outputs
    y_perm = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0], [1000.0, 2000.0]])
    pair_pos = np.array([3, 0, 2, 1])
    y = oracle.finalize_routing(y_perm, pair_pos, 2, 2)
    assert y.tolist() == [[1001.0, 2002.0], [110.0, 220.0]]
    s = np.array([[0.5, 0.5], [-1.0, 1.0]])
    assert oracle.finalize_routing(y_perm, pair_pos, 2, 2, s).tolist() == [[1001.5, 2002.5], [109.0, 221.0]]


def test_shared_expert_is_the_plain_ffn():
    cfg = mi.CONFIGS["hy3_decode"].with_(T=3, H=64, E=4, k=2, I=64, I_s=64)
    inp = mi.generate(cfg)
    s = oracle.shared_expert(inp.x, inp.w13_s, inp.w2_s)
    np.testing.assert_allclose(s, oracle.expert_ffn(inp.x, inp.w13_s, inp.w2_s), rtol=0, atol=0)
    # closed form: zero weights give zero output
    z = oracle.shared_expert(inp.x, np.zeros_like(inp.w13_s), inp.w2_s)
    assert (z == 0).all()


def test_tokens_variant_matches_full_forward():
    cfg = mi.CONFIGS["long_prefill"].with_(T=40, H=64, E=12, k=3, I=64, zipf_beta=0.3, n_dead=2)
    inp = mi.generate(cfg)
    full = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2)
    toks = np.array([0, 7, 13, 39])
    part = oracle.moe_layer_forward_tokens(toks, inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2)
    np.testing.assert_allclose(part["y"], full["y"][toks], rtol=1e-12, atol=1e-14)
    for key in ("topk_idx", "counts", "offsets", "sorted_pair", "pair_pos"):
        assert (part[key] == full[key]).all()
