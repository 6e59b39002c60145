"""Pins of the W4A8 layer oracle (MXFP8 hidden state x MXFP4 expert weights, act quantised to MXFP8
before the down projection; Qwen3-MoE practice, W4A8 section; Hy3 practice 5.2), against what the
pages and the mathematics fix: a hand-worked example where every input is exact and the act
quantisation ties and saturates (tests/golden/w4a8_hand.json), brute force with explicit loops on
tiny inputs in the dense masked form (sum over all experts, weight 0 for the unchosen ones), the
shared expert as an additive term, and the reduction to the plain expert FFN where act is exactly
representable."""
import json
import os

import numpy as np

import moe_inputs as mi
import oracle
from oracle.mx import e4m3_decode, mx_quantize_e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w4a8_hand.json")


def _bf16(v):
    return mi.f32_to_bf16_bits(np.asarray(v, np.float32))


def test_hand_worked_example():
    g = json.load(open(GOLDEN))
    s = g["shape"]
    T, H, E, k, I = s["T"], s["H"], s["E"], s["k"], s["I"]
    x = np.zeros((T, H))
    for t, h, v in g["x_nonzero"]:
        x[t, h] = v
    w13 = np.zeros((E, 2 * I, H))
    for e, r, c, v in g["w13_nonzero"]:
        w13[e, r, c] = v
    w2 = np.zeros((E, H, I))
    for e, r, c, v in g["w2_nonzero"]:
        w2[e, r, c] = v
    xc, xs = mx_quantize_e4m3(x)
    assert (oracle.mx_dequantize_e4m3(xc, xs) == x).all()          # x is exact in MXFP8
    assert (oracle.mxfp4_weights(w13) == w13).all() and (oracle.mxfp4_weights(w2) == w2).all()
    r = oracle.moe_layer_forward_w4a8(xc, xs, np.float32(g["logits"]), k, s["gate"], _bf16(w13), _bf16(w2))
    want = np.zeros((T, H))
    for t, row in g["y"].items():
        for h, v in row.items():
            want[int(t), int(h)] = v
    assert (r["y"] == want).all(), r["y"][:, :6]
    for t, vals in g["act_values"].items():
        codes, scales = r["act"][int(t) * k]
        deq = oracle.mx_dequantize_e4m3(codes[None], scales[None])[0]
        assert (deq[:len(vals)] == vals).all() and (deq[len(vals):] == 0).all()


def _ffn_loops(x, w13, w2):
    """One token through the W4A8 FFN with explicit loops: the gate/up sums, SiLU * up, the MXFP8 rule
    applied element by element (block amax, power-of-two scale, E4M3 grid by nearest-even search over
    the representable values), the down sums."""
    H, n2 = len(x), len(w13)
    I = n2 // 2
    h = [sum(w13[r][c] * x[c] for c in range(H)) for r in range(n2)]
    act = [h[i] / (1.0 + np.exp(-h[i])) * h[I + i] for i in range(I)]
    grid = np.unique(np.abs(e4m3_decode(np.arange(256, dtype=np.uint8))))
    grid = grid[np.isfinite(grid) & (grid <= 448)]
    q = []
    for b in range(0, I, 32):
        blk = act[b:b + 32]
        amax = max(abs(v) for v in blk)
        X = 2.0 ** max(-127, int(np.floor(np.log2(amax))) - 8) if amax > 0 else 2.0 ** -127
        for v in blk:
            a = min(abs(v) / X, 448.0)
            d = np.abs(grid - a)
            best = grid[d == d.min()]
            if best.size > 1:  # a tie: the value whose code has an even mantissa
                codes = [int(oracle.mx.e4m3_encode(np.array([c]))[0]) for c in best]
                best = [c for c, cd in zip(best, codes) if cd % 2 == 0]
            q.append(np.copysign(float(best[0]), v) * X)
    return [sum(w2[o][i] * q[i] for i in range(I)) for o in range(len(w2))]


def test_brute_force_dense_masked_form():
    rng = np.random.default_rng(5)
    T, H, E, k, I = 3, 64, 4, 2, 32
    x = rng.normal(size=(T, H))
    xc, xs = mx_quantize_e4m3(x)
    xq = oracle.mx_dequantize_e4m3(xc, xs)
    w13 = _bf16(rng.normal(0, 0.3, size=(E, 2 * I, H)))
    w2 = _bf16(rng.normal(0, 0.3, size=(E, H, I)))
    logits = np.float32(np.round(rng.normal(size=(T, E)) * 256) / 256)
    r = oracle.moe_layer_forward_w4a8(xc, xs, logits, k, "softmax", w13, w2)
    tw, ti = oracle.gating_topk(logits, k, "softmax")
    for t in range(T):
        want = np.zeros(H)
        for e in range(E):
            m = tw[t][list(ti[t]).index(e)] if e in ti[t] else 0.0
            w13e, w2e = oracle.mxfp4_weights(w13[e]), oracle.mxfp4_weights(w2[e])
            out = _ffn_loops(list(xq[t]), w13e.tolist(), w2e.tolist())
            want += m * np.array(out)
        np.testing.assert_allclose(r["y"][t], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_shared_expert_adds_its_quantised_ffn():
    cfg = mi.CONFIGS["hy3_decode"].with_(T=5, H=128, E=6, k=2, I=64, I_s=64)
    inp = mi.generate(cfg)
    xc, xs = mx_quantize_e4m3(oracle.bf16_to_f64(inp.x))
    a = oracle.moe_layer_forward_w4a8(xc, xs, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                      cfg.routed_scaling_factor, cfg.eps)
    b = oracle.moe_layer_forward_w4a8(xc, xs, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                      cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)
    s, _, _ = oracle.ffn_w4a8(a["x"], oracle.mxfp4_weights(inp.w13_s), oracle.mxfp4_weights(inp.w2_s))
    np.testing.assert_allclose(b["y"] - a["y"], s, rtol=1e-12, atol=1e-12 * np.abs(s).max())
    # a token subset gives the same rows
    c = oracle.moe_layer_forward_w4a8(xc, xs, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                      cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s, tokens=[3, 1])
    np.testing.assert_allclose(c["y"], b["y"][[3, 1]], rtol=1e-12, atol=1e-15)


def test_reduces_to_the_plain_ffn_when_act_is_representable_and_differs_otherwise():
    # act exactly representable: x = e0, gate rows >= 48 (SiLU(g) = g in float64), up rows powers of two
    H, I = 32, 32
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    w13 = np.zeros((2 * I, H))
    w13[:I, 0] = 64.0
    w13[I:, 0] = 2.0 ** -(np.arange(I) % 4) / 4  # act in {16, 8, 4, 2}: exact at the block scale 2^-4
    w2 = np.eye(H, I) * 0.5
    out, _, _ = oracle.ffn_w4a8(x, w13, w2)
    assert (out == oracle.expert_ffn(x, w13, w2)).all()
    # Gaussian values: the act quantisation changes the result, by at most half an E4M3 step of act
    rng = np.random.default_rng(1)
    x = oracle.mx_dequantize_e4m3(*mx_quantize_e4m3(rng.normal(size=(4, 64))))
    w13 = oracle.mxfp4_weights(rng.normal(0, 0.2, size=(64, 64)))
    w2 = oracle.mxfp4_weights(rng.normal(0, 0.2, size=(64, 32)))
    out, codes, scales = oracle.ffn_w4a8(x, w13, w2)
    plain = oracle.expert_ffn(x, w13, w2)
    assert np.abs(out - plain).max() > 0
    h = x @ w13.T
    act = h[:, :32] / (1 + np.exp(-h[:, :32])) * h[:, 32:]
    deq = oracle.mx_dequantize_e4m3(codes, scales)
    X = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=1)
    sat = np.abs(act) / X > 448  # the block maximum may lie in (448, 512) X: clipped to 448 X
    assert (np.abs(deq - act)[~sat] <= 2.0 ** -4 * np.abs(act)[~sat] + 2.0 ** -10 * X[~sat]).all()
    assert (np.abs(deq[sat]) == 448 * X[sat]).all()
    np.testing.assert_allclose(out, deq @ w2.T, rtol=1e-13)
