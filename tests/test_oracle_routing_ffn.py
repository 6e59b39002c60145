"""Pins of the oracle's init-routing, expert FFN and grouped GEMMs.

Passages pinned: Qwen3-MoE practice, "GMM enablement and routing optimisation"
(init-routing order, per-expert token counts, grouped matmul) and "MoE TP
optimisation: computation decomposition" (FFN, [gate; up] concat, SwiGLU);
Hy3 practice section 6.2 (group_list = per-expert counts); the LLM-inference
note, section 5 "matrix principle of tensor parallelism" (column split
concatenates, K split sums).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_routing_hand_example():
    g = _load("routing_hand.json")
    counts, offsets, sp, pp = oracle.init_routing(np.array(g["topk_idx"], np.int32), g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert sp.tolist() == g["sorted_pair"]
    assert pp.tolist() == g["pair_pos"]


def _brute_routing(idx_flat, E):
    """Counting sort written as two plain loops."""
    buckets = [[] for _ in range(E)]
    for p, e in enumerate(idx_flat):
        buckets[e].append(p)
    counts = [len(b) for b in buckets]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    sp = [p for b in buckets for p in b]
    pp = [0] * len(sp)
    for pos, p in enumerate(sp):
        pp[p] = pos
    return counts, offsets, sp, pp


@pytest.mark.parametrize("T,E,k,seed", [(1, 1, 1, 0), (5, 3, 2, 1), (37, 16, 4, 2), (64, 128, 8, 3), (9, 200, 8, 4)])
def test_routing_brute_force_and_invariants(T, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, sp, pp = oracle.init_routing(idx, E)
    bc, bo, bsp, bpp = _brute_routing(idx.reshape(-1).tolist(), E)
    assert counts.tolist() == bc and offsets.tolist() == bo
    assert sp.tolist() == bsp and pp.tolist() == bpp
    P = T * k
    assert counts.sum() == P and offsets[-1] == P and (np.diff(offsets) >= 0).all()
    assert sorted(sp.tolist()) == list(range(P))           # bijection
    assert (pp[sp] == np.arange(P)).all()                    # inverse
    flat = idx.reshape(-1)
    for e in range(E):
        seg = sp[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()                      # stable: ascending p


def test_routing_all_on_one_expert_and_rejects_bad_index():
    idx = np.full((7, 1), 3, np.int32)
    counts, offsets, sp, pp = oracle.init_routing(idx, 5)
    assert counts.tolist() == [0, 0, 0, 7, 0]
    assert sp.tolist() == list(range(7))
    with pytest.raises(ValueError):
        oracle.init_routing(np.array([[5]], np.int32), 5)


def test_expand_rows():
    x = np.arange(12).reshape(4, 3)
    sp = np.array([5, 0, 7, 2, 1, 3, 4, 6])
    got = oracle.expand_rows(x, sp, 2)
    assert got.tolist() == [x[2].tolist(), x[0].tolist(), x[3].tolist(), x[1].tolist(),
                            x[0].tolist(), x[1].tolist(), x[2].tolist(), x[3].tolist()]


def test_bf16_widening_closed_forms():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3EAA, 0x7F7F, 0x0001], np.uint16)
    v = oracle.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 0.0 and v[3] == 0.0 and math.copysign(1, v[3]) < 0
    assert v[4] == (1 + 42 / 128) * 0.25  # 0.33203125
    assert v[5] == (2 - 2.0 ** -7) * 2.0 ** 127
    assert v[6] == 2.0 ** -133


def test_swiglu_chunk_identity_vs_torch():
    rng = np.random.default_rng(0)
    h = rng.normal(size=(7, 20)) * 3
    th = torch.from_numpy(h)
    x0, x1 = torch.chunk(th, 2, -1)
    ref = (torch.nn.functional.silu(x0) * x1).numpy()
    np.testing.assert_allclose(oracle.swiglu(h), ref, rtol=1e-13, atol=1e-15)


def test_ffn_hand_example():
    g = _load("ffn_hand.json")
    x = np.array([g["x"]])
    w13 = np.array(g["w13"])
    w2 = np.array(g["w2"])
    act = oracle.swiglu(x @ w13.T)
    np.testing.assert_allclose(act[0], g["act"], rtol=1e-15)
    np.testing.assert_allclose(oracle.expert_ffn(x, w13, w2)[0], g["out"], rtol=1e-15)
    # the concat order matters: [up; gate] gives another answer
    swapped = np.concatenate([w13[2:], w13[:2]])
    assert not np.allclose(oracle.expert_ffn(x, swapped, w2)[0], g["out"])


def test_expert_ffn_triple_loop():
    rng = np.random.default_rng(1)
    n, H, I = 3, 5, 4
    x, w13, w2 = rng.normal(size=(n, H)), rng.normal(size=(2 * I, H)), rng.normal(size=(H, I))
    out = np.zeros((n, H))
    for r in range(n):
        a = []
        for i in range(I):
            g = sum(x[r, c] * w13[i, c] for c in range(H))
            u = sum(x[r, c] * w13[I + i, c] for c in range(H))
            a.append(g / (1 + math.exp(-g)) * u)
        for o in range(H):
            out[r, o] = sum(a[i] * w2[o, i] for i in range(I))
    np.testing.assert_allclose(oracle.expert_ffn(x, w13, w2), out, rtol=1e-12, atol=1e-14)


def test_expert_ffn_vs_torch_bf16_inputs():
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(6, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w13 = ((rng.normal(size=(64, 64)) * 0.02).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w2 = ((rng.normal(size=(64, 32)) * 0.02).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    tx = torch.from_numpy(x.astype(np.int32) << 16).view(torch.float32).double()
    t13 = torch.from_numpy(w13.astype(np.int32) << 16).view(torch.float32).double()
    t2 = torch.from_numpy(w2.astype(np.int32) << 16).view(torch.float32).double()
    g, u = torch.chunk(torch.nn.functional.linear(tx, t13), 2, -1)
    ref = torch.nn.functional.linear(torch.nn.functional.silu(g) * u, t2).numpy()
    np.testing.assert_allclose(oracle.expert_ffn(x, w13, w2), ref, rtol=1e-12, atol=1e-14)


def test_grouped_gemms_rowwise_brute_force_with_empty_experts():
    rng = np.random.default_rng(4)
    E, H, I = 5, 8, 6
    counts = [3, 0, 1, 0, 4]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    M = offsets[-1]
    x = rng.normal(size=(M, H))
    w13 = rng.normal(size=(E, 2 * I, H))
    w2 = rng.normal(size=(E, H, I))
    scale = rng.normal(size=M)
    act = oracle.grouped_gemm_swiglu(x, w13, offsets)
    out = oracle.grouped_gemm(act, w2, offsets, scale)
    for pos in range(M):
        e = int(np.searchsorted(offsets, pos, side="right") - 1)
        h = w13[e] @ x[pos]
        a = h[:I] / (1 + np.exp(-h[:I])) * h[I:]
        np.testing.assert_allclose(act[pos], a, rtol=1e-12)
        np.testing.assert_allclose(out[pos], scale[pos] * (w2[e] @ a), rtol=1e-12)


def test_tensor_parallel_split_identities():
    """Column split of gate/up concatenates; K split of down sums (LLM-inference note section 5)."""
    rng = np.random.default_rng(5)
    H, I = 16, 8
    x = rng.normal(size=(4, H))
    w13 = rng.normal(size=(2 * I, H))
    w2 = rng.normal(size=(H, I))
    full = oracle.expert_ffn(x, w13, w2)
    h = I // 2
    parts = []
    for r in range(2):
        w13_r = np.concatenate([w13[r * h:(r + 1) * h], w13[I + r * h:I + (r + 1) * h]])
        parts.append(oracle.expert_ffn(x, w13_r, w2[:, r * h:(r + 1) * h]))
    np.testing.assert_allclose(parts[0] + parts[1], full, rtol=1e-12, atol=1e-12)
