"""Pins of the oracle's expert-range routing (the expert-parallel form of init-routing).

Passage: Qwen3-MoE low-latency inference practice, MoE EP with AllGather +
ReduceScatter (W4A8 section): after the all-gather, init_routing_v2 keeps only
the tokens of the experts in this rank's range; the GMMs and finalize-routing
then give this rank's partial output, which the reduce-scatter sums over ranks.
Pinned by a hand-worked example, by reduction to plain init-routing on the
whole range, by brute force on tiny inputs, and by the partition identity: the
partial layer outputs of a partition of the experts sum to the whole layer.
"""
import json
import os

import numpy as np
import pytest

import moe_inputs as mi
import oracle


def test_range_routing_hand_example():
    with open(os.path.join(os.path.dirname(__file__), "golden", "routing_range_hand.json")) as f:
        g = json.load(f)
    idx = np.array(g["topk_idx"], np.int32)
    for r in g["ranges"]:
        counts, offsets, sp, pp = oracle.init_routing_range(idx, g["E"], r["e0"], r["e1"])
        assert counts.tolist() == r["counts"]
        assert offsets.tolist() == r["offsets"]
        assert sp.tolist() == r["sorted_pair"]
        assert pp.tolist() == r["pair_pos"]


def test_whole_range_is_init_routing():
    rng = np.random.default_rng(1)
    idx = np.stack([rng.choice(24, 4, replace=False) for _ in range(100)]).astype(np.int32)
    a = oracle.init_routing(idx, 24)
    b = oracle.init_routing_range(idx, 24, 0, 24)
    for u, v in zip(a, b):
        assert (u == v).all()


@pytest.mark.parametrize("seed", range(4))
def test_range_routing_brute_force_and_partition(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 30, 10, 3
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    flat = idx.reshape(-1)
    cuts = np.sort(rng.choice(np.arange(1, E), 3, replace=False))
    bounds = [0, *cuts.tolist(), E]
    all_sp, seen = [], np.zeros(flat.size, int)
    for e0, e1 in zip(bounds[:-1], bounds[1:]):
        counts, offsets, sp, pp = oracle.init_routing_range(idx, E, e0, e1)
        # brute force: a local pair's position counts the local pairs before it in (local expert, p) order
        for p in range(flat.size):
            if e0 <= flat[p] < e1:
                before = sum(1 for q in range(flat.size)
                             if e0 <= flat[q] < e1 and (flat[q], q) < (flat[p], p))
                assert pp[p] == before and sp[before] == p
                seen[p] += 1
            else:
                assert pp[p] == -1
        assert counts.tolist() == [int((flat == e).sum()) for e in range(e0, e1)]
        assert offsets[-1] == sp.size
        all_sp.extend(sp.tolist())
    # the ranges partition the pairs, and their concatenated orders are the whole-range order
    assert (seen == 1).all()
    assert all_sp == oracle.init_routing(idx, E)[2].tolist()


def test_partial_layers_of_a_partition_sum_to_the_layer():
    cfg = mi.CONFIGS["tiny"].with_(T=20, E=12, k=3, H=128, I=64)
    inp = mi.generate(cfg)
    full = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2)
    acc = np.zeros_like(full["y"])
    for e0, e1 in ((0, 5), (5, 6), (6, 12)):
        part = oracle.moe_layer_forward_range(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, e0, e1)
        # the partial output is the dense masked sum over the range's experts (brute force per token)
        for t in range(cfg.T):
            ref = np.zeros(cfg.H)
            for j in range(cfg.k):
                e = int(part["topk_idx"][t, j])
                if e0 <= e < e1:
                    ref += part["topk_w"][t, j] * oracle.expert_ffn(inp.x[t:t + 1], inp.w13[e], inp.w2[e])[0]
            np.testing.assert_allclose(part["y"][t], ref, rtol=1e-12, atol=1e-12)
        acc += part["y"]
    np.testing.assert_allclose(acc, full["y"], rtol=1e-12, atol=1e-12)


def test_range_rejects_bad_bounds():
    idx = np.zeros((2, 1), np.int32)
    for e0, e1 in ((0, 0), (2, 1), (-1, 2), (0, 5)):
        with pytest.raises(ValueError):
            oracle.init_routing_range(idx, 4, e0, e1)
