"""GPU parity of expert-range routing (the expert-parallel form of init-routing) and of the
partial layers it feeds, through the C ABI, against the oracle.

Passage: Qwen3-MoE low-latency inference practice, MoE EP with AllGather + ReduceScatter:
init_routing_v2 keeps the tokens of this rank's expert range, the GMMs run on those experts and
finalize-routing gives the rank's partial output, which the reduce-scatter sums over ranks.  On
one GPU the ranks' slices run one after another and their partial outputs are summed here.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import assert_close, dev, dev_bf16, host, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_fwd_gb300 import build
    build.build()
    import moe_expert_layer_fwd_gb300 as m
    return m


RANGE_CASES = [
    # T, E, k, H, [(e0, e1), ...]
    (16, 8, 2, 256, [(0, 8), (0, 3), (3, 4), (4, 8), (7, 8)]),
    (4096, 128, 8, 64, [(0, 16), (16, 128), (60, 61)]),
    (3, 1024, 32, 128, [(0, 512), (512, 1024), (1000, 1024)]),
    (20000, 7, 3, 64, [(0, 1), (1, 7), (3, 5)]),
]


@pytest.mark.parametrize("T,E,k,H,ranges", RANGE_CASES)
def test_init_routing_range_parity(moe, T, E, k, H, ranges):
    import torch
    rng = np.random.default_rng(T + E)
    p = rng.dirichlet(np.full(E, 0.3))
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32) \
        if T * E <= 2_000_000 else rng.integers(0, E, size=(T, k)).astype(np.int32)
    x = mi.normal_bf16(1, 1, (T, H))
    d_idx, d_x = dev(idx), dev_bf16(x)
    for e0, e1 in ranges:
        counts, offsets, sp, pp = oracle.init_routing_range(idx, E, e0, e1)
        o = moe.moe_init_routing_range(d_idx, E, e0, e1, d_x)
        torch.cuda.synchronize()
        n = int(offsets[-1])
        assert (host(o["counts"]) == counts).all()
        assert (host(o["offsets"]) == offsets).all()
        assert (host(o["sorted_pair"])[:n] == sp).all()
        assert (host(o["pair_pos"]) == pp).all()
        xe = host(o["x_exp"][:n].view(torch.int16)).view(np.uint16)
        assert (xe == oracle.expand_rows(x, sp, k)).all()
        assert moe.moe_get_device_status(o["ws"]) == 0


def test_init_routing_range_rejects_bad_bounds(moe):
    idx = dev(np.zeros((4, 2), np.int32))
    for e0, e1 in ((0, 0), (3, 2), (-1, 2), (0, 9)):
        with pytest.raises(moe.MoEError):
            moe.moe_init_routing_range(idx, 8, e0, e1)


@pytest.mark.parametrize("cfg,parts", [
    (mi.CONFIGS["tiny"].with_(T=64, E=16, k=4, H=256, I=128), [(0, 5), (5, 6), (6, 16)]),
    (mi.CONFIGS["long_prefill"].with_(T=1500, H=512, E=24, k=4, I=192, zipf_beta=0.5, n_dead=3),
     [(0, 12), (12, 24)]),
    (mi.CONFIGS["hy3_decode"].with_(T=48, H=256, E=32, k=8, I=128, n_shared=0, I_s=0), [(0, 8), (8, 32)]),
])
def test_partial_layers_of_an_expert_partition(moe, cfg, parts):
    """Range routing -> local gate/up GEMM -> local down GEMM -> finalize = the range's partial output;
    the partial outputs of a partition of the experts sum to the whole layer."""
    import torch
    inp = mi.generate(cfg)
    full = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                    cfg.routed_scaling_factor, cfg.eps)
    x, logits = dev_bf16(inp.x), dev(inp.logits)
    w13p = moe.moe_prepack_w13(dev_bf16(inp.w13))
    w2 = dev_bf16(inp.w2)
    bias = dev(inp.bias) if inp.bias is not None else None
    topk_w, topk_idx = moe.moe_gating_topk(logits, cfg.k, cfg.gate, bias, cfg.routed_scaling_factor, cfg.eps)
    acc = np.zeros_like(full["y"])
    for e0, e1 in parts:
        ref = oracle.moe_layer_forward_range(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, e0, e1,
                                             inp.bias, cfg.routed_scaling_factor, cfg.eps)
        o = moe.moe_init_routing_range(topk_idx, cfg.E, e0, e1, x)
        act = moe.moe_grouped_gemm_swiglu(o["x_exp"], w13p[e0:e1], o["offsets"])
        y_perm = moe.moe_grouped_gemm(act, w2[e0:e1], o["offsets"], topk_w, o["sorted_pair"])
        y = moe.moe_finalize_routing(y_perm, o["pair_pos"], cfg.T, cfg.k)
        torch.cuda.synchronize()
        assert (host(o["pair_pos"]) == ref["pair_pos"]).all()
        got = host_bf16_f64(y)
        assert_close(got, ref["y"], f"partial y [{e0},{e1})")
        acc += got
        assert moe.moe_get_device_status(o["ws"]) == 0
    assert_close(acc, full["y"], "sum of the partial outputs")


def test_mxfp4_partial_layer_on_a_local_expert_range(moe):
    """The 4-bit-weight GEMMs on a local expert slice: weights quantised and prepacked for all 16
    experts, sliced to [4, 12) with Mxfp4Weights.experts (the pointer offsets include/moe.h states),
    routed with moe_init_routing_range, both 4-bit GEMMs and finalize -> the range's partial output,
    against the oracle's partial layer on the MXFP4-decoded weights."""
    import torch
    cfg = mi.CONFIGS["qwen3_decode"].with_(T=24, H=256, E=16, k=4, I=128)
    e0, e1 = 4, 12
    inp = mi.generate(cfg)
    ref = oracle.moe_layer_forward_range(inp.x, inp.logits, cfg.k, cfg.gate, oracle.mxfp4_weights(inp.w13),
                                         oracle.mxfp4_weights(inp.w2), e0, e1)
    w13q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w13)), gate_up=True).experts(e0, e1)
    w2q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w2)), gate_up=False).experts(e0, e1)
    topk_w, topk_idx = moe.moe_gating_topk(dev(inp.logits), cfg.k, cfg.gate)
    o = moe.moe_init_routing_range(topk_idx, cfg.E, e0, e1)
    torch.cuda.synchronize()
    n_loc = int(o["offsets"][-1].item())
    assert (host(o["offsets"]) == ref["offsets"]).all() and (host(o["pair_pos"]) == ref["pair_pos"]).all()
    x16 = moe.moe_gather_rows_f16(dev_bf16(inp.x), o["sorted_pair"], cfg.k, M=n_loc)
    act = moe.moe_grouped_gemm_swiglu_mxfp4(x16, w13q, o["offsets"])
    y_perm = moe.moe_grouped_gemm_mxfp4(act, w2q, o["offsets"], topk_w, o["sorted_pair"])
    y = moe.moe_finalize_routing(y_perm, o["pair_pos"], cfg.T, cfg.k)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(o["ws"]) == 0
    assert_close(host_bf16_f64(y), ref["y"], f"4-bit partial y [{e0},{e1})")
