"""Whole-layer GPU parity (moe_layer_forward through the C ABI) against the oracle.

Small workloads are compared on every output element; the two full-size
prefill workloads are launched exactly as bench.py launches them and compared
bit-exactly on their routing (all tokens) and within tolerance on the outputs
of a sample of tokens that the oracle computes one by one.
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


def _layer(moe, cfg):
    return moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                        cfg.n_shared, cfg.I_s)


def _run(moe, cfg, inp, layer=None):
    layer = layer or _layer(moe, cfg)
    t = dict(x=dev_bf16(inp.x), logits=dev(inp.logits), w13=moe.moe_prepack_w13(dev_bf16(inp.w13)),
             w2=dev_bf16(inp.w2), bias=dev(inp.bias) if inp.bias is not None else None,
             w13_s=moe.moe_prepack_w13(dev_bf16(inp.w13_s)) if inp.w13_s is not None else None,
             w2_s=dev_bf16(inp.w2_s) if inp.w2_s is not None else None)
    layer.forward(**t)
    return layer, t


def _check_routing(moe, layer, ref):
    assert (host(layer.topk_idx) == ref["topk_idx"]).all()
    assert (host(layer.counts) == ref["counts"]).all()
    assert (host(layer.intermediate("offsets")) == ref["offsets"]).all()
    assert (host(layer.intermediate("sorted_pair")) == ref["sorted_pair"]).all()
    assert (host(layer.intermediate("pair_pos")) == ref["pair_pos"]).all()
    np.testing.assert_allclose(host(layer.topk_w), ref["topk_w"], rtol=2e-6, atol=1e-7)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK


SMALL = [
    mi.CONFIGS["tiny"],
    mi.CONFIGS["qwen3_decode"],
    mi.CONFIGS["hy3_decode"],
    mi.CONFIGS["tiny"].with_(T=1, E=1, k=1),                                   # dense MLP
    mi.CONFIGS["tiny"].with_(T=1),                                             # one token
    mi.CONFIGS["hy3_decode"].with_(T=3, H=256, E=64, k=8, I=128, I_s=256),    # shared I_s != I
    mi.CONFIGS["long_prefill"].with_(T=1000, H=512, E=16, k=4, I=256, zipf_beta=0.5, n_dead=3),  # wide tiles, ragged
    mi.CONFIGS["hy3_prefill"].with_(T=600, H=256, E=24, k=6, I=192, I_s=128, zipf_beta=0.4, n_dead=2),
    # >= 256 pairs per expert (compute-bound GEMM instance), K % 128 = 64 in the down GEMM
    mi.CONFIGS["hy3_prefill"].with_(T=1000, H=384, E=8, k=4, I=192, I_s=320, zipf_beta=0.3, n_dead=1),
    # the fused op's bias placement (inside the sigmoid), shared expert
    mi.CONFIGS["hy3_decode"].with_(T=24, H=256, E=32, k=8, I=128, I_s=128, gate="sigmoid_inner_bias", bias_std=0.5),
    # the documented limits: E = 1024 experts, k = 32
    mi.CONFIGS["tiny"].with_(T=64, H=256, E=1024, k=32, I=128),
    # a few rows per routed expert, but a shared expert over 40 tokens: the CTA-pair instances
    mi.CONFIGS["hy3_decode"].with_(T=40, H=256, E=64, k=4, I=128, I_s=128),
    # gating and routing in one kernel up to T*k = 4096 (decode instances), four kernels above
    mi.CONFIGS["qwen3_decode"].with_(T=512, H=256, I=128),
    mi.CONFIGS["qwen3_decode"].with_(T=513, H=256, I=128),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: f"{c.name}-T{c.T}-E{c.E}-k{c.k}-H{c.H}-I{c.I}")
def test_layer_parity_full(moe, cfg):
    inp = mi.generate(cfg)
    ref = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                   cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)
    layer, _ = _run(moe, cfg, inp)
    _check_routing(moe, layer, ref)
    import torch
    xe = host(layer.intermediate("x_exp").view(torch.int16)).view(np.uint16)
    assert (xe == ref["x_exp"]).all()
    assert_close(host_bf16_f64(layer.intermediate("act")), ref["act"], "act")
    assert_close(host_bf16_f64(layer.intermediate("y_perm")), ref["y_perm"], "y_perm")
    if cfg.n_shared:
        assert_close(host_bf16_f64(layer.intermediate("shared")), ref["shared"], "shared expert")
    assert_close(host_bf16_f64(layer.y), ref["y"], "y")


def test_layer_all_tokens_on_one_expert(moe):
    cfg = mi.CONFIGS["tiny"].with_(T=300, E=8, k=2)
    inp = mi.generate(cfg)
    inp.logits[:, 5] = 50.0  # every token picks expert 5 first
    ref = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2)
    assert ref["counts"][5] == cfg.T
    layer, _ = _run(moe, cfg, inp)
    _check_routing(moe, layer, ref)
    assert_close(host_bf16_f64(layer.y), ref["y"], "y")


def test_layer_empty_batch(moe):
    """T = 0: nothing to compute, no launch, MOE_OK."""
    import torch
    cfg = mi.CONFIGS["tiny"]
    inp = mi.generate(cfg)
    layer = moe.MoELayer(0, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate)
    assert moe.moe_layer_kernel_launches(layer.desc) == 0
    y = layer.forward(x=torch.empty((0, cfg.H), dtype=torch.bfloat16, device="cuda"),
                      logits=torch.empty((0, cfg.E), dtype=torch.float32, device="cuda"),
                      w13=moe.moe_prepack_w13(dev_bf16(inp.w13)), w2=dev_bf16(inp.w2))
    torch.cuda.synchronize()
    assert y.shape == (0, cfg.H)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK


def test_layer_is_deterministic(moe):
    cfg = mi.CONFIGS["hy3_decode"]
    inp = mi.generate(cfg)
    layer, t = _run(moe, cfg, inp)
    y1 = layer.y.clone()
    layer.forward(**t)
    import torch
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), layer.y.view(torch.int16))


def _sample_tokens(T, counts_ref, topk_idx, n=48):
    """Evenly spread tokens plus tokens routed to the hottest and to the rarest active experts."""
    toks = set(np.linspace(0, T - 1, n // 2).astype(int).tolist())
    hot = int(np.argmax(counts_ref))
    active = np.nonzero(counts_ref)[0]
    rare = int(active[np.argmin(counts_ref[active])])
    for e in (hot, rare):
        rows = np.nonzero((topk_idx == e).any(1))[0]
        toks.update(rows[: n // 4].tolist())
    return np.array(sorted(toks))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["hy3_prefill", "long_prefill"])
def test_layer_parity_full_size_sampled(moe, name):
    cfg = mi.CONFIGS[name]
    inp = mi.generate(cfg)
    w_ref, idx_ref = oracle.gating_topk(inp.logits, cfg.k, cfg.gate, inp.bias, cfg.routed_scaling_factor, cfg.eps)
    counts_ref = np.bincount(idx_ref.ravel(), minlength=cfg.E)
    toks = _sample_tokens(cfg.T, counts_ref, idx_ref)
    ref = oracle.moe_layer_forward_tokens(toks, inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                          cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)
    layer, _ = _run(moe, cfg, inp)
    _check_routing(moe, layer, ref)
    y = host_bf16_f64(layer.y[dev(toks.astype(np.int64))])
    assert_close(y, ref["y"], f"{name} sampled y")
    # properties that hold at any size: finite output, nothing left unwritten
    import torch
    assert torch.isfinite(layer.y.float()).all()
