"""GPU parity of the MoE front end (fused residual add + RMSNorm + cast, router gate GEMM)
through the C ABI, against the oracle.

Passage: Qwen3-MoE low-latency inference practice, "fused RMSNorm + Cast" (FP32 for the gate,
BF16 for the experts, one op for add + RMSNorm + cast).
Bars: the residual stream is bit-exact (one bf16 rounding of an exact sum on both sides); the
FP32 output within 1e-5 of the float64 value (fp32 sum of squares and rsqrt); the BF16 output
within one bf16 rounding of the float64 value; the logits within the fp32 dot-product bound
gamma_H * sum_h |y_h w_h| (any summation order), gamma_H = H u / (1 - H u), u = 2^-24.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import assert_bf16_rounding_close, assert_close, dev, dev_bf16, host, host_bf16_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_fwd_gb300 import build
    build.build()
    import moe_expert_layer_fwd_gb300 as m
    return m


def _bf16(seed, tid, shape, mean=0.0, std=1.0):
    return mi.normal_bf16(seed, tid, shape, mean, std)


@pytest.mark.parametrize("T,H,with_res", [(1, 256, True), (37, 2048, True), (37, 2048, False), (300, 4096, True),
                                          (5, 8192, True), (2048, 64, False)])
def test_add_rms_norm_cast_parity(moe, T, H, with_res):
    import torch
    h = _bf16(T + H, 1, (T, H))
    res = _bf16(T + H, 2, (T, H), 0.0, 3.0) if with_res else None
    w = _bf16(T + H, 3, (H,), 1.0, 0.1)
    eps = 1e-6
    y_ref, y16_ref, r_ref = oracle.add_rms_norm_cast(h, res, w, eps)
    y32, y16, r = moe.moe_add_rms_norm_cast(dev_bf16(h), dev_bf16(res) if with_res else None, dev_bf16(w), eps)
    torch.cuda.synchronize()
    if with_res:
        assert (host_bf16_f64(r) == r_ref).all()
    got = host(y32).astype(np.float64)
    assert np.abs(got - y_ref).max() <= 1e-5 * np.abs(y_ref).max()
    assert_bf16_rounding_close(host_bf16_f64(y16), y_ref, "y_bf16")


def test_add_rms_norm_cast_in_place_residual(moe):
    import torch
    T, H = 64, 1024
    h, res, w = _bf16(9, 1, (T, H)), _bf16(9, 2, (T, H)), _bf16(9, 3, (H,), 1.0, 0.1)
    _, _, r_ref = oracle.add_rms_norm_cast(h, res, w, 1e-5)
    d_res = dev_bf16(res)
    moe.moe_add_rms_norm_cast(dev_bf16(h), d_res, dev_bf16(w), 1e-5, residual_out=d_res)
    torch.cuda.synchronize()
    assert (host_bf16_f64(d_res) == r_ref).all()


@pytest.mark.parametrize("T,H,E", [(1, 256, 8), (100, 2048, 128), (1000, 4096, 192), (77, 512, 1024),
                                   (4096, 2048, 128)])
def test_router_logits_parity(moe, T, H, E):
    import torch
    rng = np.random.default_rng(T + E)
    y = rng.normal(size=(T, H)).astype(np.float32)
    wg = _bf16(E, 4, (E, H), 0.0, 0.05)
    ref = oracle.router_logits(y, wg)
    bound_terms = np.abs(y.astype(np.float64)) @ np.abs(oracle.bf16_to_f64(wg)).T
    u = 2.0 ** -24
    gamma = H * u / (1 - H * u)
    got = host(moe.moe_router_logits(dev(y), dev_bf16(wg))).astype(np.float64)
    torch.cuda.synchronize()
    assert (np.abs(got - ref) <= gamma * bound_terms + 1e-30).all()


def test_front_end_feeds_the_layer(moe):
    """add + RMSNorm + cast -> router logits -> the layer, against the oracle taking the same steps
    (the oracle routes on the GPU's logits: routing parity is conditional on the logits)."""
    import torch
    cfg = mi.CONFIGS["tiny"].with_(T=48, H=256, E=16, k=4, I=128)
    inp = mi.generate(cfg)
    res = _bf16(5, 2, (cfg.T, cfg.H), 0.0, 2.0)
    w = _bf16(5, 3, (cfg.H,), 1.0, 0.1)
    wg = _bf16(5, 4, (cfg.E, cfg.H), 0.0, 0.1)
    y32, y16, _ = moe.moe_add_rms_norm_cast(dev_bf16(inp.x), dev_bf16(res), dev_bf16(w), 1e-6)
    logits = moe.moe_router_logits(y32, dev_bf16(wg))
    y_ref, _, _ = oracle.add_rms_norm_cast(inp.x, res, w, 1e-6)
    assert_close(host(logits).astype(np.float64), oracle.router_logits(y_ref, wg), "router logits", 1e-4, 1e-5)
    layer = moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate)
    layer.forward(x=y16, logits=logits, w13=moe.moe_prepack_w13(dev_bf16(inp.w13)), w2=dev_bf16(inp.w2))
    torch.cuda.synchronize()
    x16 = host(y16.view(torch.int16)).view(np.uint16)
    ref = oracle.moe_layer_forward(x16, host(logits), cfg.k, cfg.gate, inp.w13, inp.w2)
    assert (host(layer.topk_idx) == ref["topk_idx"]).all()
    assert_close(host_bf16_f64(layer.y), ref["y"], "layer y")


# ---------------------------------------------------------------- MXFP8 (W4A8 front end)
@pytest.mark.parametrize("T,H,with_res", [(1, 256, True), (37, 2048, True), (64, 4096, False), (300, 8192, True)])
def test_add_rms_norm_mxfp8_parity(moe, T, H, with_res):
    """Codes and scales are integers decided by fp32 arithmetic: the oracle quantises the GPU's own
    fp32 normalised row (same precision); that row is itself checked against float64."""
    import torch
    from oracle.mx import mx_dequantize_e4m3, mx_quantize_e4m3
    h = _bf16(T + H, 11, (T, H))
    res = _bf16(T + H, 12, (T, H), 0.0, 3.0) if with_res else None
    w = _bf16(T + H, 13, (H,), 1.0, 0.3)
    eps = 1e-6
    codes, scales, y32, r = moe.moe_add_rms_norm_mxfp8(dev_bf16(h), dev_bf16(res) if with_res else None,
                                                       dev_bf16(w), eps)
    torch.cuda.synchronize()
    y_ref, _, r_ref = oracle.add_rms_norm_cast(h, res, w, eps)
    y_gpu = host(y32).astype(np.float64)
    assert np.abs(y_gpu - y_ref).max() <= 1e-5 * np.abs(y_ref).max()
    if with_res:
        assert (host_bf16_f64(r) == r_ref).all()
    c_ref, s_ref = mx_quantize_e4m3(y_gpu)
    assert (host(scales) == s_ref).all()
    assert (host(codes) == c_ref).all()
    # the dequantised row: half an E4M3 step of each element, or +-448 X where y / X > 448 (clipped)
    back = mx_dequantize_e4m3(host(codes), host(scales))
    x = np.exp2(host(scales).astype(np.float64) - 127.0).repeat(32, axis=1)
    sat = np.abs(y_gpu) / x > 448
    assert (np.abs(back - y_gpu)[~sat] <= 2.0 ** -4 * np.abs(y_gpu)[~sat] + 2.0 ** -10 * x[~sat]).all()
    assert (np.abs(back[sat]) == 448 * x[sat]).all()
    _end_to_end_mx_agreement(host(codes), host(scales), y_ref, f"T={T} H={H}")


def _end_to_end_mx_agreement(codes, scales, y_ref, what):
    """The GPU's codes against the oracle quantising its own float64 row (not the GPU's fp32 row).
    The fp32 and float64 rows differ by ~1e-7 relative, so a code or a scale can differ only where
    that decides a rounding: a scale byte only for a block whose amax lies within 1e-5 of a power of
    two, a code only by one E4M3 step, for an element within 1e-5 of the midpoint of the two
    neighbouring E4M3 values.  Reports the rate of differing codes."""
    from oracle.mx import e4m3_decode, mx_quantize_e4m3
    c_ref, s_ref = mx_quantize_e4m3(y_ref)
    T, H = codes.shape
    blk = y_ref.reshape(T, H // 32, 32)
    amax = np.abs(blk).max(axis=-1)
    s_diff = scales != s_ref
    if s_diff.any():
        frac = np.log2(amax[s_diff])
        assert (np.abs(frac - np.rint(frac)) <= 1e-5).all(), f"{what}: scale differs away from a power of two"
    same_scale = np.repeat(~s_diff, 32, axis=1)
    mag, mag_ref = codes & 0x7F, c_ref & 0x7F
    differ = (codes != c_ref) & ~((mag == 0) & (mag_ref == 0)) & same_scale
    n = int(differ.sum())
    if n:
        assert (np.abs(mag[differ].astype(int) - mag_ref[differ].astype(int)) == 1).all(), \
            f"{what}: a code differs by more than one E4M3 step"
        x = np.exp2(scales.astype(np.float64) - 127.0).repeat(32, axis=1)
        v = np.abs(y_ref[differ]) / x[differ]
        mid = (np.abs(e4m3_decode(codes[differ])) + np.abs(e4m3_decode(c_ref[differ]))) / 2
        assert (np.abs(v - mid) <= 1e-5 * v).all(), f"{what}: a differing code is not at a rounding boundary"
    print(f"MXFP8 end to end ({what}): {n} of {codes.size} codes ({n / codes.size:.2e}) and "
          f"{int(s_diff.sum())} of {scales.size} scales differ from the float64 oracle, each at a rounding boundary")


def test_mxfp8_zero_rows_and_saturation(moe):
    import torch
    from oracle.mx import mx_quantize_e4m3
    T, H = 4, 256
    h = np.zeros((T, H), np.uint16)          # bf16 zeros: y = 0 everywhere -> scale byte 0, codes 0
    h[1] = mi.normal_bf16(3, 1, (H,))
    h[2, :32] = 0x3F80                       # a block of equal values 1.0 (each 448 after scaling? no:
    w = np.full(H, 0x3F80, np.uint16)        #  amax/X in [256, 512): 1.0 -> 256 exactly)
    codes, scales, y32, _ = moe.moe_add_rms_norm_mxfp8(dev_bf16(h), None, dev_bf16(w), 1e-6)
    torch.cuda.synchronize()
    assert (host(scales)[0] == 0).all() and (host(codes)[0] == 0).all()
    c_ref, s_ref = mx_quantize_e4m3(host(y32).astype(np.float64))
    assert (host(codes) == c_ref).all() and (host(scales) == s_ref).all()
