"""GPU parity of the MXFP4-weight decode path (W4A8 section of the Qwen3-MoE practice: MXFP4
expert weights) against the oracle, through the C ABI.

* the quantiser: codes and scale bytes bit-exact against oracle.mx_quantize_e2m1;
* the two grouped GEMMs on weights the oracle quantised: f16 token rows that the oracle reads
  exactly; act (f16) and y_perm (bf16) within one rounding of the oracle's float64 result on the
  decoded weights, and within the layer tolerance;
* scale exponents spread over many binades inside a row (the per-row exponent offset);
* the layer composed from the C entry points at the qwen3_decode size, launched as bench.py's
  4-bit leg launches it: routing bit-exact for all tokens, y of sampled tokens within tolerance.
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


def _torch():
    import torch
    return torch


def _segments(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _f16_input(seed, shape, std=1.0):
    """Seeded token rows that are exactly f16 (the 4-bit GEMMs' operand type)."""
    return oracle.bf16_to_f64(mi.normal_bf16(seed, 11, shape, 0.0, std)).astype(np.float16)


def _assert_f16_rounding_close(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = 2.0 ** -11 * np.abs(ref) + 2e-3 * np.abs(ref).max()
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside one f16 rounding, e.g. {np.argwhere(bad)[:3]}"


def _assert_bf16_rounding_close(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = 2.0 ** -8 * np.abs(ref) + 2e-3 * np.abs(ref).max()
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside one bf16 rounding, e.g. {np.argwhere(bad)[:3]}"


# ---------------------------------------------------------------- quantiser
def test_mxfp4_quantize_bit_exact(moe):
    w = mi.normal_bf16(3, 1, (96, 512), 0.0, 0.02)
    f = oracle.bf16_to_f64(w).reshape(96, 16, 32)
    f[0, 0] = 0.0                                    # all-zero block
    f[0, 1] = 0.0
    f[0, 1, 7] = -2.0 ** -130                        # subnormal amax
    f[1, 0, :8] = [6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25]  # E2M1 ties (scale 1)
    f[1, 0, 8:16] = [-6.0, -5.0, -3.5, -2.5, -1.75, -1.25, -0.75, -0.25]
    f[2, 3] = 1e30                                   # large scale
    f[3, 3, :] = 7.9                                 # saturation at 6 * scale
    w = mi.f32_to_bf16_bits(f.reshape(96, 512).astype(np.float32))
    codes_ref, scales_ref = oracle.mx_quantize_e2m1(oracle.bf16_to_f64(w))
    codes, scales = moe.moe_mxfp4_quantize(dev_bf16(w))
    assert (host(scales) == scales_ref).all(), "scale bytes differ"
    assert (host(codes) == codes_ref).all(), "codes differ"


# ---------------------------------------------------------------- grouped GEMMs
def _quantised(w_bf16):
    """Oracle-side quantisation of bf16 weights [E, n, K]: (codes, scales, decoded float64)."""
    E, n, K = w_bf16.shape
    c, s = oracle.mx_quantize_e2m1(oracle.bf16_to_f64(w_bf16).reshape(E * n, K))
    return c.reshape(E, n, K // 2), s.reshape(E, n, K // 32), oracle.mx_dequantize_e2m1(c, s).reshape(E, n, K)


GEMM_CASES = [
    ([5, 0, 40, 1, 17], 320, 192),        # 2 token tiles in one expert, empty expert, K tail (5 x 64)
    ([3, 0, 8, 1, 2, 5, 0, 33], 1024, 512),
    ([1], 256, 128),
    ([0, 0, 7], 192, 64),
]


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_grouped_gemm_swiglu_mxfp4_parity(moe, counts, H, I):
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    seed = 100 + M + H + I
    x16 = _f16_input(seed, (M, H))
    w13 = mi.normal_bf16(seed, 2, (E, 2 * I, H), 0.0, 0.02)
    codes, scales, w13_deq = _quantised(w13)
    ref = oracle.grouped_gemm_swiglu(x16.astype(np.float64), w13_deq, off)
    wq = moe.moe_mxfp4_prepack(dev(codes), dev(scales), gate_up=True)
    act = moe.moe_grouped_gemm_swiglu_mxfp4(dev(x16), wq, dev(off))
    got = host(act).astype(np.float64)
    assert_close(got, ref, "act")
    _assert_f16_rounding_close(got, ref, "act")


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_grouped_gemm_down_mxfp4_parity(moe, counts, H, I):
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    N = max(128, H // 128 * 128)
    seed = 200 + M + H
    a16 = _f16_input(seed, (M, I), 0.5)
    w2 = mi.normal_bf16(seed, 3, (E, N, I), 0.0, 0.02)
    codes, scales, w2_deq = _quantised(w2)
    topk_w = (np.abs(mi.normal_f32(seed, 5, (M, 1))) + 0.1).astype(np.float32)
    sorted_pair = np.random.default_rng(seed).permutation(M).astype(np.int32)
    ref = oracle.grouped_gemm(a16.astype(np.float64), w2_deq, off, topk_w.reshape(-1)[sorted_pair])
    wq = moe.moe_mxfp4_prepack(dev(codes), dev(scales), gate_up=False)
    out = moe.moe_grouped_gemm_mxfp4(dev(a16), wq, dev(off), dev(topk_w), dev(sorted_pair))
    got = host_bf16_f64(out)
    assert_close(got, ref, "y_perm")
    _assert_bf16_rounding_close(got, ref, "y_perm")
    ref1 = oracle.grouped_gemm(a16.astype(np.float64), w2_deq, off)
    _assert_bf16_rounding_close(host_bf16_f64(moe.moe_grouped_gemm_mxfp4(dev(a16), wq, dev(off))), ref1, "plain")


def test_mxfp4_gemm_wide_scale_range(moe):
    """Rows whose block scales span 35 binades (plus all-zero blocks and an all-zero row): the
    per-row exponent offset keeps every block exact in f16."""
    rng = np.random.default_rng(9)
    E, N, K, M = 2, 256, 512, 20
    codes = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    scales = rng.integers(127 - 30, 127 + 6, size=(E, N, K // 32)).astype(np.uint8)
    scales[:, :, 0] = 127 + 5          # the row's largest block
    scales[0, 3, 2] = 0                 # a block at 2^-127 (far below the row's largest: dropped)
    codes[0, 4, :] = 0                  # an all-zero row
    scales[0, 4, :] = 0
    deq = oracle.mx_dequantize_e2m1(codes.reshape(E * N, K // 2), scales.reshape(E * N, K // 32)).reshape(E, N, K)
    a16 = _f16_input(17, (M, K), 0.5)
    off = _segments([7, 13])
    ref = oracle.grouped_gemm(a16.astype(np.float64), deq, off)
    wq = moe.moe_mxfp4_prepack(dev(codes), dev(scales), gate_up=False)
    got = host_bf16_f64(moe.moe_grouped_gemm_mxfp4(dev(a16), wq, dev(off)))
    assert_close(got, ref, "wide")
    _assert_bf16_rounding_close(got, ref, "wide")
    assert (got[:7, 4] == 0).all() and (got[7:, 4] != 0).any()  # expert 0's row 4 is zero, expert 1's is not


def test_mxfp4_gemm_rejects_inconsistent_offsets(moe):
    torch = _torch()
    off = np.array([0, 5, 3, 8], np.int32)
    codes = np.zeros((3, 256, 128), np.uint8)
    scales = np.full((3, 256, 8), 127, np.uint8)
    wq = moe.moe_mxfp4_prepack(dev(codes), dev(scales), gate_up=True)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    act = torch.full((8, 128), 7.0, dtype=torch.float16, device="cuda")
    moe.moe_grouped_gemm_swiglu_mxfp4(dev(_f16_input(1, (8, 256))), wq, dev(off), act=act, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert (act.float() == 7.0).all()


def test_gather_rows_f16(moe):
    T, k, H = 40, 3, 192
    x = mi.normal_bf16(4, 1, (T, H), 0.0, 3.0)
    f = oracle.bf16_to_f64(x)
    f[0, :4] = [1e6, -1e6, 65520.0, 2.0 ** -20]       # saturation and f16 subnormals
    x = mi.f32_to_bf16_bits(f.astype(np.float32))
    sp = np.random.default_rng(4).permutation(T * k).astype(np.int32)
    got = host(moe.moe_gather_rows_f16(dev_bf16(x), dev(sp), k)).astype(np.float64)
    ref = np.clip(oracle.bf16_to_f64(x)[sp // k], -65504.0, 65504.0).astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)
    # pair indices outside [0, T*k) (also small negative ones, which divide to token 0): row skipped, flagged
    torch = _torch()
    bad = sp.copy()
    bad[3], bad[5] = -1, T * k
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = torch.full((T * k, H), 7.0, dtype=torch.float16, device="cuda")
    moe.moe_gather_rows_f16(dev_bf16(x), dev(bad), k, out=out, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    o = host(out).astype(np.float64)
    assert (o[3] == 7.0).all() and (o[5] == 7.0).all()
    keep = np.ones(T * k, bool)
    keep[[3, 5]] = False
    np.testing.assert_array_equal(o[keep], ref[keep])


# ---------------------------------------------------------------- the layer on 4-bit weights (moe.Mxfp4Layer, as bench.py runs it)
@pytest.mark.parametrize("name,over", [("qwen3_decode", dict(T=24, H=512, E=16, I=256)),
                                       ("tiny", dict(I=128)),
                                       pytest.param("qwen3_decode", {}, marks=pytest.mark.slow)])
def test_mxfp4_layer_parity(moe, name, over):
    cfg = mi.CONFIGS[name].with_(**over)
    inp = mi.generate(cfg)
    w13q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w13)), gate_up=True)
    w2q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w2)), gate_up=False)
    layer = moe.Mxfp4Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps)
    y_dev = layer.forward(dev_bf16(inp.x), dev(inp.logits), w13q, w2q,
                          dev(inp.bias) if inp.bias is not None else None)
    toks = np.arange(cfg.T) if cfg.T * cfg.E * cfg.I * cfg.H < 2 ** 31 else np.array([0, cfg.T - 1])
    ref = oracle.moe_layer_forward_tokens_mxfp4(toks, inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                                cfg.routed_scaling_factor, cfg.eps)
    assert (host(layer.topk_idx) == ref["topk_idx"]).all()
    assert (host(layer.routing["offsets"]) == ref["offsets"]).all()
    assert (host(layer.routing["sorted_pair"]) == ref["sorted_pair"]).all()
    assert (host(layer.routing["pair_pos"]) == ref["pair_pos"]).all()
    y = host_bf16_f64(y_dev)
    assert_close(y[toks], ref["y"], f"{name} y")
    assert _torch().isfinite(y_dev.float()).all()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    assert moe.moe_get_device_status(layer.routing_ws) == moe.MOE_OK
