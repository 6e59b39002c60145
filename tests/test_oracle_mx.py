"""Pins of the oracle's MXFP8 (E4M3) dynamic quantisation.

Passage: Qwen3-MoE low-latency inference practice, W4A8 section (MXFP8 quantisation of the
hidden state: npu_dynamic_mx_quant; fused add + RMSNorm + MXFP8 quant with round_mode 'rint',
dst_type float8_e4m3fn).  Pinned by closed forms of the E4M3 grid, by torch's float8_e4m3fn
conversion (inside the finite range), by exhaustive encode/decode of all 254 finite codes, and by
the block-scale rule on hand-made blocks.
"""
import numpy as np
import pytest
import torch

from oracle.mx import e4m3_decode, e4m3_encode, e4m3_round, mx_dequantize_e4m3, mx_quantize_e4m3


def test_e4m3_grid_closed_forms():
    cases = {0.0: 0.0, 1.0: 1.0, 1.0625: 1.0, 1.1875: 1.25, 1.125: 1.125, 448.0: 448.0, 460.0: 448.0,
             1e6: 448.0, 2.0 ** -9: 2.0 ** -9, 2.0 ** -10: 0.0, 3 * 2.0 ** -11: 2.0 ** -9, -3.3: -3.25,
             240.0: 240.0, 248.0: 256.0, 17.0: 16.0}
    for v, ref in cases.items():
        assert e4m3_round(np.float64(v)) == ref, v


def test_all_codes_round_trip():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = e4m3_decode(codes)
    assert (e4m3_encode(vals)[vals != 0] == codes[vals != 0]).all()
    assert (e4m3_round(vals) == vals).all()
    assert np.abs(vals).max() == 448.0


def test_e4m3_matches_torch_in_range():
    rng = np.random.default_rng(0)
    v = (rng.normal(size=50000) * np.exp(rng.uniform(-12, 6, size=50000))).astype(np.float32)
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert (e4m3_round(v.astype(np.float64)) == ref).all()


def test_block_scale_rule():
    blk = np.zeros((2, 32))
    blk[0, 5] = 1.0          # amax 1 -> floor(log2) 0 -> shared -8 -> scale byte 119
    blk[0, 6] = -0.0078125   # 2^-7 -> 2^-7 / 2^-8 = 2 exactly
    codes, scales = mx_quantize_e4m3(blk)
    assert scales[:, 0].tolist() == [119, 0]            # second block all zero -> byte 0
    assert e4m3_decode(codes[0, 5]) == 256.0 and e4m3_decode(codes[0, 6]) == -2.0
    assert (codes[1] == 0).all()
    back = mx_dequantize_e4m3(codes, scales)
    np.testing.assert_array_equal(back[0], blk[0])
    # amax just below a power of two: 1.99 -> shared -8, 1.99 * 256 = 509.4 saturates to 448
    c2, s2 = mx_quantize_e4m3(np.full((1, 32), 1.99))
    assert s2[0, 0] == 119 and e4m3_decode(c2[0, 0]) == 448.0


@pytest.mark.parametrize("seed", range(3))
def test_dequantisation_error_bound(seed):
    rng = np.random.default_rng(seed)
    v = rng.normal(size=(64, 256)) * np.exp(rng.uniform(-8, 8, size=(64, 1)))
    codes, scales = mx_quantize_e4m3(v)
    back = mx_dequantize_e4m3(codes, scales)
    x = np.exp2(scales.astype(np.float64) - 127.0).repeat(32, axis=1)
    # below saturation the error is at most half a quantum of v's binade in units of the scale
    q = np.abs(v) / x
    ok = q <= 448
    bound = 0.5 * np.exp2(np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3.0) * x
    assert (np.abs(back - v)[ok] <= bound[ok] * (1 + 1e-12)).all()


# ---------------------------------------------------------------- MXFP4 (E2M1) weights
import oracle  # noqa: E402
from oracle.mx import E2M1_GRID, e2m1_round_index, mx_dequantize_e2m1, mx_quantize_e2m1  # noqa: E402


def test_e2m1_grid_closed_forms():
    cases = {0.0: 0.0, 0.2: 0.0, 0.25: 0.0, 0.26: 0.5, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0,
             5.0: 4.0, 5.1: 6.0, 7.0: 6.0, 100.0: 6.0, -1.3: -1.5, -0.74: -0.5}
    for v, ref in cases.items():
        got = np.sign(v) * E2M1_GRID[e2m1_round_index(np.float64(v))]
        assert got == ref, v


def test_e2m1_blocks_and_packing():
    w = np.zeros((2, 64))
    w[0, 0], w[0, 1], w[0, 2] = 6.0, -0.5, 1.0    # amax 6 -> floor(log2 6) = 2 -> shared 0 -> scale byte 127
    w[0, 33] = 0.75                               # second block: amax 0.75 -> floor -1 -> shared -3
    w[1, 5] = 3.0 * 2.0 ** -10                    # amax 3*2^-10 -> floor -9 -> shared -11: 3.0 exactly
    codes, scales = mx_quantize_e2m1(w)
    assert scales.tolist() == [[127, 124], [116, 0]]
    assert codes[0, 0] == (7 | (8 | 1) << 4)      # 6.0 (idx 7) low nibble, -0.5 (sign, idx 1) high nibble
    assert codes[0, 1] & 0xF == 2                 # 1.0 -> idx 2
    assert (codes[0, 16] >> 4) == 7               # element 33: 0.75 / 2^-3 = 6.0 -> idx 7, high nibble
    back = mx_dequantize_e2m1(codes, scales)
    np.testing.assert_array_equal(back, w)


@pytest.mark.parametrize("seed", range(3))
def test_e2m1_error_bound(seed):
    rng = np.random.default_rng(seed)
    w = rng.normal(0, 0.02, size=(32, 256))
    codes, scales = mx_quantize_e2m1(w)
    back = mx_dequantize_e2m1(codes, scales)
    x = np.exp2(scales.astype(np.float64) - 127.0).repeat(32, axis=1)
    q = np.abs(w) / x
    half = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0)) * x
    ok = q <= 6
    assert (np.abs(back - w)[ok] <= half[ok] * (1 + 1e-12)).all()
    assert (np.abs(back[~ok]) == 6 * x[~ok]).all()


def _representable_mxfp4(rng, shape):
    """Weights that MXFP4 holds exactly: E2M1 grid values times a power of two per block of 32,
    each block's largest magnitude being 4 or 6 times its scale (so the scale rule picks it)."""
    R, K = shape
    v = rng.choice(E2M1_GRID, size=(R, K)) * rng.choice([-1.0, 1.0], size=(R, K))
    v = v.reshape(R, K // 32, 32)
    v[:, :, 0] = rng.choice([4.0, 6.0, -4.0, -6.0], size=(R, K // 32))
    X = rng.integers(-12, -3, size=(R, K // 32, 1)).astype(np.float64)
    return (v * np.exp2(X)).reshape(R, K)


def test_mxfp4_weights_identity_on_representable():
    rng = np.random.default_rng(5)
    w = _representable_mxfp4(rng, (24, 128))
    np.testing.assert_array_equal(oracle.mxfp4_weights(w), w)
    np.testing.assert_array_equal(oracle.mxfp4_weights(w.reshape(2, 12, 128)), w.reshape(2, 12, 128))


def _layer_inputs(seed, T=6, H=64, E=4, k=2, I=32):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, H))
    logits = rng.normal(size=(T, E)).astype(np.float32)
    w13 = rng.normal(0, 0.05, size=(E, 2 * I, H))
    w2 = rng.normal(0, 0.05, size=(E, H, I))
    return rng, x, logits, w13, w2, k


def test_mxfp4_layer_is_the_layer_on_decoded_weights():
    rng, x, logits, w13, w2, k = _layer_inputs(1)
    E, twoI, H = w13.shape
    toks = np.arange(x.shape[0])
    # representable weights: the 4-bit layer is the bf16 layer's definition exactly
    w13r = _representable_mxfp4(rng, (E * twoI, H)).reshape(w13.shape)
    w2r = _representable_mxfp4(rng, (E * H, w2.shape[2])).reshape(w2.shape)
    a = oracle.moe_layer_forward_tokens_mxfp4(toks, x, logits, k, "softmax", w13r, w2r)
    b = oracle.moe_layer_forward_tokens(toks, x, logits, k, "softmax", w13r, w2r)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-13, atol=1e-15)
    # each of the two weights goes through the quantiser: w2 alone, then w13 alone
    a = oracle.moe_layer_forward_tokens_mxfp4(toks, x, logits, k, "softmax", w13r, w2)
    b = oracle.moe_layer_forward_tokens(toks, x, logits, k, "softmax", w13r, oracle.mxfp4_weights(w2))
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-14)
    a = oracle.moe_layer_forward_tokens_mxfp4(toks, x, logits, k, "softmax", w13, w2r)
    b = oracle.moe_layer_forward_tokens(toks, x, logits, k, "softmax", oracle.mxfp4_weights(w13), w2r)
    np.testing.assert_allclose(a["y"], b["y"], rtol=1e-12, atol=1e-14)
    # and on general weights it is not the bf16 layer (4-bit weights round visibly)
    a = oracle.moe_layer_forward_tokens_mxfp4(toks, x, logits, k, "softmax", w13, w2)
    b = oracle.moe_layer_forward_tokens(toks, x, logits, k, "softmax", w13, w2)
    rel = np.abs(a["y"] - b["y"]).max() / np.abs(b["y"]).max()
    assert 1e-3 < rel < 0.5


def _nearest_e2m1_index_brute(q: float) -> int:
    """Nearest E2M1 magnitude by searching all eight, ties to the even index (even mantissa bit),
    anything beyond 6 -> 6."""
    a = min(abs(q), 6.0)
    d = [abs(a - g) for g in E2M1_GRID]
    best = min(d)
    cands = [i for i, x in enumerate(d) if x == best]
    even = [i for i in cands if i % 2 == 0]
    return even[0] if even else cands[0]


@pytest.mark.parametrize("seed", range(4))
def test_e2m1_rounding_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    # values on a fine dyadic grid (many exact ties) and plain random values, up to beyond 6
    q = np.concatenate([np.round(rng.uniform(-7, 7, 4000) * 8) / 8, rng.uniform(-7, 7, 4000)])
    got = e2m1_round_index(q)
    ref = np.array([_nearest_e2m1_index_brute(float(v)) for v in q])
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("seed", range(3))
def test_mxfp4_scale_rule_via_frexp(seed):
    import math
    rng = np.random.default_rng(200 + seed)
    w = rng.normal(0, 1, size=(16, 128)) * np.exp2(rng.integers(-30, 30, size=(16, 1)))
    w[0, :32] = 0.0
    codes, scales = mx_quantize_e2m1(w)
    for r in range(16):
        for b in range(4):
            amax = float(np.abs(w[r, 32 * b:32 * b + 32]).max())
            if amax == 0.0:
                assert scales[r, b] == 0
                continue
            m, e = math.frexp(amax)          # amax = m * 2^e, 0.5 <= m < 1: floor(log2 amax) = e - 1
            assert int(scales[r, b]) - 127 == max(-127, min(127, (e - 1) - 2))
    # and every decoded element is the brute-force nearest grid point of v / scale, with v's sign
    back = mx_dequantize_e2m1(codes, scales)
    x = np.exp2(scales.astype(np.float64) - 127.0).repeat(32, axis=1)
    for v, bk, s in zip(w.ravel()[:2000], back.ravel()[:2000], x.ravel()[:2000]):
        i = _nearest_e2m1_index_brute(v / s)
        assert bk == (np.sign(v) if i else 1.0) * E2M1_GRID[i] * s
