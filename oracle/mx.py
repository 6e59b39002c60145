"""MXFP8 (E4M3) dynamic quantisation and MXFP4 (E2M1) weights (oracle).  Test infrastructure only.

Source: Qwen3-MoE low-latency inference practice (Atlas A3/950), MoE EP / W4A8 section: the
MXFP8 quantisation of the hidden state (npu_dynamic_mx_quant, giving the MXFP8 data and its
scale), and the fused residual add + RMSNorm + MXFP8 dynamic quantisation
(npu_add_rms_norm_dynamic_mx_quant(..., round_mode='rint', dst_type=float8_e4m3fn), giving the
MX data, the residual and the scale).

Readings (the pages name the format, not its rules): the OCP microscaling (MX) format --
blocks of 32 consecutive elements along the hidden dimension share one power-of-two scale
X = 2^(floor(log2(amax)) - 8) stored as an E8M0 byte (exponent + 127, clamped to [-127, 127]),
8 being the largest exponent of an E4M3 normal; every element is v / X rounded to E4M3 with
round-half-to-even ('rint') and saturated to +-448; an all-zero block gets scale byte 0 and zero
codes.  E4M3 (the "fn" variant): sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals
with exponent 0 (2^-6 * m/8), no infinities, 0x7F/0xFF not produced.

MXFP4 expert weights (same section: the W4A8 path's weights are MXFP4).  Reading: the same block
rule with the E2M1 element -- blocks of 32 along the weight's input dimension, scale
X = 2^(floor(log2 amax) - 2) (2 being the largest E2M1 exponent), elements v / X rounded to the E2M1
grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} nearest-even and saturated at 6; a code is sign << 3 | magnitude
index, two codes per byte with element 2j in the low nibble.  ``mxfp4_weights`` gives the float64
weights such a checkpoint holds.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_round(q) -> np.ndarray:
    """Round float64 magnitudes-with-sign to the nearest E4M3 value (ties to even), saturating."""
    q = np.asarray(q, np.float64)
    a = np.minimum(np.abs(q), E4M3_MAX)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                      # subnormal binade shares the quantum 2^-9
    quantum = np.exp2(e - 3.0)
    r = np.rint(a / quantum) * quantum           # rint: halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.sign(q) * r, 0.0 * q)


def e4m3_encode(v) -> np.ndarray:
    """E4M3 values (already representable) -> code bytes."""
    v = np.asarray(v, np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = a >= 2.0 ** -6
    exp_b = np.where(normal, e + 7, 0).astype(np.int64)
    mant = np.where(normal, a / np.exp2(e) - 1.0, a / 2.0 ** -6) * 8.0
    code = (exp_b << 3) | np.rint(mant).astype(np.int64)
    return (np.where(a > 0, code, 0).astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(c) -> np.ndarray:
    """Code bytes -> float64 values."""
    c = np.asarray(c, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    eb = (c >> 3) & 0xF
    m = c & 0x7
    return s * np.where(eb > 0, (1.0 + m / 8.0) * np.exp2(eb - 7.0), (m / 8.0) * 2.0 ** -6)


def mx_quantize_e4m3(v, block: int = 32):
    """v [..., n] (n a multiple of 32) -> (codes uint8 [..., n], scales uint8 [..., n/32])."""
    v = np.asarray(v, np.float64)
    shp = v.shape
    b = v.reshape(*shp[:-1], shp[-1] // block, block)
    amax = np.abs(b).max(axis=-1)
    fl = np.floor(np.log2(np.where(amax > 0, amax, 1.0)))
    shared = np.clip(fl - 8.0, -127.0, 127.0)
    shared = np.where(amax > 0, shared, -127.0)
    scales = (shared + 127.0).astype(np.uint8)
    q = e4m3_round(b / np.exp2(shared)[..., None])
    codes = e4m3_encode(q).reshape(shp)
    return codes, scales


def mx_dequantize_e4m3(codes, scales, block: int = 32) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    shp = codes.shape
    vals = e4m3_decode(codes).reshape(*shp[:-1], shp[-1] // block, block)
    x = np.exp2(np.asarray(scales, np.float64) - 127.0)
    return (vals * x[..., None]).reshape(shp)


# ---------------------------------------------------------------- MXFP4 (E2M1) weights
# The W4A8 path's expert weights (Qwen3-MoE practice, W4A8 section: MXFP4 weights).  Same block
# rule with the E2M1 element: blocks of 32 along the reduction dimension K, scale
# X = 2^(floor(log2 amax) - 2) (2 = the largest E2M1 exponent), elements v / X rounded to the E2M1
# grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} (with sign) nearest-even, saturating at +-6.  Code: sign bit 3,
# magnitude index 0..7 in bits 0-2 (E2M1: 2 exponent bits, 1 mantissa bit).  Two codes per byte,
# element 2j in the low nibble, 2j+1 in the high nibble.
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round_index(q) -> np.ndarray:
    """Magnitude index (0..7) of the E2M1 value nearest |q|, ties to the even mantissa, saturating."""
    a = np.minimum(np.abs(np.asarray(q, np.float64)), 6.0)
    # the grid's quantum: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.rint(a / quantum) * quantum                       # halves to even multiples of the quantum
    r = np.minimum(r, 6.0)
    return np.searchsorted(E2M1_GRID, r).astype(np.int64)


def mx_quantize_e2m1(w, block: int = 32):
    """w [R, K] (K a multiple of 32) -> (codes uint8 [R, K/2], scales uint8 [R, K/32])."""
    w = np.asarray(w, np.float64)
    R, K = w.shape
    b = w.reshape(R, K // block, block)
    amax = np.abs(b).max(axis=-1)
    fl = np.floor(np.log2(np.where(amax > 0, amax, 1.0)))
    shared = np.where(amax > 0, np.clip(fl - 2.0, -127.0, 127.0), -127.0)
    q = b / np.exp2(shared)[..., None]
    idx = e2m1_round_index(q)
    sign = (np.signbit(q) & (idx > 0)).astype(np.int64)
    code = (sign << 3 | idx).reshape(R, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, (shared + 127.0).astype(np.uint8)


def mx_dequantize_e2m1(codes, scales, block: int = 32) -> np.ndarray:
    """codes [R, K/2], scales [R, K/32] -> the float64 weights they encode."""
    codes = np.asarray(codes, np.uint8).astype(np.int64)
    R, K2 = codes.shape
    c = np.empty((R, 2 * K2), np.int64)
    c[:, 0::2] = codes & 0xF
    c[:, 1::2] = codes >> 4
    v = np.where(c & 8, -1.0, 1.0) * E2M1_GRID[c & 7]
    x = np.exp2(np.asarray(scales, np.float64) - 127.0).repeat(block, axis=1)
    return v * x


def mxfp4_weights(w) -> np.ndarray:
    """The float64 weights an MXFP4 checkpoint holds for w [..., K] (bf16 bits or floats): w quantised
    block by block along its last axis and decoded again."""
    w = np.asarray(w)
    if w.dtype == np.uint16:
        w = (w.astype(np.uint32) << 16).view(np.float32)
    K = w.shape[-1]
    codes, scales = mx_quantize_e2m1(np.asarray(w, np.float64).reshape(-1, K))
    return mx_dequantize_e2m1(codes, scales).reshape(w.shape)
