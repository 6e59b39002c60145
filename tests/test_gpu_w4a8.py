"""GPU parity of the W4A8 path -- MXFP8 activations x MXFP4 expert weights on the block-scaled
tensor-core MMA (Qwen3-MoE practice, MoE EP W4A8 section; Hy3 practice 5.2) -- against the oracle,
through the C ABI.

* the one-time weight layout and the MXFP8 row gather: bit-exact against the layout their
  definitions state;
* the down GEMM on MXFP8 rows and MXFP4 weights the oracle quantised: every output within one bf16
  rounding of the float64 product of the decoded operands (the hardware applies both scales);
* the gate/up GEMM: act codes and scales against the oracle quantising its own float64 SwiGLU
  output -- equal except where the fp32 and float64 values straddle a rounding boundary, and
  then one E4M3 step apart;
* the whole W4A8 layer (moe_layer_forward_w4a8) against oracle.moe_layer_forward_w4a8: routing
  bit-exact, y within max-rel 2e-2 and mean-rel 5e-3, with and without a shared expert, several
  token tiles in one expert, I_s != I, and at the full decode and prefill sizes on sampled tokens.
Both GEMM instances are covered: 32 token columns per tile (at most 32 rows per expert on average)
and 112 (more), including ragged tails, 400 and 620 experts.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import assert_close, dev, dev_bf16, host, host_bf16_f64
from oracle.mx import e4m3_decode, mx_quantize_e2m1, mx_quantize_e4m3

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


def _padded_sf(scales):
    """[rows, K/32] E8M0 bytes -> the padded scale rows [rows, K/128, 16] the W4A8 GEMMs read."""
    R, nb = scales.shape
    out = np.zeros((R, nb // 4, 16), np.uint8)
    out[:, :, :4] = scales.reshape(R, nb // 4, 4)
    return out


def _mx8(v):
    """float64 rows -> (codes, padded scale rows, decoded values), quantised by the oracle."""
    codes, scales = mx_quantize_e4m3(v)
    return codes, _padded_sf(scales), oracle.mx_dequantize_e4m3(codes, scales)


def _mx4(w):
    """float weights [E, n_out, K] -> (codes [E,n_out,K/2], scales [E,n_out,K/32], decoded), by the oracle."""
    E, n, K = w.shape
    c, s = mx_quantize_e2m1(w.reshape(-1, K))
    return c.reshape(E, n, K // 2), s.reshape(E, n, K // 32), oracle.mx_dequantize_e2m1(c, s).reshape(E, n, K)


# ---------------------------------------------------------------- layout kernels
@pytest.mark.parametrize("gate_up,E,n_out,K", [(True, 2, 256, 256), (True, 1, 512, 128), (False, 3, 256, 384)])
def test_w4a8_prepack_layout(moe, gate_up, E, n_out, K):
    rng = np.random.default_rng(E + n_out + K)
    codes = rng.integers(0, 256, size=(E, n_out, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 255, size=(E, n_out, K // 32), dtype=np.uint8)
    w = moe.moe_w4a8_prepack(dev(codes), dev(scales), gate_up=gate_up)
    R = np.arange(n_out)
    if gate_up:
        I = n_out // 2
        f = 128 * (R // 256) + 32 * ((R // 32) % 4) + 16 * ((R // 128) % 2) + R % 16
        src = np.where(R % 32 < 16, f, I + f)
    else:
        src = R
    rows = codes[:, src, :].reshape(E * n_out // 256, 256, K // 128, 64)
    want_codes = rows.transpose(0, 2, 1, 3)  # [tile, chunk, row, 64 bytes]
    assert (host(w.codes) == want_codes).all()
    sc = scales[:, src, :].reshape(E * n_out, K // 32)
    want_sf = np.zeros((E * n_out // 256, K // 128, 2, 512), np.uint8)
    for row in range(E * n_out):
        t, r = divmod(row, 256)
        half, r = divmod(r, 128)
        for b in range(K // 32):
            want_sf[t, b // 4, half, (r % 32) * 16 + (r // 32) * 4 + b % 4] = sc[row, b]
    assert (host(w.sf) == want_sf).all()


def test_gather_rows_mx(moe):
    rng = np.random.default_rng(3)
    T, k, H = 37, 3, 256
    xc = rng.integers(0, 256, size=(T, H), dtype=np.uint8)
    xs = rng.integers(0, 255, size=(T, H // 32), dtype=np.uint8)
    sp = rng.permutation(T * k).astype(np.int32)
    codes, sf = moe.moe_gather_rows_mx(dev(xc), dev(xs), dev(sp), k)
    assert (host(codes) == xc[sp // k]).all()
    assert (host(sf) == _padded_sf(xs)[sp // k]).all()
    _, sf_tok = moe.moe_gather_rows_mx(dev(xc), dev(xs))
    assert (host(sf_tok) == _padded_sf(xs)).all()
    # a pair index outside [0, T*k) is skipped and reported
    torch = _torch()
    bad = sp.copy()
    bad[5] = T * k
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    moe.moe_gather_rows_mx(dev(xc), dev(xs), dev(bad), k, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK


# ---------------------------------------------------------------- the two GEMMs
GEMM_CASES = [
    # (rows per expert, H, I): empty experts, 1 row, a full 32-row tile, 33 and 70 rows (several token
    # tiles in one expert), K of one and of several 128-K stages
    ([3, 0, 1, 32, 33, 0, 70, 5], 256, 128),
    ([1] * 12 + [0] * 4, 512, 256),
    ([40, 2, 0, 9], 1024, 384),          # I = 384: a window of 3 chunks in the down GEMM
    ([2, 0, 65, 7], 768, 640),           # H = 768: 6 chunks (a full and a partial window); I = 640: 5
    # more than 32 rows per expert on average: the 112-column instance (tiles of 112 token rows, MMA N
    # the tile's rows rounded up to 16), ragged tails of 1, 52 and 76 rows, exact multiples of 112
    ([300, 0, 1, 111, 112, 113, 224, 500], 256, 128),
    ([200, 150, 0, 90], 768, 640),       # 6 and 5 chunks: full and partial 2-chunk windows
    ([120] * 6 + [0] * 2, 512, 256),
    # 400 experts: three token windows for the gate/up GEMM, two for the down GEMM (its routing weights
    # take the room); 620: two for both
    ([34] * 400, 256, 128),
    ([34] * 620, 256, 128),
]


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_down_gemm_w4a8_parity(moe, counts, H, I):
    """y_perm = w * (act . w2^T) on MXFP8 act and MXFP4 w2 the oracle quantised: within one bf16 rounding
    of the float64 product of the decoded operands."""
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    rng = np.random.default_rng(M + H + I)
    a = rng.normal(size=(M, I)) * np.exp2(rng.integers(-3, 4, size=(M, 1)))   # rows of different scales
    ac, asf, adq = _mx8(a)
    w2 = oracle.bf16_to_f64(mi.normal_bf16(M + H, 3, (E, H, I), 0.0, 0.02))
    wc, ws_, wdq = _mx4(w2)
    topk_w = (np.abs(rng.normal(size=(M,))) + 0.1).astype(np.float32)
    sp = rng.permutation(M).astype(np.int32)
    ref = oracle.grouped_gemm(adq, wdq, off, topk_w[sp])
    w = moe.moe_w4a8_prepack(dev(wc), dev(ws_), gate_up=False)
    out = moe.moe_grouped_gemm_w4a8(dev(ac), dev(asf), w, dev(off), dev(topk_w), dev(sp))
    got = host_bf16_f64(out)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max()
    assert (np.abs(got - ref) <= bound).all(), np.abs(got - ref).max()
    assert_close(got, ref, "y_perm (W4A8)")


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_gate_up_gemm_w4a8_parity(moe, counts, H, I):
    """act (MXFP8) against the oracle's float64 SwiGLU of the decoded operands, quantised by the oracle."""
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    x = oracle.bf16_to_f64(mi.normal_bf16(M + I, 1, (M, H)))
    xc, xsf, xdq = _mx8(x)
    w13 = oracle.bf16_to_f64(mi.normal_bf16(M + I, 2, (E, 2 * I, H), 0.0, 0.02))
    wc, wsc, wdq = _mx4(w13)
    act_ref = oracle.grouped_gemm_swiglu(xdq, wdq, off)
    c_ref, s_ref = mx_quantize_e4m3(act_ref)
    w = moe.moe_w4a8_prepack(dev(wc), dev(wsc), gate_up=True)
    act, act_sf = moe.moe_grouped_gemm_swiglu_w4a8(dev(xc), dev(xsf), w, dev(off))
    codes = host(act)
    sf = host(act_sf)
    assert (sf[:, :, 4:] == 0).all()
    scales = sf[:, :, :4].reshape(M, I // 32)
    # scales: equal except for a block whose float64 maximum lies within 1e-5 of a power of two
    blk = np.abs(act_ref).reshape(M, I // 32, 32).max(axis=-1)
    s_diff = scales != s_ref
    if s_diff.any():
        fr = np.log2(blk[s_diff])
        assert (np.abs(fr - np.rint(fr)) <= 1e-5).all()
    same = np.repeat(~s_diff, 32, axis=1)
    mag, mag_ref = codes & 0x7F, c_ref & 0x7F
    differ = (codes != c_ref) & ~((mag == 0) & (mag_ref == 0)) & same
    n = int(differ.sum())
    assert n <= max(4, 2e-3 * codes.size), f"{n} of {codes.size} act codes differ"
    if n:
        assert (np.abs(mag[differ].astype(int) - mag_ref[differ].astype(int)) == 1).all()
        X = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=1)
        v = np.abs(act_ref[differ]) / X[differ]
        mid = (np.abs(e4m3_decode(codes[differ])) + np.abs(e4m3_decode(c_ref[differ]))) / 2
        assert (np.abs(v - mid) <= 1e-3 * v + 1e-3).all(), "a differing code is not at a rounding boundary"
    print(f"W4A8 act codes: {n} of {codes.size} differ from the float64 oracle's, each at a rounding boundary")


def test_w4a8_gemm_rejects_inconsistent_offsets(moe):
    torch = _torch()
    off = np.array([0, 5, 3, 8], np.int32)
    xc, xsf, _ = _mx8(np.ones((8, 256)))
    wc, wsc, _ = _mx4(np.ones((3, 256, 256)) * 0.01)
    w = moe.moe_w4a8_prepack(dev(wc), dev(wsc), gate_up=True)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    act = torch.full((8, 128), 7, dtype=torch.uint8, device="cuda")
    moe.moe_grouped_gemm_swiglu_w4a8(dev(xc), dev(xsf), w, dev(off), act=act, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert (act == 7).all()


# ---------------------------------------------------------------- the whole W4A8 layer
def _run_layer(moe, cfg, inp, tokens=None):
    torch = _torch()
    xc, xs = mx_quantize_e4m3(oracle.bf16_to_f64(inp.x))
    d16 = dev_bf16
    q = lambda w, gu: moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(d16(w)), gate_up=gu)
    w13, w2 = q(inp.w13, True), q(inp.w2, False)
    w13_s = q(inp.w13_s, True) if cfg.n_shared else None
    w2_s = q(inp.w2_s, False) if cfg.n_shared else None
    layer = moe.W4a8Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                          cfg.n_shared, cfg.I_s)
    y = layer.forward(dev(xc), dev(xs), dev(inp.logits), w13, w2, dev(inp.bias) if inp.bias is not None else None,
                      w13_s, w2_s)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    ref = oracle.moe_layer_forward_w4a8(xc, xs, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                        cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s, tokens=tokens)
    assert (host(layer.topk_idx) == ref["topk_idx"]).all(), "routing differs"
    assert (host(layer.counts) == ref["counts"]).all()
    got = host_bf16_f64(y)[ref["tokens"]]
    return got, ref


LAYER_CASES = [
    mi.CONFIGS["tiny"],
    mi.CONFIGS["hy3_decode"].with_(T=8, H=256, E=16, k=4, I=128, I_s=128),        # + shared expert
    mi.CONFIGS["hy3_decode"].with_(T=6, H=512, E=8, k=2, I=256, I_s=128),         # I_s != I
    mi.CONFIGS["qwen3_decode"].with_(T=300, H=256, E=4, k=2, I=128),              # several token tiles per expert
    mi.CONFIGS["qwen3_decode"].with_(T=1, H=512, E=32, k=8, I=256),
    # the documented limits: E = 1024 experts, k = 32
    mi.CONFIGS["tiny"].with_(T=64, H=256, E=1024, k=32, I=128),
    # gating and routing in one kernel up to T*k = 4096, four kernels above
    mi.CONFIGS["qwen3_decode"].with_(T=512, H=256, I=128),
    mi.CONFIGS["qwen3_decode"].with_(T=513, H=256, I=128),
    # a few rows per routed expert, but a shared expert over 40 tokens: the 112-column instance
    mi.CONFIGS["hy3_decode"].with_(T=40, H=256, E=64, k=4, I=128, I_s=128),
    # prefill-like: the 112-column instance, with and without the shared expert
    mi.CONFIGS["hy3_prefill"].with_(T=300, H=256, E=16, k=4, I=128, I_s=256, zipf_beta=0.3, n_dead=2),
    mi.CONFIGS["long_prefill"].with_(T=1000, H=512, E=16, k=4, I=256, zipf_beta=0.5, n_dead=3),
]


@pytest.mark.parametrize("cfg", LAYER_CASES, ids=lambda c: f"{c.name}-T{c.T}-E{c.E}-I{c.I}-s{c.n_shared}")
def test_w4a8_layer_parity(moe, cfg):
    got, ref = _run_layer(moe, cfg, mi.generate(cfg))
    assert_close(got, ref["y"], f"W4A8 layer {cfg.name}")


@pytest.mark.parametrize("name", ["qwen3_decode", "hy3_decode", "hy3_prefill", "long_prefill"])
def test_w4a8_layer_full_size_sampled_tokens(moe, name):
    """The full sizes (decode: the 32-column GEMMs; prefill: the 112-column ones), launched as the bench
    launches them: routing of every token bit-exact, y of four tokens (first, last and two between)
    against the oracle, which quantises each needed expert."""
    cfg = mi.CONFIGS[name]
    tokens = np.array([0, cfg.T // 3, 2 * cfg.T // 3, cfg.T - 1])
    got, ref = _run_layer(moe, cfg, mi.generate(cfg), tokens)
    assert_close(got, ref["y"], f"W4A8 layer {name}")


def test_w4a8_layer_all_tokens_on_one_expert(moe):
    """One expert takes every token (300 rows: three 112-row token tiles of one expert, the last one
    ragged), the rest share the other slot."""
    cfg = mi.CONFIGS["tiny"].with_(T=300, E=8, k=2)
    inp = mi.generate(cfg)
    inp.logits[:, 5] = 50.0  # every token picks expert 5 first
    got, ref = _run_layer(moe, cfg, inp)
    assert ref["counts"][5] == cfg.T
    assert_close(got, ref["y"], "W4A8 layer, one expert")


def test_w4a8_layer_empty_batch(moe):
    """T = 0: nothing to compute, no launch, MOE_OK."""
    torch = _torch()
    cfg = mi.CONFIGS["tiny"]
    layer = moe.W4a8Layer(0, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate)
    assert layer.launches == 0
    inp = mi.generate(cfg)
    q = lambda w, gu: moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(dev_bf16(w)), gate_up=gu)
    xc = torch.empty((0, cfg.H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((0, cfg.H // 32), dtype=torch.uint8, device="cuda")
    lg = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    y = layer.forward(xc, xs, lg, q(inp.w13, True), q(inp.w2, False))
    torch.cuda.synchronize()
    assert y.shape == (0, cfg.H)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
