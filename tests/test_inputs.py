"""The seeded input generator: Philox known-answer vectors, distributions, workload shapes."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle


def test_philox_known_answer_vectors():
    # Known-answer vectors of Philox4x32-10 published with the Random123 library
    assert mi.philox4x32_10([0, 0, 0, 0], [0, 0]).tolist() == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert mi.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2).tolist() == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert mi.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]).tolist() == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_normal_moments_and_determinism():
    z = mi.normal_f32(0, 1, (1 << 20,))
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert (mi.normal_f32(0, 1, (1000,)) == z[:1000]).all()
    w = mi.bf16_bits_to_f32(mi.normal_bf16(0, 2, (1 << 18,), 0.0, 0.02))
    assert abs(w.std() - 0.02) < 2e-4


def test_bf16_conversions_round_trip():
    f = np.float32([1.0, -2.5, 3.140625, 1.00390625, 1.01171875])
    b = mi.f32_to_bf16_bits(f)
    # 1.00390625 is halfway between 1 and 1+2^-7: ties to even -> 1.0; 1.01171875 -> 1.015625
    assert mi.bf16_bits_to_f32(b).tolist() == [1.0, -2.5, 3.140625, 1.0, 1.015625]


def test_logits_on_grid():
    cfg = mi.CONFIGS["qwen3_decode"]
    inp = mi.generate(cfg, weights=False)
    assert inp.logits.shape == (64, 128) and inp.logits.dtype == np.float32
    assert (inp.logits * 256 == np.round(inp.logits * 256)).all()


@pytest.mark.parametrize("name", ["hy3_prefill", "long_prefill"])
def test_zipf_workloads_have_hot_and_empty_experts(name):
    cfg = mi.CONFIGS[name]
    inp = mi.generate(cfg, weights=False)
    _, idx = oracle.gating_topk(inp.logits, cfg.k, cfg.gate, inp.bias, cfg.routed_scaling_factor)
    c = np.bincount(idx.ravel(), minlength=cfg.E)
    ratio = c.max() / c.mean()
    assert 5.0 <= ratio <= 10.0, ratio
    assert (c == 0).sum() >= 1


def test_stream_slices_equal_the_full_stream():
    full = mi.normal_bf16(3, 2, (4099,), 0.0, 0.02)
    for start, n in ((0, 4099), (1, 5), (3, 1), (4, 8), (1001, 2000), (4098, 1)):
        assert (mi.normal_bf16_slice(3, 2, start, (n,), 0.0, 0.02) == full[start:start + n]).all()
    cfg = mi.CONFIGS["tiny"].with_(E=5)
    inp = mi.generate(cfg)
    for e in range(cfg.E):
        w13, w2 = mi.expert_weights(cfg, e)
        assert (w13 == inp.w13[e]).all() and (w2 == inp.w2[e]).all()
