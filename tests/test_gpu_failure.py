"""Failure detection on the GPU without a fault: a bounded wait is made to run out (the gate/up GEMM's
gather flags are never set, moe_debug_set), the kernel records MOE_ERR_TIMEOUT in the workspace
status and returns; the host reads the status, clears it, and the next forward on the same context
is correct.  No trap, no assert, no endless loop."""
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


def test_gather_wait_timeout_is_reported_and_recoverable(moe):
    import time
    import torch
    # >= 256 pairs per expert: the gate/up GEMM gathers its rows in-kernel and waits on their flags
    cfg = mi.CONFIGS["long_prefill"].with_(T=1024, H=256, E=8, k=4, I=128, zipf_beta=0.2, n_dead=0)
    inp = mi.generate(cfg)
    t = dict(x=dev_bf16(inp.x), logits=dev(inp.logits), w13=moe.moe_prepack_w13(dev_bf16(inp.w13)),
             w2=dev_bf16(inp.w2))
    layer = moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate)
    assert moe.moe_layer_kernel_launches(layer.desc) == 7  # the in-kernel gather is taken
    L = moe.lib()
    try:
        assert L.moe_debug_set(1, 50_000_000) == moe.MOE_OK   # 50 ms
        assert L.moe_debug_set(2, 1) == moe.MOE_OK
        t0 = time.time()
        layer.forward(**t)
        st = moe.moe_get_device_status(layer.ws)               # synchronises
        dt = time.time() - t0
    finally:
        L.moe_debug_set(2, 0)
        L.moe_debug_set(1, 0)
    assert st == moe.MOE_ERR_TIMEOUT
    assert dt < 10.0
    # the context is usable: clear the sticky word, run again, check the result
    assert L.moe_workspace_init(layer.ws.data_ptr(), layer.ws.numel(), None) == moe.MOE_OK
    layer.forward(**t)
    assert moe.moe_get_device_status(layer.ws) == moe.MOE_OK
    ref = oracle.moe_layer_forward(inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2)
    torch.cuda.synchronize()
    assert (host(layer.topk_idx) == ref["topk_idx"]).all()
    assert_close(host_bf16_f64(layer.y), ref["y"], "y after recovery")
