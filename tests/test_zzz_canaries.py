"""Guard regions around every output buffer (the stand-in for a memory checker, which is not run on
this hardware): each output of each C entry point is the middle of a larger buffer whose 4 KB before
and after hold a known pattern; after the call both guards must be unchanged, and the outputs must
still be right.  Named to run last."""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import assert_close, dev, dev_bf16, host, host_bf16_f64

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_fwd_gb300 import build
    build.build()
    import moe_expert_layer_fwd_gb300 as m
    return m


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD_BYTES of `fill` on each side."""

    def __init__(self, shape, dtype, fill):
        import torch
        self.n = int(np.prod(shape)) if len(shape) else 1
        item = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // item
        self.buf = torch.full((self.n + 2 * self.g,), fill, dtype=dtype, device="cuda")
        self.ref = self.buf[: self.g].clone()
        self.t = self.buf[self.g: self.g + self.n].view(*shape)

    def intact(self) -> bool:
        import torch
        torch.cuda.synchronize()
        as_int = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[self.buf.element_size()]
        head = self.buf[: self.g].view(as_int)
        tail = self.buf[self.g + self.n:].view(as_int)
        ref = self.ref.view(as_int)
        return bool((head == ref).all()) and bool((tail == ref).all())


def test_guards_around_every_output(moe):
    import torch
    cfg = mi.CONFIGS["qwen3_decode"].with_(T=24, H=512, E=16, I=256)
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    P = T * k
    inp = mi.generate(cfg)
    ref = oracle.moe_layer_forward(inp.x, inp.logits, k, cfg.gate, inp.w13, inp.w2)

    # a1
    tw = Guarded((T, k), torch.float32, 1234.5)
    ti = Guarded((T, k), torch.int32, -7)
    moe.moe_gating_topk(dev(inp.logits), k, cfg.gate, None, 1.0, cfg.eps, topk_w=tw.t, topk_idx=ti.t)
    assert tw.intact() and ti.intact()
    assert (host(ti.t) == ref["topk_idx"]).all()

    # a2 (with the row gather)
    outs = dict(counts=Guarded((E,), torch.int32, -7), offsets=Guarded((E + 1,), torch.int32, -7),
                sorted_pair=Guarded((P,), torch.int32, -7), pair_pos=Guarded((P,), torch.int32, -7),
                x_exp=Guarded((P, H), torch.bfloat16, 7.0))
    x = dev_bf16(inp.x)
    moe.moe_init_routing(ti.t, E, x=x, out={n: g.t for n, g in outs.items()})
    assert all(g.intact() for g in outs.values())
    assert (host(outs["sorted_pair"].t) == ref["sorted_pair"]).all()
    off, sp, pp = outs["offsets"].t, outs["sorted_pair"].t, outs["pair_pos"].t

    # a3, a4, a6
    act = Guarded((P, I), torch.bfloat16, 7.0)
    w13p = moe.moe_prepack_w13(dev_bf16(inp.w13))
    moe.moe_grouped_gemm_swiglu(outs["x_exp"].t, w13p, off, act=act.t)
    assert act.intact()
    # the same GEMM gathering its rows from x: writes only act, and the same bits
    act_g = Guarded((P, I), torch.bfloat16, 7.0)
    moe.moe_grouped_gemm_swiglu(x, w13p, off, act=act_g.t, row_src=sp, k=k)
    assert act_g.intact()
    assert torch.equal(act_g.t.view(torch.int16), act.t.view(torch.int16))
    yp = Guarded((P, H), torch.bfloat16, 7.0)
    moe.moe_grouped_gemm(act.t, dev_bf16(inp.w2), off, tw.t, sp, out=yp.t)
    assert yp.intact()
    y = Guarded((T, H), torch.bfloat16, 7.0)
    moe.moe_finalize_routing(yp.t, pp, T, k, y=y.t)
    assert y.intact()
    assert_close(host_bf16_f64(y.t), ref["y"], "y (bf16 path)")

    # the 4-bit path: row gather, both GEMMs
    x16 = Guarded((P, H), torch.float16, 7.0)
    moe.moe_gather_rows_f16(x, sp, k, out=x16.t)
    assert x16.intact()
    w13q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w13)), gate_up=True)
    w2q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(dev_bf16(inp.w2)), gate_up=False)
    a16 = Guarded((P, I), torch.float16, 7.0)
    moe.moe_grouped_gemm_swiglu_mxfp4(x16.t, w13q, off, act=a16.t)
    assert a16.intact()
    yp4 = Guarded((P, H), torch.bfloat16, 7.0)
    moe.moe_grouped_gemm_mxfp4(a16.t, w2q, off, tw.t, sp, out=yp4.t)
    assert yp4.intact()
    y4 = Guarded((T, H), torch.bfloat16, 7.0)
    moe.moe_finalize_routing(yp4.t, pp, T, k, y=y4.t)
    assert y4.intact()
    ref4 = oracle.moe_layer_forward_tokens_mxfp4(np.arange(T), inp.x, inp.logits, k, cfg.gate, inp.w13, inp.w2)
    assert_close(host_bf16_f64(y4.t), ref4["y"], "y (4-bit path)")


@pytest.mark.parametrize("T,E,k", [(24, 16, 8), (300, 8, 2)], ids=["32-column", "112-column"])
def test_guards_around_w4a8_outputs(moe, T, E, k):
    """The W4A8 outputs (MXFP8 row gather, gate/up codes and scales, down rows) inside guard regions,
    on the decode (32-column) and prefill (112-column) GEMM instances: guards unchanged, and each
    output bit-equal to the same call into a plain buffer."""
    import torch
    from oracle.mx import mx_quantize_e4m3
    cfg = mi.CONFIGS["qwen3_decode"].with_(T=T, H=512, E=E, k=k, I=256)
    H, I, P = cfg.H, cfg.I, T * k
    inp = mi.generate(cfg)
    _, idx = oracle.gating_topk(inp.logits, k, cfg.gate)
    counts, off, sp, _ = oracle.init_routing(idx, E)
    assert (P > 32 * E) == (T == 300)  # which instance the GEMMs take
    xc, xs = mx_quantize_e4m3(oracle.bf16_to_f64(inp.x))
    q = lambda w, gu: moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(dev_bf16(w)), gate_up=gu)
    w13, w2 = q(inp.w13, True), q(inp.w2, False)
    d_off, d_sp = dev(off), dev(sp)
    topk_w = torch.rand(P, dtype=torch.float32, device="cuda") + 0.1

    gc, gs = Guarded((P, H), torch.uint8, 0x5A), Guarded((P, H // 128, 16), torch.uint8, 0x5A)
    moe.moe_gather_rows_mx(dev(xc), dev(xs), d_sp, k, out_codes=gc.t, out_sf=gs.t)
    assert gc.intact() and gs.intact()
    pc, ps = moe.moe_gather_rows_mx(dev(xc), dev(xs), d_sp, k)
    assert torch.equal(gc.t, pc) and torch.equal(gs.t, ps)

    ac, asf = Guarded((P, I), torch.uint8, 0x5A), Guarded((P, I // 128, 16), torch.uint8, 0x5A)
    moe.moe_grouped_gemm_swiglu_w4a8(gc.t, gs.t, w13, d_off, act=ac.t, act_sf=asf.t)
    assert ac.intact() and asf.intact()
    pa, pas = moe.moe_grouped_gemm_swiglu_w4a8(pc, ps, w13, d_off)
    assert torch.equal(ac.t, pa) and torch.equal(asf.t, pas)

    yp = Guarded((P, H), torch.bfloat16, 7.0)
    moe.moe_grouped_gemm_w4a8(ac.t, asf.t, w2, d_off, topk_w, d_sp, out=yp.t)
    assert yp.intact()
    py = moe.moe_grouped_gemm_w4a8(pa, pas, w2, d_off, topk_w, d_sp)
    assert torch.equal(yp.t.view(torch.int16), py.view(torch.int16))
