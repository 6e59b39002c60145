"""The workspace-free init-routing entry point against the regular one, through the C ABI.

moe_init_routing_static_scratch exists for callers that cannot allocate device
memory (allocator callbacks, fully pre-reserved memory, latency-critical host
threads): its scratch is a fixed device array inside the library.  This file
is collected last so that a failure here never hides the rest of the suite; it
must pass both alone in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    from moe_expert_layer_fwd_gb300 import build
    build.build()
    import moe_expert_layer_fwd_gb300 as moe
    return moe, torch


def _routing_case(seed, T, E, k, H):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(E, 0.3))
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    x = rng.integers(-2 ** 15, 2 ** 15, size=(T, H), dtype=np.int16)
    return idx, x


def _outputs(torch, T, E, k, H, fill):
    P = T * k
    return dict(counts=torch.full((E,), fill, dtype=torch.int32, device="cuda"),
                offsets=torch.full((E + 1,), fill, dtype=torch.int32, device="cuda"),
                sorted_pair=torch.full((P,), fill, dtype=torch.int32, device="cuda"),
                pair_pos=torch.full((P,), fill, dtype=torch.int32, device="cuda"),
                x_exp=torch.full((P, H), fill, dtype=torch.int16, device="cuda"))


def _call_static(moe, torch, idx_d, x_d, T, E, k, H, o):
    stream = torch.cuda.current_stream().cuda_stream
    return moe.lib().moe_init_routing_static_scratch(
        idx_d.data_ptr(), T, E, k, x_d.data_ptr(), H, o["x_exp"].data_ptr(), o["counts"].data_ptr(),
        o["offsets"].data_ptr(), o["sorted_pair"].data_ptr(), o["pair_pos"].data_ptr(), stream)


def _call_regular(moe, torch, idx_d, x_d, T, E, k, H, o):
    stream = torch.cuda.current_stream().cuda_stream
    need = moe.lib().moe_init_routing_workspace_size(T, E, k)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st = moe.lib().moe_init_routing(
        idx_d.data_ptr(), T, E, k, x_d.data_ptr(), H, o["x_exp"].data_ptr(), o["counts"].data_ptr(),
        o["offsets"].data_ptr(), o["sorted_pair"].data_ptr(), o["pair_pos"].data_ptr(), ws.data_ptr(), need, stream)
    return st


def test_static_scratch_matches_workspace_routing_twice_in_a_row(env):
    moe, torch = env
    # two different problems back to back: the second call runs on scratch the first one left behind
    for seed, (T, E, k, H) in enumerate([(4096, 192, 8, 64), (300, 37, 3, 128)]):
        idx, x = _routing_case(seed, T, E, k, H)
        idx_d = torch.from_numpy(idx).cuda()
        x_d = torch.from_numpy(x).cuda()
        ref = _outputs(torch, T, E, k, H, -7)
        got = _outputs(torch, T, E, k, H, 5)
        assert _call_regular(moe, torch, idx_d, x_d, T, E, k, H, ref) == moe.MOE_OK
        assert _call_static(moe, torch, idx_d, x_d, T, E, k, H, got) == moe.MOE_OK
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "sorted_pair", "pair_pos", "x_exp"):
            assert torch.equal(got[name], ref[name]), f"call {seed}: {name} differs"


def test_static_scratch_rejects_problems_beyond_its_limit(env):
    moe, torch = env
    # E = 1024 needs 2 * n_chunks * 1024 * 4 bytes: over 1 MiB once T*k > 65536
    T, E, k = 8200, 1024, 16
    stream = torch.cuda.current_stream().cuda_stream
    d = torch.zeros(16, dtype=torch.int32, device="cuda").data_ptr()
    st = moe.lib().moe_init_routing_static_scratch(d, T, E, k, None, 0, None, d, d, d, d, stream)
    assert st == moe.MOE_ERR_UNSUPPORTED
