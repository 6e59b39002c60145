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


# (T, E, k, H): the 1 MiB limit exactly (E = 1024 at T*k = 65536, and E = 512 at T*k = 131072),
# a single token, and no row gather (H = 0)
ORACLE_CASES = [(8192, 1024, 8, 64), (16384, 512, 8, 0), (1, 16, 4, 128), (777, 40, 5, 0)]


@pytest.mark.parametrize("T,E,k,H", ORACLE_CASES)
def test_static_scratch_matches_the_oracle(env, T, E, k, H):
    """Counts, offsets, both permutations and the gathered rows bit for bit against the oracle's
    counting sort and row expansion."""
    moe, torch = env
    import oracle
    idx, x = _routing_case(T + E, T, E, k, max(H, 64))
    counts, offsets, sp, pp = oracle.init_routing(idx, E)
    idx_d = torch.from_numpy(idx).cuda()
    got = _outputs(torch, T, E, k, max(H, 64), 3)
    stream = torch.cuda.current_stream().cuda_stream
    x_d = torch.from_numpy(x).cuda() if H else None
    st = moe.lib().moe_init_routing_static_scratch(
        idx_d.data_ptr(), T, E, k, x_d.data_ptr() if H else None, H, got["x_exp"].data_ptr() if H else None,
        got["counts"].data_ptr(), got["offsets"].data_ptr(), got["sorted_pair"].data_ptr(),
        got["pair_pos"].data_ptr(), stream)
    assert st == moe.MOE_OK
    torch.cuda.synchronize()
    assert (got["counts"].cpu().numpy() == counts).all()
    assert (got["offsets"].cpu().numpy() == offsets).all()
    assert (got["sorted_pair"].cpu().numpy() == sp).all()
    assert (got["pair_pos"].cpu().numpy() == pp).all()
    if H:
        xe = got["x_exp"].cpu().numpy().view(np.uint16)
        assert (xe == oracle.expand_rows(x.view(np.uint16), sp, k)).all()
    else:
        assert (got["x_exp"] == 3).all()  # no gather asked for: untouched


@pytest.mark.parametrize("T,E,k", [(8200, 1024, 16), (65537, 1024, 1)])
def test_static_scratch_rejects_problems_beyond_its_limit(env, T, E, k):
    moe, torch = env
    # E = 1024 needs 2 * n_chunks * 1024 * 4 bytes: over 1 MiB once T*k > 65536 (65537 is the first)
    stream = torch.cuda.current_stream().cuda_stream
    d = torch.zeros(16, dtype=torch.int32, device="cuda").data_ptr()
    st = moe.lib().moe_init_routing_static_scratch(d, T, E, k, None, 0, None, d, d, d, d, stream)
    assert st == moe.MOE_ERR_UNSUPPORTED
