"""moe_dispatch_static_scratch: the dispatch entry point that allocates nothing.

Some callers cannot allocate device memory (their device memory is entirely
pre-reserved by their own allocator, or they must not call cudaMalloc because
it synchronises the device).  This entry point takes no workspace; its scratch
is a fixed 1 MiB array inside libmoe.so.  The test checks, through the C ABI,
that two calls in a row give exactly the outputs of moe_dispatch (integer
work and row copies, so bit for bit), and that a shape needing more scratch
than the array holds is refused before anything is launched.
This file is named to be collected last.
"""
from __future__ import annotations

import ctypes

import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def moe():
    from routing_expert_ffn_gb300 import build
    build.build()
    from routing_expert_ffn_gb300 import moe as m
    m.lib()
    return m


def _inputs(moe, T, d, E, k, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    C = moe.Config(T=T, d=d, E=E, k=k, H=128, dtype="bf16", gating="softmax_topk")
    x = torch.randn(T, d, device="cuda", generator=g).bfloat16()
    W_r = torch.randn(d, E, device="cuda", generator=g) / d ** 0.5
    _, idx, _ = moe.route(C, x, W_r)
    return C, x, idx


@pytest.mark.gpu
@pytest.mark.parametrize("T,d,E,k", [(4096, 2048, 64, 6), (8192, 2048, 128, 8), (777, 256, 8, 2)])
def test_static_scratch_dispatch_matches_workspace_dispatch(moe, T, d, E, k):
    C, x, idx = _inputs(moe, T, d, E, k, seed=T + E)
    ref = moe.dispatch(C, x, idx)
    for call in range(2):  # the second call runs on the scratch the first one left behind
        got = moe.dispatch_static_scratch(C, x, idx)
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "perm", "slot_of", "x_perm"):
            assert torch.equal(got[key][: ref[key].shape[0]], ref[key]), (call, key)
    assert moe.get_device_status() == 0


@pytest.mark.gpu
def test_static_scratch_dispatch_skips_out_of_range_expert(moe):
    """One routed pair names an expert outside [0, E): both entry points give it no slot
    (slot_of -1), leave it out of every bucket, and flag it in the device status word."""
    C, x, idx = _inputs(moe, 1000, 256, 8, 2, seed=11)
    moe.get_device_status()  # start from a clear status word
    bad = idx.clone()
    bad[517, 1] = C.E + 3
    ref = moe.dispatch(C, x, bad)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 6  # MOE_ERR_DEVICE_INDEX
    for call in range(2):
        got = moe.dispatch_static_scratch(C, x, bad)
        torch.cuda.synchronize()
        assert moe.get_device_status() == 6, call
        n = int(ref["offsets"][-1].item())
        assert n == C.T * C.k - 1
        assert int(got["slot_of"][517, 1].item()) == -1
        for key in ("counts", "offsets", "slot_of"):
            assert torch.equal(got[key], ref[key]), (call, key)
        assert torch.equal(got["perm"][:n], ref["perm"][:n]), call
        assert torch.equal(got["x_perm"][:n], ref["x_perm"][:n]), call


@pytest.mark.gpu
def test_static_scratch_dispatch_refuses_oversized_shapes(moe):
    # 8 * E * ceil(T / 128) bytes of scratch; E = 256, T = 70000 needs more than 1 MiB
    C = moe.Config(T=70000, d=256, E=256, k=2, H=128, dtype="bf16")
    fake = 0x10000
    r = moe.lib().moe_dispatch_static_scratch(ctypes.byref(C.c()), fake, fake, fake, fake, fake,
                                               fake, fake, None)
    assert r == 3
