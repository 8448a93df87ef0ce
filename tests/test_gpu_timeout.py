"""Failure detection on the GPU: a bounded wait that runs out.

The fault-injection build of the library (libmoe_fault.so: the same sources compiled with
MOE_FAULT_INJECTION, bounded waits limited to 50 ms) exports one test switch,
moe_test_drop_gemm_loads.  With it on, the grouped expert GEMM's producers issue no TMA
loads, so the bytes its MMA warp waits for never arrive: no memory is touched, and every
wait of the kernel gives up at its limit.  The test checks that the layer call returns,
that the device status word then reads MOE_ERR_TIMEOUT, and that the same context runs a
normal layer call correctly right afterwards (the status word is clear again).
"""
from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest

from oracle import moe_oracle as orc
from routing_expert_ffn_gb300 import inputs as gen
from tests import harness

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def moe_fault():
    from routing_expert_ffn_gb300 import build, moe
    build.build(fault=True)
    L = moe.load_library(build.LIB_FAULT)
    L.moe_test_drop_gemm_loads.restype = ctypes.c_int
    L.moe_test_drop_gemm_loads.argtypes = [ctypes.c_int]
    saved = moe._lib
    moe._lib = L  # the binding's calls go to the fault-injection build in this module
    yield moe, L
    L.moe_test_drop_gemm_loads(0)
    moe._lib = saved


def test_gemm_wait_times_out_and_context_recovers(moe_fault):
    moe, L = moe_fault
    cfg, inp = harness.workload("dsv2_lite", T=600)
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp)
    layer = moe.Layer(C, w)
    assert moe.get_device_status() == 0
    assert L.moe_test_drop_gemm_loads(1) == 0
    t0 = time.perf_counter()
    layer(x, r)  # returns at once: the launches are asynchronous
    st = moe.get_device_status()  # synchronises: the GEMMs' waits give up after 50 ms each
    elapsed = time.perf_counter() - t0
    assert st == MOE_ERR_TIMEOUT
    assert elapsed < 30.0
    assert L.moe_test_drop_gemm_loads(0) == 0
    out = layer(x, r)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                            inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                            residual_mode=cfg.residual, residual=inp["residual"])
    got = out.float().cpu().numpy()
    assert harness.max_rel_err(got, ref["out"]) <= harness.tolerance(cfg)
