"""C-ABI host logic, without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything."""
from __future__ import annotations

import ctypes
import math
import os
import re

import pytest

from routing_expert_ffn_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    from routing_expert_ffn_gb300 import moe
    return moe


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declarations_are_exported(L):
    lib = L.lib()
    names = _declared_functions()
    assert "moe_layer_forward" in names and len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(L.EXPORTED)


def test_status_strings_and_adaptive_tau(L):
    assert L.status_string(0) == "ok"
    assert "workspace" in L.status_string(3)
    assert abs(L.adaptive_tau(0.0) - 0.5) < 1e-7
    assert abs(L.adaptive_tau(math.log(3.0)) - 0.25) < 1e-7
    assert abs(L.adaptive_tau(-3.0) - 1.0 / (1.0 + math.exp(-3.0))) < 1e-7


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails its host checks


def _cfg(L, **kw):
    base = dict(T=64, d=256, E=8, k=2, H=128, n_shared=0, H_shared=0, dtype="bf16",
                gating="softmax_topk", residual="input")
    base.update(kw)
    return L.Config(**base).c()


@pytest.mark.parametrize("kw,code", [
    (dict(k=9), 1), (dict(k=0), 1), (dict(E=300, k=2), 1), (dict(T=-1), 1), (dict(d=0), 1),
    (dict(d=200), 2), (dict(H=100), 2), (dict(n_shared=1, H_shared=64), 2),
    (dict(dtype="f32", d=96), 2), (dict(n_shared=1, H_shared=0), 1),
    (dict(E=64, k=33), 1), (dict(T=(1 << 27) + 1, E=16, k=8), 2), (dict(T=(1 << 21) + 1, k=8), 2),
    (dict(dtype="f32", H=96), 2), (dict(dtype="f32", n_shared=1, H_shared=96), 2),
])
def test_route_rejects_bad_configs(L, kw, code):
    c = _cfg(L, **kw)
    r = L.lib().moe_route(ctypes.byref(c), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == code


def test_pair_limit_boundary(L):
    """2^24 routed pairs are accepted (the workspace query answers), one token more is not."""
    lib = L.lib()
    ok = _cfg(L, T=1 << 21, E=16, k=8)
    over = _cfg(L, T=(1 << 21) + 1, E=16, k=8)
    assert lib.moe_dispatch_workspace_size(ctypes.byref(ok)) > 0
    assert lib.moe_dispatch_workspace_size(ctypes.byref(over)) == 0


def test_route_rejects_null_and_misaligned(L):
    c = _cfg(L)
    lib = L.lib()
    big = 1 << 40
    assert lib.moe_route(ctypes.byref(c), None, FAKE, None, FAKE, FAKE, FAKE, FAKE, big, None) == 1
    assert lib.moe_route(ctypes.byref(c), FAKE + 4, FAKE, None, FAKE, FAKE, FAKE, FAKE, big, None) == 1
    assert lib.moe_route(ctypes.byref(c), FAKE, FAKE, FAKE + 8, FAKE, FAKE, FAKE, FAKE, big, None) == 1
    assert lib.moe_route(None, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, big, None) == 1
    need = lib.moe_route_workspace_size(ctypes.byref(c))
    assert need > 0  # bf16 layers route on the tensor cores and need scratch
    assert lib.moe_route(ctypes.byref(c), FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, need - 1, None) == 3
    assert lib.moe_route_workspace_size(ctypes.byref(_cfg(L, dtype="f32"))) == 0


def test_workspace_checks(L):
    c = _cfg(L)
    lib = L.lib()
    need = lib.moe_dispatch_workspace_size(ctypes.byref(c))
    assert need > 0
    r = lib.moe_dispatch(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None)
    assert r == 3
    full = lib.moe_workspace_size(ctypes.byref(c), 0)
    cond = lib.moe_workspace_size(ctypes.byref(c), 1)
    assert cond > full > 0
    w = L.moe_weights(FAKE, None, FAKE, FAKE, None, None)
    r = lib.moe_layer_forward(ctypes.byref(c), ctypes.byref(w), FAKE, None, float("nan"), FAKE,
                              None, None, FAKE, full - 1, None)
    assert r == 3
    # condensation of an fp32 layer is not supported
    c32 = _cfg(L, dtype="f32")
    r = lib.moe_layer_forward(ctypes.byref(c32), ctypes.byref(w), FAKE, None, 0.9, FAKE,
                              None, None, FAKE, 1 << 40, None)
    assert r == 2
    # external residual needs a residual pointer
    ce = _cfg(L, residual="external")
    r = lib.moe_layer_forward(ctypes.byref(ce), ctypes.byref(w), FAKE, None, float("nan"), FAKE,
                              None, None, FAKE, 1 << 40, None)
    assert r == 1
    # shared experts need shared weights
    cs = _cfg(L, n_shared=1, H_shared=128)
    r = lib.moe_expert_ffn(ctypes.byref(cs), ctypes.byref(w), FAKE, FAKE, None, FAKE, FAKE, FAKE,
                           FAKE, 1 << 40, None)
    assert r == 1


def test_condensation_limits(L):
    """Condensation takes bf16 layers of at most 65536 tokens (checked on the host)."""
    lib = L.lib()
    w = L.moe_weights(FAKE, None, FAKE, FAKE, None, None)
    cbig = _cfg(L, T=65537)
    r = lib.moe_condense(ctypes.byref(cbig), FAKE, FAKE, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == 2
    r = lib.moe_layer_forward(ctypes.byref(cbig), ctypes.byref(w), FAKE, None, 0.9, FAKE,
                              None, None, FAKE, 1 << 40, None)
    assert r == 2
    r = lib.moe_layer_forward_ex(ctypes.byref(cbig), ctypes.byref(w), FAKE, None, 0.9, FAKE, None,
                                 None, None, FAKE, 1 << 40, None, None)
    assert r == 2
    c32 = _cfg(L, dtype="f32")
    r = lib.moe_condense(ctypes.byref(c32), FAKE, FAKE, 0.9, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == 2


def test_layer_forward_ex_argument_checks(L):
    lib = L.lib()
    c = _cfg(L)
    w = L.moe_weights(FAKE, None, FAKE, FAKE, None, None)
    full = lib.moe_workspace_size(ctypes.byref(c), 0)
    # workspace too small, misaligned partial output, missing output
    assert lib.moe_layer_forward_ex(ctypes.byref(c), ctypes.byref(w), FAKE, None, float("nan"),
                                    FAKE, FAKE, None, None, FAKE, full - 1, None, None) == 3
    assert lib.moe_layer_forward_ex(ctypes.byref(c), ctypes.byref(w), FAKE, None, float("nan"),
                                    FAKE, FAKE + 2, None, None, FAKE, full, None, None) == 1
    assert lib.moe_layer_forward_ex(ctypes.byref(c), ctypes.byref(w), FAKE, None, float("nan"),
                                    None, FAKE, None, None, FAKE, full, None, None) == 1
    # zero tokens: nothing to do, with or without a second stream
    c0 = _cfg(L, T=0)
    assert lib.moe_layer_forward_ex(ctypes.byref(c0), ctypes.byref(w), None, None, float("nan"),
                                    None, None, None, None, None, 0, None, FAKE) == 0


def test_layer_backward_argument_checks(L):
    lib = L.lib()
    w = L.moe_weights(FAKE, None, FAKE, FAKE, None, None)
    c = _cfg(L)
    need = lib.moe_layer_backward_workspace_size(ctypes.byref(c), 0)
    assert lib.moe_layer_backward_workspace_size(ctypes.byref(c), 1) > need > 0
    nan = float("nan")
    args = lambda cfg, d_out, tau, ws_bytes: (ctypes.byref(cfg), ctypes.byref(w), FAKE, d_out, tau,
                                              FAKE, None, FAKE, None, FAKE, FAKE, None, None, FAKE,
                                              ws_bytes, None)
    assert lib.moe_layer_backward(*args(c, FAKE, nan, need - 1)) == 3      # workspace too small
    assert lib.moe_layer_backward(*args(c, None, nan, need)) == 1          # no output gradient
    c32 = _cfg(L, dtype="f32")
    assert lib.moe_layer_backward(*args(c32, FAKE, nan, 1 << 40)) == 2     # fp32 layers
    cbig = _cfg(L, T=70000)
    assert lib.moe_layer_backward(*args(cbig, FAKE, 0.9, 1 << 40)) == 2    # condensing T > 65536
    c0 = _cfg(L, T=0)
    assert lib.moe_layer_backward(ctypes.byref(c0), ctypes.byref(w), None, None, nan, None, None,
                                  None, None, None, None, None, None, None, 0, None) == 0


def test_zero_tokens_is_a_no_op(L):
    c = _cfg(L, T=0)
    lib = L.lib()
    assert lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, 0, None) == 0
    w = L.moe_weights(FAKE, None, FAKE, FAKE, None, None)
    assert lib.moe_layer_forward(ctypes.byref(c), ctypes.byref(w), None, None, float("nan"), None,
                                 None, None, None, 0, None) == 0
