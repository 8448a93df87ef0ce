"""Layer backward (moe_layer_backward) vs the fp64 oracle's chain rule, on one GPU.

Routing is bit-exact (the same forward recompute as the forward tests).  Gradients are
compared as max|gpu - oracle| <= BWD_TOL * max|oracle| per tensor, with BWD_TOL = 1e-2, the
bound the layer statement gives bf16 outputs.  The backward chains two more bf16 roundings
than the forward (the output gradient dy = g * d_out and the SwiGLU gradient dA are rounded
to bf16 before their GEMMs, on top of the recomputed pre-activations and h), each worth up to
2^-9 relative, accumulated over K = d, 2H or the expert's rows in fp32; measured on every case
here the largest error is 0.998e-2 (a small expert's down-projection weight gradient), and
the kernels are deterministic, so the same inputs give the same error on every run.
"""
from __future__ import annotations

import math
from dataclasses import replace

import numpy as np
import pytest

from oracle import moe_oracle as orc
from routing_expert_ffn_gb300 import inputs as gen
from tests import harness

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BWD_TOL = 1e-2

SMALL = {
    # softmax top-k, shared expert, residual = x (DeepSeek-V2-Lite-like, narrow)
    "softmax_shared": replace(gen.CONFIGS["dsv2_lite"], name="bwd_softmax_shared", T=300, d=512,
                              E=8, k=2, H=256, n_shared=1, H_shared=256),
    # renormalised top-k with a Zipf router bias, no shared expert (Qwen3-like, narrow)
    "renorm_zipf": replace(gen.CONFIGS["qwen3_30b_a3b"], name="bwd_renorm_zipf", T=300, d=512,
                           E=16, k=4, H=128),
    # sigmoid top-1, FarSkip external residual, shared expert (Llama-4-Scout-like, narrow)
    "sigmoid_farskip": replace(gen.CONFIGS["llama4_scout_farskip"], name="bwd_sigmoid_farskip",
                               T=200, d=512, E=4, k=1, H=256, n_shared=1, H_shared=256),
    # two shared experts (their gradients span two weight slices)
    "two_shared": replace(gen.CONFIGS["dsv2_lite"], name="bwd_two_shared", T=130, d=256, E=4,
                          k=2, H=128, n_shared=2, H_shared=128),
}


@pytest.fixture(scope="module")
def moe():
    from routing_expert_ffn_gb300 import build
    build.build()
    from routing_expert_ffn_gb300 import moe as m
    m.lib()
    return m


def _np(t):
    return t.detach().float().cpu().numpy()


def _case(moe, cfg, seed=21):
    inp = harness.condition(cfg, gen.make_inputs(cfg))
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp)
    rng = np.random.default_rng(seed)
    d_out_np = gen.round_to_bf16(rng.standard_normal((cfg.T, cfg.d)).astype(np.float32))
    d_out = torch.from_numpy(d_out_np).to("cuda").to(torch.bfloat16)
    return inp, C, w, x, d_out, d_out_np


def _err(got, ref):
    return harness.max_rel_err(got, ref)


def _check(g, ref, cfg, experts=None):
    assert _err(_np(g["d_x"]), ref["dx"]) <= BWD_TOL, "d_x"
    assert _err(_np(g["dW_r"]), ref["dW_r"]) <= BWD_TOL, "dW_r"
    if ref["d_bias"] is not None:
        assert _err(_np(g["d_bias"]), ref["d_bias"]) <= BWD_TOL, "d_bias"
    es = range(cfg.E) if experts is None else experts
    for e in es:
        if np.any(ref["dW_gu"][e]):
            assert _err(_np(g["dW_gu"][e]), ref["dW_gu"][e]) <= BWD_TOL, ("dW_gu", e)
            assert _err(_np(g["dW_down"][e]), ref["dW_down"][e]) <= BWD_TOL, ("dW_down", e)
        else:  # an expert no token chose: zero gradient
            assert not torch.any(g["dW_gu"][e]) and not torch.any(g["dW_down"][e]), e
    for s in range(cfg.n_shared):
        assert _err(_np(g["dWs_gu"][s]), ref["dWs_gu"][s]) <= BWD_TOL, ("dWs_gu", s)
        assert _err(_np(g["dWs_down"][s]), ref["dWs_down"][s]) <= BWD_TOL, ("dWs_down", s)
    if ref["d_residual"] is not None:
        np.testing.assert_array_equal(_np(g["d_residual"]), ref["d_residual"].astype(np.float32))


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_small(moe, name):
    cfg = SMALL[name]
    inp, C, w, x, d_out, d_out_np = _case(moe, cfg)
    g = moe.layer_backward(C, w, x, d_out, d_residual=True)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = orc.layer_backward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating, d_out_np,
                             residual_mode=cfg.residual, residual=inp["residual"])
    _check(g, ref, cfg)


def test_backward_with_condensation(moe):
    """Near-duplicate tokens condensed at tau = 0.95: a condensed pair's expert gradient lands
    on its representative's token (Luffy review, referee major comment 1), everything against
    the oracle's chain rule through the same condensed forward."""
    cfg = replace(gen.CONFIGS["luffy_condense"], name="bwd_condense", T=600, d=512, E=4, k=2,
                  H=256, n_centroids=16, copy_fraction=0.4, noise_rel=0.02)
    tau = 0.95
    inp, C, w, x, d_out, d_out_np = _case(moe, cfg)
    g = moe.layer_backward(C, w, x, d_out, tau=tau)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    ref = orc.layer_backward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating, d_out_np,
                             residual_mode=cfg.residual, residual=inp["residual"], tau=tau)
    n_cond = int((ref["rep_of"] != np.arange(len(ref["rep_of"]))).sum())
    assert n_cond > 0.2 * len(ref["rep_of"]), n_cond  # the workload condenses a good share
    _check(g, ref, cfg)


def test_backward_full_width_decode_shape(moe):
    """DeepSeek-V2-Lite widths (d = 2048, 64 experts, H = 1408, 2 shared experts) at 64 tokens:
    the input, router and shared gradients in full, the routed weight gradients of the first
    three experts that received tokens and of one that received none."""
    cfg = gen.CONFIGS["dsv2_lite_decode"]
    inp, C, w, x, d_out, d_out_np = _case(moe, cfg)
    g = moe.layer_backward(C, w, x, d_out)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    idx = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)[1]
    used = sorted(set(idx.ravel().tolist()))
    unused = sorted(set(range(cfg.E)) - set(used))
    experts = used[:3] + unused[:1]
    ref = orc.layer_backward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating, d_out_np,
                             residual_mode=cfg.residual, residual=inp["residual"],
                             grad_experts=experts)
    _check(g, ref, cfg, experts=experts)


def test_backward_full_size_dsv2_lite(moe):
    """The DeepSeek-V2-Lite-shaped layer at its full 4096 tokens: the input and router
    gradients of every token, both shared experts' weight gradients, and the routed weight
    gradients of three experts (the first, a middle and the last expert index)."""
    cfg = gen.CONFIGS["dsv2_lite"]
    inp, C, w, x, d_out, d_out_np = _case(moe, cfg)
    g = moe.layer_backward(C, w, x, d_out)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    experts = [0, cfg.E // 2, cfg.E - 1]
    ref = orc.layer_backward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating, d_out_np,
                             residual_mode=cfg.residual, residual=inp["residual"],
                             grad_experts=experts)
    _check(g, ref, cfg, experts=experts)


def test_backward_deterministic(moe):
    cfg = SMALL["softmax_shared"]
    inp, C, w, x, d_out, _ = _case(moe, cfg)
    a = moe.layer_backward(C, w, x, d_out)
    b = moe.layer_backward(C, w, x, d_out)
    torch.cuda.synchronize()
    for key in ("d_x", "dW_r", "dW_gu", "dW_down", "dWs_gu", "dWs_down"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("condense", [False, True])
def test_backward_poisoned_workspace(moe, condense):
    """Every byte of the backward's scratch set to 0xFF before the call (NaN in every float, -1
    in every index) gives the same gradient bits as a zeroed workspace, and every gradient
    element is written (the gradient buffers start as NaN)."""
    if condense:
        cfg = replace(gen.CONFIGS["luffy_condense"], name="bwd_poison_condense", T=600, d=512,
                      E=4, k=2, H=256, n_centroids=16, copy_fraction=0.4, noise_rel=0.02)
        tau = 0.95
    else:
        cfg, tau = SMALL["softmax_shared"], math.nan
    inp, C, w, x, d_out, _ = _case(moe, cfg)
    bwd = moe.Backward(C, w, condense=condense)
    runs = []
    for fill in (0, 255):
        bwd.ws.fill_(fill)
        for v in bwd.grads.values():
            if v is not None:
                v.fill_(float("nan"))
        g = bwd(x, d_out, tau)
        runs.append({k: v.clone() for k, v in g.items() if v is not None})
    torch.cuda.synchronize()
    a, b = runs
    for key in a:
        assert not torch.isnan(a[key]).any().item(), key
        assert torch.equal(a[key], b[key]), key
    assert moe.get_device_status() == 0
