"""CUDA path vs the fp64 oracle, through the C ABI (libmoe.so) on one GPU.

Bit-exact: routing indices, counts, offsets, permutation, slot map, x_perm,
condensation assignment.  Within max|gpu - oracle| <= tol * max|oracle|
(1e-4 fp32 layers, 1e-2 bf16 layers): gates, expert outputs, layer outputs.
Small cases run every token; the full-size workloads compare sampled tokens
(their routing and permutation are still compared in full).
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import moe_oracle as orc
from routing_expert_ffn_gb300 import inputs as gen
from tests import harness

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NAMES = gen.CONFIG_ORDER
# Token counts the oracle runs whole layers on in seconds, spanning several m-tiles and a ragged tail.
SMALL_T = {"tiny_fp32": 256, "dsv2_lite": 600, "qwen3_30b_a3b": 700, "llama4_scout_farskip": 300,
           "luffy_condense": 1000}


@pytest.fixture(scope="module")
def moe():
    from routing_expert_ffn_gb300 import build
    build.build()
    from routing_expert_ffn_gb300 import moe as m
    m.lib()
    return m


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float16) else t.detach().cpu().numpy()


def _setup(moe, name, T=None, x_kind=None, **over):
    cfg, inp = harness.workload(name, T, x_kind)
    C = moe.Config.from_workload(cfg)
    for k_, v in over.items():
        setattr(C, k_, v)
    w, x, r = moe.upload(C, inp)
    return cfg, inp, C, w, x, r


def _sample_tokens(T, n=48, seed=0):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    return np.array(sorted(s))


def _status_ok(moe):
    assert moe.get_device_status() == 0


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("name", NAMES)
def test_router_full_size(moe, name):
    cfg, inp, C, w, x, r = _setup(moe, name)
    logits, idx, gate = moe.route(C, x, w.W_r, w.router_bias)
    torch.cuda.synchronize()
    l_ref, idx_ref, g_ref = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    np.testing.assert_array_equal(_np(idx), idx_ref)
    # fp32-accurate logits: sequential fp32 FMA (fp32 layers) or tensor-core fp32
    # accumulation of exact bf16 x bf16 products (bf16 layers)
    assert harness.max_rel_err(_np(logits), l_ref) < 5e-5
    np.testing.assert_allclose(_np(gate), g_ref, rtol=2e-5, atol=1e-7)
    _status_ok(moe)


@pytest.mark.parametrize("E,k,gating", [(16, 1, "sigmoid_topk"), (64, 6, "softmax_topk"),
                                         (128, 8, "softmax_topk_renorm"), (200, 8, "softmax_topk"),
                                         (256, 32, "softmax_topk_renorm")])
def test_router_exact_ties(moe, E, k, gating):
    """Small-integer tokens, router weights and bias: every logit is an integer that the
    tensor-core path (exact bf16 terms, fp32 accumulation) and the fp64 oracle both compute
    exactly, and logits tie often (a fifth of the experts copy another one's weights), so the
    selection must follow the tie rule -- the lower expert index first -- bit for bit."""
    rng = np.random.default_rng(1000 + E + k)
    T, d = 777, 256
    x = rng.integers(-2, 3, size=(T, d)).astype(np.float32)
    W_r = rng.integers(-3, 4, size=(d, E)).astype(np.float32)
    W_r[:, 1::5] = W_r[:, 0::5][:, : W_r[:, 1::5].shape[1]]
    bias = rng.integers(-2, 3, size=E).astype(np.float32) if gating == "softmax_topk_renorm" else None
    if bias is not None:
        bias[1::5] = bias[0::5][: bias[1::5].shape[0]]
    C = moe.Config(T=T, d=d, E=E, k=k, H=128, n_shared=0, H_shared=0, dtype="bf16",
                   gating=gating, residual="none")
    xd = torch.from_numpy(x).to(device="cuda", dtype=torch.bfloat16)
    logits, idx, gate = moe.route(C, xd, torch.from_numpy(W_r).cuda(),
                                  torch.from_numpy(bias).cuda() if bias is not None else None)
    torch.cuda.synchronize()
    l_ref, idx_ref, g_ref = orc.route(x, W_r, bias, k, gating)
    np.testing.assert_array_equal(_np(logits), l_ref.astype(np.float32))  # integers, exact
    srt = -np.sort(-l_ref, axis=1)
    assert np.mean(srt[:, : k] == srt[:, 1 : k + 1]) > 0.05  # ties inside the top k + 1
    np.testing.assert_array_equal(_np(idx), idx_ref)
    np.testing.assert_allclose(_np(gate), g_ref, rtol=2e-5, atol=1e-7)
    _status_ok(moe)


@pytest.mark.parametrize("E", [8, 33, 64, 65, 96, 128, 129])
def test_router_terms_side_by_side_boundary(moe, E):
    """Up to E = 128 the tensor-core router puts the three bf16 terms of W_r side by side
    along N and splits K over d: in one MMA up to E = 64 (N = 3 x E rounded up to 32, at
    most 256), in two (terms 1 and 2, then term 3) above; past 128 the terms follow one
    another along K.  Both sides of both boundaries, 1000 tokens (a ragged last m-tile),
    every token against the oracle."""
    from dataclasses import replace
    cfg = replace(gen.CONFIGS["qwen3_30b_a3b"], name=f"router{E}", T=1000, d=512, E=E, k=2, H=128,
                  n_shared=1, H_shared=128, router_bias="none")
    inp = harness.condition(cfg, gen.make_inputs(cfg))
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp)
    logits, idx, gate = moe.route(C, x, w.W_r, w.router_bias)
    torch.cuda.synchronize()
    l_ref, idx_ref, g_ref = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    np.testing.assert_array_equal(_np(idx), idx_ref)
    assert harness.max_rel_err(_np(logits), l_ref) < 5e-5
    np.testing.assert_allclose(_np(gate), g_ref, rtol=2e-5, atol=1e-7)
    _status_ok(moe)


# ------------------------------------------------------------------ dispatch
@pytest.mark.parametrize("name", NAMES)
def test_dispatch_full_size(moe, name):
    cfg, inp, C, w, x, r = _setup(moe, name)
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    out = moe.dispatch(C, x, idx)
    torch.cuda.synchronize()
    counts, offsets, perm, slot_of = orc.dispatch(_np(idx), cfg.E)
    np.testing.assert_array_equal(_np(out["counts"]), counts)
    np.testing.assert_array_equal(_np(out["offsets"]), offsets)
    np.testing.assert_array_equal(_np(out["perm"])[: cfg.P], perm)
    np.testing.assert_array_equal(_np(out["slot_of"]), slot_of)
    # rows moved bit for bit
    ref = x.index_select(0, out["perm"][: cfg.P].long())
    assert torch.equal(out["x_perm"][: cfg.P], ref)
    _status_ok(moe)


def test_dispatch_empty_buckets_and_skew(moe):
    cfg, inp, C, w, x, r = _setup(moe, "qwen3_30b_a3b")
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    out = moe.dispatch(C, x, idx)
    counts = _np(out["counts"])
    assert (counts == 0).any() and counts.max() > 4 * cfg.P / cfg.E
    assert counts.sum() == cfg.P


# ------------------------------------------------------------------ expert FFN
def _ffn_check(moe, name, T):
    cfg, inp, C, w, x, r = _setup(moe, name, T=T)
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    y, so = moe.expert_ffn(C, w, d["x_perm"], d["offsets"], None, x)
    torch.cuda.synchronize()
    perm = _np(d["perm"])[: cfg.P]
    offsets = _np(d["offsets"])
    rng = np.random.default_rng(1)
    slots = np.unique(np.concatenate([rng.choice(cfg.P, size=min(256, cfg.P), replace=False),
                                      offsets[1:-1] - 1, offsets[:-1][offsets[:-1] < cfg.P],
                                      [cfg.P - 1]]))
    expert_of_slot = np.searchsorted(offsets, slots, side="right") - 1
    yg = _np(y)[slots]
    yr = np.zeros_like(yg, dtype=np.float64)
    for e in np.unique(expert_of_slot):
        m = expert_of_slot == e
        yr[m] = orc.swiglu_expert(inp["x"][perm[slots[m]]], inp["W_gu"][e], inp["W_down"][e])
    assert harness.max_rel_err(yg, yr) <= harness.tolerance(cfg), name
    if cfg.n_shared:
        toks = _sample_tokens(cfg.T, 64)
        sr = orc.shared_experts(inp["x"][toks], inp["Ws_gu"], inp["Ws_down"])
        assert harness.max_rel_err(_np(so)[toks], sr) <= harness.tolerance(cfg), name
    _status_ok(moe)


@pytest.mark.parametrize("name", NAMES)
def test_expert_ffn_small(moe, name):
    _ffn_check(moe, name, SMALL_T[name])


@pytest.mark.parametrize("name", ["dsv2_lite", "qwen3_30b_a3b", "llama4_scout_farskip"])
def test_expert_ffn_full_size(moe, name):
    _ffn_check(moe, name, None)


# Group sizes around every tile boundary of the expert GEMMs: empty, one row, and one short of,
# at and one past 16, 128, 192, 256, 384, 448 and 512 rows, so that every way a group splits
# into 256-row pair tiles and tail tiles of at most 192 rows (N rounded up to 16; a tail of more
# than 128 rows loads its halves with the 128-row box) occurs; and 14, 32 and 33 rows past one
# pair and 32 past two (small tails, N = 16 or 32, beside the pairs of the same group).
GROUP_SIZES = [0, 1, 15, 16, 17, 127, 128, 129, 191, 192, 193, 255, 256, 257, 383, 384, 385,
               447, 448, 449, 511, 512, 513, 200, 270, 288, 289, 544]


def test_expert_ffn_group_sizes_every_row(moe):
    T = 1300
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite", T=T)
    P = cfg.P
    sizes = GROUP_SIZES + [0] * (cfg.E - len(GROUP_SIZES))
    sizes[-1] = P - sum(GROUP_SIZES)
    assert sizes[-1] > 0
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    _, rows_inp = harness.workload("dsv2_lite", P)  # any bf16 rows; weights do not depend on T
    rows = rows_inp["x"]
    x_perm = torch.from_numpy(rows).to(device=x.device, dtype=C.torch_dtype)
    off_d = torch.from_numpy(offsets).to(x.device)
    y, _ = moe.expert_ffn(C, w, x_perm, off_d, None, x)
    torch.cuda.synchronize()
    yg = _np(y)
    for e, n in enumerate(sizes):
        if n == 0:
            continue
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        ref = orc.swiglu_expert(rows[sl], inp["W_gu"][e], inp["W_down"][e])
        err = harness.max_rel_err(yg[sl], ref)
        assert err <= harness.tolerance(cfg), (e, n, err)
    _status_ok(moe)


def test_expert_ffn_tails_only_batch_every_row(moe):
    """A batch of at most 128 tokens: every group (and the shared experts' one group of T rows)
    is a single tail tile, which the GEMM runs with its tails-only ring layout.  Group sizes
    around the 16-row N steps and the 64-row token box, up to T; every slot and every shared
    row against the oracle."""
    T = 128
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite", T=T)
    P = cfg.P
    head = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 31, 33, 0, 96, 112]
    sizes = head + [0] * (cfg.E - len(head))
    rest = P - sum(head)
    for e in range(len(head), cfg.E):  # the remaining rows in groups of at most T
        sizes[e] = min(T, rest)
        rest -= sizes[e]
    assert rest == 0 and max(sizes) <= T
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    _, rows_inp = harness.workload("dsv2_lite", P)
    rows = rows_inp["x"]
    x_perm = torch.from_numpy(rows).to(device=x.device, dtype=C.torch_dtype)
    off_d = torch.from_numpy(offsets).to(x.device)
    y, so = moe.expert_ffn(C, w, x_perm, off_d, None, x)
    torch.cuda.synchronize()
    yg = _np(y)
    for e, n in enumerate(sizes):
        if n == 0:
            continue
        sl = slice(int(offsets[e]), int(offsets[e + 1]))
        ref = orc.swiglu_expert(rows[sl], inp["W_gu"][e], inp["W_down"][e])
        err = harness.max_rel_err(yg[sl], ref)
        assert err <= harness.tolerance(cfg), (e, n, err)
    ref_s = orc.shared_experts(inp["x"], inp["Ws_gu"], inp["Ws_down"])
    assert harness.max_rel_err(_np(so), ref_s) <= harness.tolerance(cfg)
    _status_ok(moe)


def test_expert_ffn_small_batch_refuses_oversized_bucket(moe):
    """Offsets that no dispatch writes (a bucket of more rows than the batch has tokens) on a
    batch of at most 128 tokens: the routed GEMM refuses them on the device, computes no tile
    and reports MOE_ERR_DEVICE_INDEX; the next valid call is unaffected."""
    T = 100
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite", T=T)
    P = cfg.P
    sizes = [200, P - 200] + [0] * (cfg.E - 2)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    _, rows_inp = harness.workload("dsv2_lite", P)
    x_perm = torch.from_numpy(rows_inp["x"]).to(device=x.device, dtype=C.torch_dtype)
    y, _ = moe.expert_ffn(C, w, x_perm, torch.from_numpy(offsets).to(x.device), None, x)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 6  # MOE_ERR_DEVICE_INDEX
    assert not torch.any(y != 0).item()  # no routed tile ran
    _layer_check(moe, "dsv2_lite", T=T)
    _status_ok(moe)


# ------------------------------------------------------------------ combine / round trip
def test_round_trip_identity_experts(moe):
    """dispatch -> identity experts (y = x_perm) -> combine with gates summing to 1 == x."""
    cfg, inp, C, w, x, r = _setup(moe, "qwen3_30b_a3b", T=1000)
    C.residual = "none"
    _, idx, gate = moe.route(C, x, w.W_r, w.router_bias)  # renormalised gates
    d = moe.dispatch(C, x, idx)
    out = moe.combine(C, d["x_perm"], None, d["slot_of"], None, gate, x)
    torch.cuda.synchronize()
    assert torch.equal(out, x)


# ------------------------------------------------------------------ whole layer
def _layer_check(moe, name, T=None, tau=math.nan, residual=None, tokens=None):
    cfg, inp, C, w, x, r = _setup(moe, name, T=T)
    if residual is not None:
        C.residual = residual
    lay = moe.Layer(C, w, condense=tau <= 1.0)
    idx = torch.empty((C.T, C.k), dtype=torch.int32, device=x.device)
    ncond = torch.zeros(1, dtype=torch.int32, device=x.device)
    out = lay(x, r, tau, topk_idx_out=idx, n_condensed_out=ncond)
    torch.cuda.synchronize()
    toks = np.arange(C.T) if tokens is None else tokens
    ref = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                            inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                            residual_mode=C.residual, residual=inp["residual"],
                            tau=None if not tau <= 1.0 else tau, tokens=toks)
    np.testing.assert_array_equal(_np(idx), ref["idx"])
    err = harness.max_rel_err(_np(out)[toks], ref["out"])
    assert err <= harness.tolerance(cfg), (name, err)
    expected_cond = int((ref["rep_of"] != np.arange(len(ref["rep_of"]))).sum())
    assert int(ncond.item()) == expected_cond
    _status_ok(moe)
    return out, ref


@pytest.mark.parametrize("name", NAMES)
def test_layer_small(moe, name):
    _layer_check(moe, name, T=SMALL_T[name])


@pytest.mark.parametrize("name", NAMES)
def test_layer_small_moe_part_only(moe, name):
    """The residual dominates max|out|; the routed + shared part alone meets the same bound."""
    _layer_check(moe, name, T=SMALL_T[name], residual="none")


@pytest.mark.parametrize("name", NAMES)
def test_layer_full_size_sampled(moe, name):
    cfg = gen.CONFIGS[name]
    tau = cfg.taus[0] if cfg.taus else math.nan
    _layer_check(moe, name, tau=tau, tokens=_sample_tokens(cfg.T, 48))


def test_layer_full_size_every_token_dsv2_lite(moe):
    """The DeepSeek-V2-Lite-shaped layer at its full 4096 tokens, every token of the output
    against the oracle (its whole fp64 layer, about 570 GFLOP, takes seconds on the host)."""
    _layer_check(moe, "dsv2_lite")


def test_expert_ffn_full_size_every_slot_dsv2_lite(moe):
    """Every one of the 24576 routed slots (and every token's shared output) of the
    DeepSeek-V2-Lite-shaped expert FFN against the oracle's SwiGLU experts."""
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite")
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    y, so = moe.expert_ffn(C, w, d["x_perm"], d["offsets"], None, x)
    torch.cuda.synchronize()
    _, offsets, perm, _ = orc.dispatch(orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k,
                                                 cfg.gating)[1], cfg.E)
    np.testing.assert_array_equal(_np(d["perm"])[: cfg.P], perm)
    yr = np.zeros((cfg.P, cfg.d))
    for e in range(cfg.E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            yr[a:b] = orc.swiglu_expert(inp["x"][perm[a:b]], inp["W_gu"][e], inp["W_down"][e])
    assert harness.max_rel_err(_np(y)[: cfg.P], yr) <= harness.tolerance(cfg)
    sr = orc.shared_experts(inp["x"], inp["Ws_gu"], inp["Ws_down"])
    assert harness.max_rel_err(_np(so), sr) <= harness.tolerance(cfg)
    _status_ok(moe)


@pytest.mark.parametrize("E,k", [(256, 8), (64, 32)])
def test_layer_max_experts_and_k(moe, E, k):
    """The largest E (256: router split-K path, 257-entry group tables in the dispatch and both
    GEMM kernels) and the largest k (32) the boundary takes, renormalised gates and a shared
    expert; every token against the oracle."""
    from dataclasses import replace
    cfg = replace(gen.CONFIGS["qwen3_30b_a3b"], name=f"e{E}k{k}", T=600, d=256, E=E, k=k, H=128,
                  n_shared=1, H_shared=128, router_bias="none")
    inp = harness.condition(cfg, gen.make_inputs(cfg))
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp)
    lay = moe.Layer(C, w)
    idx = torch.empty((C.T, C.k), dtype=torch.int32, device=x.device)
    out = lay(x, r, math.nan, topk_idx_out=idx)
    torch.cuda.synchronize()
    ref = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                            inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                            residual_mode=C.residual, residual=inp["residual"], tau=None,
                            tokens=np.arange(C.T))
    np.testing.assert_array_equal(_np(idx), ref["idx"])
    assert harness.max_rel_err(_np(out), ref["out"]) <= harness.tolerance(cfg)
    _status_ok(moe)


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 777])
def test_layer_ragged_token_counts(moe, T):
    _layer_check(moe, "dsv2_lite", T=T)
    _layer_check(moe, "tiny_fp32", T=min(T, 256))


def test_layer_k_equals_E_identical_experts(moe):
    """k = E, identical experts, renormalised gates: the layer is one dense SwiGLU FFN."""
    cfg, inp = harness.workload("tiny_fp32")
    from dataclasses import replace
    E = 4
    cfgk = replace(cfg, E=E, k=E, gating="softmax_topk_renorm", residual="none", n_shared=0)
    C = moe.Config.from_workload(cfgk)
    inp2 = dict(inp)
    inp2["W_r"] = inp["W_r"][:, :E].copy()
    inp2["W_gu"] = np.repeat(inp["W_gu"][:1], E, axis=0)
    inp2["W_down"] = np.repeat(inp["W_down"][:1], E, axis=0)
    inp2["Ws_gu"] = inp["Ws_gu"][:0]
    inp2["Ws_down"] = inp["Ws_down"][:0]
    w, x, _ = moe.upload(C, inp2)
    out = moe.Layer(C, w)(x)
    torch.cuda.synchronize()
    dense = orc.swiglu_expert(inp["x"], inp["W_gu"][0], inp["W_down"][0])
    assert harness.max_rel_err(_np(out), dense) <= 1e-4


def test_layer_deterministic(moe):
    cfg, inp, C, w, x, r = _setup(moe, "qwen3_30b_a3b", T=2048)
    lay = moe.Layer(C, w)
    a = lay(x, r).clone()
    b = lay(x, r)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# Workspace poisoning: every byte of the layer's scratch set to 0xFF before the call (NaN in
# every float, -1 in every index) must give the same output bits as a zeroed workspace, and
# every output element must be written (the output starts as NaN).  This would catch a kernel
# that reads scratch the same call has not written (a table, a counter, a padding row).
POISON_CASES = [("dsv2_lite", 600, math.nan), ("qwen3_30b_a3b", 700, math.nan),
                ("luffy_condense", 1024, 0.95), ("dsv2_lite_decode", None, math.nan),
                ("tiny_fp32", 256, math.nan), ("llama4_scout_farskip", 300, math.nan)]


@pytest.mark.parametrize("name,T,tau", POISON_CASES)
def test_layer_poisoned_workspace(moe, name, T, tau):
    cfg, inp, C, w, x, r = _setup(moe, name, T=T)
    lay = moe.Layer(C, w, condense=tau <= 1.0)
    outs = []
    for fill in (0, 255):
        lay.ws.fill_(fill)
        out = torch.full((C.T, C.d), float("nan"), dtype=C.torch_dtype, device=x.device)
        idx = torch.full((C.T, C.k), -7, dtype=torch.int32, device=x.device)
        lay(x, r, tau, out=out, topk_idx_out=idx)
        outs.append((out, idx))
    torch.cuda.synchronize()
    (a, ia), (b, ib) = outs
    assert not torch.isnan(a).any().item()
    assert torch.equal(a, b)
    assert torch.equal(ia, ib)
    _status_ok(moe)


@pytest.mark.parametrize("name", ["dsv2_lite", "llama4_scout_farskip"])
def test_layer_ex_poisoned_workspace(moe, name):
    """The same for moe_layer_forward_ex: shared experts on a second stream and the partial
    activation written beside the output."""
    cfg, inp, C, w, x, r = _setup(moe, name, T=600)
    lay = moe.Layer(C, w)
    aux = torch.cuda.Stream()
    outs = []
    for fill in (0, 255):
        lay.ws.fill_(fill)
        out = torch.full((C.T, C.d), float("nan"), dtype=C.torch_dtype, device=x.device)
        part = torch.full_like(out, float("nan"))
        lay(x, r, out=out, partial_out=part, aux_stream=aux)
        outs.append((out, part))
    torch.cuda.synchronize()
    (a, pa), (b, pb) = outs
    assert not torch.isnan(a).any().item() and not torch.isnan(pa).any().item()
    assert torch.equal(a, b) and torch.equal(pa, pb)
    _status_ok(moe)


@pytest.mark.parametrize("residual,n_shared,T", [("external", 1, 300), ("input_plus_external", 0, 300),
                                                 ("input", 2, 100), ("none", 1, 129)])
def test_layer_matches_step_by_step_one_expert_per_token(moe, residual, n_shared, T):
    """One routed expert per token (the Llama-4-Scout shape, narrowed): the layer's output and
    partial activation equal, bit for bit, what the step-by-step calls (route, dispatch,
    expert FFN, combine) give, through both layer entry points, for every residual mode, with
    and without shared experts, and on a small batch (tail tiles only)."""
    from dataclasses import replace
    cfg = replace(gen.CONFIGS["llama4_scout_farskip"], name=f"k1_{residual}_{n_shared}",
                  T=T, d=512, E=4, k=1, H=256, n_shared=n_shared, H_shared=256,
                  residual=residual)
    inp = harness.condition(cfg, gen.make_inputs(cfg))
    C = moe.Config.from_workload(cfg)
    w, x, r = moe.upload(C, inp)
    lay = moe.Layer(C, w)
    out = lay(x, r)
    part = torch.empty_like(out)
    out_ex = lay(x, r, partial_out=part, aux_stream=torch.cuda.Stream())
    _, idx, gate = moe.route(C, x, w.W_r, w.router_bias)
    dsp = moe.dispatch(C, x, idx)
    y, so = moe.expert_ffn(C, w, dsp["x_perm"], dsp["offsets"], None, x)
    ref = moe.combine(C, y, so, dsp["slot_of"], None, gate, x, r)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(out_ex, ref)
    base = torch.zeros(out.shape, dtype=torch.float32, device=out.device)
    if residual in ("input", "input_plus_external"):
        base = base + x.float()
    if residual in ("external", "input_plus_external"):
        base = base + r.float()
    if n_shared:
        base = base + so.float()
    assert torch.equal(part, base.to(torch.bfloat16))
    _status_ok(moe)


# ------------------------------------------------------------------ decode-shaped layer
def test_decode_layer_every_token(moe):
    """One decode step (64 tokens) through the full DeepSeek-V2-Lite weights: routing bit for
    bit and every output row against the oracle, through both layer entry points."""
    out, _ = _layer_check(moe, "dsv2_lite_decode")
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite_decode")
    out_ex = moe.Layer(C, w)(x, r, aux_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert torch.equal(out_ex, out)


# ------------------------------------------------------------------ FarSkip partial output + overlap
@pytest.mark.parametrize("name", ["dsv2_lite", "llama4_scout_farskip", "tiny_fp32"])
def test_layer_ex_partial_and_shared_on_second_stream(moe, name):
    """moe_layer_forward_ex: out is bit-identical to moe_layer_forward (same kernels, the
    shared experts merely run on a second stream), and the partial activation r + shared
    matches the oracle."""
    cfg, inp, C, w, x, r = _setup(moe, name, T=SMALL_T[name])
    lay = moe.Layer(C, w)
    ref_out = lay(x, r).clone()
    aux = torch.cuda.Stream()
    part = torch.empty_like(ref_out)
    out = lay(x, r, partial_out=part, aux_stream=aux)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    ref = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                            inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                            residual_mode=C.residual, residual=inp["residual"])
    assert harness.max_rel_err(_np(part), ref["partial"]) <= harness.tolerance(cfg)
    assert harness.max_rel_err(_np(out), ref["out"]) <= harness.tolerance(cfg)
    # partial output without a second stream: the same values
    part2 = torch.empty_like(part)
    lay(x, r, partial_out=part2)
    torch.cuda.synchronize()
    assert torch.equal(part, part2)
    _status_ok(moe)


def test_layer_ex_second_stream_in_cuda_graph(moe):
    """The fork/join of the shared experts is captured into one graph that begins on the
    calling stream; replays reproduce the eager result bit for bit."""
    cfg, inp, C, w, x, r = _setup(moe, "dsv2_lite", T=SMALL_T["dsv2_lite"])
    lay = moe.Layer(C, w)
    eager = lay(x, r).clone()
    aux = torch.cuda.Stream()
    out = torch.empty_like(eager)
    part = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lay(x, r, out=out, partial_out=part, aux_stream=aux)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lay(x, r, out=out, partial_out=part, aux_stream=aux)
    out.zero_()
    part.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    ref = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                            inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                            residual_mode=C.residual, residual=inp["residual"])
    assert harness.max_rel_err(_np(part), ref["partial"]) <= harness.tolerance(cfg)
    _status_ok(moe)


# ------------------------------------------------------------------ condensation
@pytest.mark.parametrize("tau_index", [0, 1])
def test_condense_full_size(moe, tau_index):
    cfg, inp, C, w, x, r = _setup(moe, "luffy_condense")
    tau = cfg.taus[tau_index]
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    rep_of, n_rep, ncond = moe.condense(C, d["x_perm"], d["offsets"], tau)
    torch.cuda.synchronize()
    counts, offsets, perm, slot_of = orc.dispatch(_np(idx), cfg.E)
    ref = orc.condense(inp["x"][perm], offsets, tau)
    np.testing.assert_array_equal(_np(rep_of)[: cfg.P], ref)
    assert int(ncond.item()) == int((ref != np.arange(cfg.P)).sum()) > 0
    reps_per_bucket = [int((ref[offsets[e]:offsets[e + 1]] == np.arange(offsets[e], offsets[e + 1])).sum())
                       for e in range(cfg.E)]
    np.testing.assert_array_equal(_np(n_rep), reps_per_bucket)
    _status_ok(moe)


def test_condense_exact_duplicates_tau_one(moe):
    cfg, inp, C, w, x, r = _setup(moe, "luffy_condense", T=2048, x_kind="duplicates")
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    rep_of, _, ncond = moe.condense(C, d["x_perm"], d["offsets"], 1.0)
    torch.cuda.synchronize()
    _, offsets, perm, _ = orc.dispatch(_np(idx), cfg.E)
    ref = orc.condense(inp["x"][perm], offsets, 1.0)
    np.testing.assert_array_equal(_np(rep_of)[: cfg.P], ref)
    assert int(ncond.item()) > 0


@pytest.mark.parametrize("sizes", [(16400, 3000), (12300, 12200)])
def test_condense_duplicates_wide_buckets(moe, sizes):
    """Buckets above and below the scan's 12256-row group limit, exact duplicates at tau = 1.

    Closed form (no oracle run at this size): every row's representative is the first
    identical row of its bucket, since distinct random rows are far from cosine 1.
    """
    rng = np.random.default_rng(7)
    d = 256  # bf16 layers take d in multiples of 256
    pool = gen.round_to_bf16(rng.standard_normal((40, d)).astype(np.float32))
    ids = [rng.integers(0, len(pool), n) for n in sizes]
    rows = np.concatenate([pool[i] for i in ids])
    P = len(rows)
    C = moe.Config(T=P, d=d, E=len(sizes), k=1, H=128, n_shared=0, H_shared=0, dtype="bf16",
                   gating="softmax_topk", residual="none")
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x_perm = torch.from_numpy(rows).to(device="cuda", dtype=torch.bfloat16)
    rep_of, n_rep, ncond = moe.condense(C, x_perm, torch.from_numpy(offsets).cuda(), 1.0)
    torch.cuda.synchronize()
    expect = np.empty(P, np.int64)
    for e, ie in enumerate(ids):
        first = {}
        for s, v in enumerate(ie):
            expect[offsets[e] + s] = offsets[e] + first.setdefault(int(v), s)
    np.testing.assert_array_equal(_np(rep_of)[:P], expect)
    assert int(ncond.item()) == P - sum(len(set(ie.tolist())) for ie in ids)
    _status_ok(moe)


def test_condense_ragged_buckets(moe):
    """Empty, single-row and ragged buckets around the scan's 32-row groups and 160-row chunks.

    Half the rows repeat rows of a small pool, the rest are drawn fresh; at tau = 1 every
    row's representative is the first identical row of its bucket (closed form: distinct
    random rows are far from cosine 1).
    """
    rng = np.random.default_rng(11)
    d = 256
    sizes = [0, 1, 31, 32, 33, 0, 161, 353, 2049]
    pool = gen.round_to_bf16(rng.standard_normal((24, d)).astype(np.float32))
    rows, expect, distinct = [], [], 0
    base = 0
    for n in sizes:
        first = {}
        for s in range(n):
            if rng.random() < 0.5:
                key, v = int(rng.integers(0, len(pool))), None
            else:
                key, v = ("fresh", base + s), gen.round_to_bf16(rng.standard_normal(d).astype(np.float32))
            rows.append(pool[key] if v is None else v)
            expect.append(base + first.setdefault(key, s))
        distinct += len(first)
        base += n
    rows = np.stack(rows)
    P = len(rows)
    C = moe.Config(T=P, d=d, E=len(sizes), k=1, H=128, n_shared=0, H_shared=0, dtype="bf16",
                   gating="softmax_topk", residual="none")
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    x_perm = torch.from_numpy(rows).to(device="cuda", dtype=torch.bfloat16)
    rep_of, n_rep, ncond = moe.condense(C, x_perm, torch.from_numpy(offsets).cuda(), 1.0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(rep_of)[:P], np.array(expect))
    per_bucket = [len(set(expect[offsets[e]:offsets[e + 1]])) for e in range(len(sizes))]
    np.testing.assert_array_equal(_np(n_rep)[: len(sizes)], per_bucket)
    assert int(ncond.item()) == P - distinct
    _status_ok(moe)


def test_condense_chains_take_the_walk(moe):
    """Buckets where rows are decided in parallel and buckets that need the greedy walk.

    Chain buckets: runs of 45 rows 7 degrees apart on a circle, each run in its own plane of
    two coordinates (so rows of different runs are orthogonal), tau = cos 20 degrees: each row
    is similar to the two rows before it, and the earliest similar row of a row is then often
    itself condensed (no chaining through condensed rows), which only the walk decides.  Their
    sizes sit around the walk's 32-row groups and staged chunks.  Other buckets hold exact
    duplicates only (decided without the walk) or nothing.  Bit for bit against the oracle on
    the same stored rows; every similarity is at least 2e-3 from tau."""
    d = 256
    tau = math.cos(math.radians(20.0))
    sizes = [40, 0, 300, 1000, 7, 64, 2100]
    chains = {0, 2, 3, 5, 6}
    rng = np.random.default_rng(5)
    pool = gen.round_to_bf16(rng.standard_normal((8, d)).astype(np.float32))
    blocks = []
    for b, n in enumerate(sizes):
        if b in chains:
            rows = np.zeros((n, d), np.float32)
            i = np.arange(n)
            ang = np.radians(7.0 * (i % 45) + 3.0 * b)
            plane = i // 45
            rows[i, 2 * plane], rows[i, 2 * plane + 1] = np.cos(ang), np.sin(ang)
        else:
            rows = pool[rng.integers(0, len(pool), size=n)]
        blocks.append(gen.round_to_bf16(rows))
    rows = np.concatenate(blocks)
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    for b, n in enumerate(sizes):
        if b in chains and n:
            S = orc.cosine_similarity_matrix(rows[offsets[b]:offsets[b + 1]])
            assert np.min(np.abs(S[np.tril_indices(n, -1)] - tau)) > 2e-3
    ref = orc.condense(rows, offsets, tau)
    walked = [b for b in chains if sizes[b] and np.any(
        (ref[offsets[b]:offsets[b + 1]] != np.arange(offsets[b], offsets[b + 1])))]
    assert walked  # chains condense rows
    P = len(rows)
    C = moe.Config(T=P, d=d, E=len(sizes), k=1, H=128, n_shared=0, H_shared=0, dtype="bf16",
                   gating="softmax_topk", residual="none")
    x_perm = torch.from_numpy(rows).to(device="cuda", dtype=torch.bfloat16)
    rep_of, n_rep, ncond = moe.condense(C, x_perm, torch.from_numpy(offsets.astype(np.int32)).cuda(),
                                        tau)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_np(rep_of)[:P], ref)
    per_bucket = [int(np.sum(ref[offsets[b]:offsets[b + 1]] == np.arange(offsets[b], offsets[b + 1])))
                  for b in range(len(sizes))]
    np.testing.assert_array_equal(_np(n_rep)[: len(sizes)], per_bucket)
    assert int(ncond.item()) == P - sum(per_bucket)
    _status_ok(moe)


def test_condense_more_than_65536_pairs(moe):
    """The Luffy workload at 40000 tokens (80000 routed pairs, buckets of about 5000 rows):
    the scratch is sized by bucket rows (each token at most once per bucket), so condensation
    takes more pairs than the 65536 it was once limited to; bit for bit against the oracle."""
    cfg, inp, C, w, x, r = _setup(moe, "luffy_condense", T=40000)
    assert cfg.P > 65536
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    rep_of, n_rep, ncond = moe.condense(C, d["x_perm"], d["offsets"], cfg.taus[0])
    torch.cuda.synchronize()
    _, idx_o, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx_o, cfg.E)
    np.testing.assert_array_equal(_np(d["perm"])[: cfg.P], perm)
    ref = orc.condense(inp["x"][perm], offsets, cfg.taus[0])
    np.testing.assert_array_equal(_np(rep_of)[: cfg.P], ref)
    assert int(ncond.item()) == int(np.sum(ref != np.arange(cfg.P)))
    _status_ok(moe)


def test_condense_tau_above_one_is_identity(moe):
    cfg, inp, C, w, x, r = _setup(moe, "luffy_condense", T=2048)
    _, idx, _ = moe.route(C, x, w.W_r, w.router_bias)
    d = moe.dispatch(C, x, idx)
    for tau in (1.5, math.nan):
        rep_of, n_rep, ncond = moe.condense(C, d["x_perm"], d["offsets"], tau)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_np(rep_of)[: cfg.P], np.arange(cfg.P))
        assert int(ncond.item()) == 0
    base = moe.Layer(C, w)(x, r)
    same = moe.Layer(C, w, condense=True)(x, r, 1.5)
    torch.cuda.synchronize()
    assert torch.equal(base, same)


def test_condensed_layer_matches_the_step_by_step_calls(moe):
    """A condensing layer call has its dispatch form the slots' row norms and hashes (its
    condensation then skips the row-statistics pass); the step-by-step calls run that pass.
    The two must give the same representatives, so the same output bit for bit (full-size
    Luffy workload, both thresholds)."""
    cfg, inp, C, w, x, r = _setup(moe, "luffy_condense")
    layer = moe.Layer(C, w, condense=True)
    for tau in cfg.taus:
        n_layer = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = layer(x, r, tau, n_condensed_out=n_layer)
        _, idx, gate = moe.route(C, x, w.W_r, w.router_bias)
        d = moe.dispatch(C, x, idx)
        rep_of, _, n_steps = moe.condense(C, d["x_perm"], d["offsets"], tau)
        y, so = moe.expert_ffn(C, w, d["x_perm"], d["offsets"], rep_of=rep_of, x=x)
        ref = moe.combine(C, y, so, d["slot_of"], rep_of, gate, x=x, residual=r)
        torch.cuda.synchronize()
        assert int(n_layer.item()) == int(n_steps.item()) > 0
        assert torch.equal(out, ref), tau
    _status_ok(moe)


def test_condensed_layer_small(moe):
    cfg = gen.CONFIGS["luffy_condense"]
    for tau in cfg.taus:
        _layer_check(moe, "luffy_condense", T=SMALL_T["luffy_condense"], tau=tau)


# ------------------------------------------------------------------ limits of the boundary
@pytest.mark.parametrize("E,T,k", [(128, 16384, 1), (128, 16383, 1), (129, 16384, 1),
                                   (128, 65536, 1), (256, 8192, 8), (256, 50000, 1),
                                   (215, 58000, 1)])
def test_dispatch_large_rank_tables(moe, E, T, k):
    """The scatter scans the (expert, 1024-pair block) count table in its own shared memory
    up to 2048 entries: E = 128 with 16 blocks is exactly that limit (and 16383 tokens a
    ragged last block under it).  E = 129 with 16 blocks (2064 entries) is one expert past
    it, and 8192, 16384, 12544 and 12255 entries lie further past; those take the separate
    one-CTA table scan.  Skewed expert choices leave empty buckets; everything bit for bit."""
    d = 256
    rng = np.random.default_rng(T + k)
    pop = np.log(np.arange(1, E + 1) ** -1.1)[rng.permutation(E)]
    pop[rng.choice(E, 5, replace=False)] = -np.inf  # never chosen: empty buckets
    # k distinct experts per token, drawn with a Zipf-like popularity
    keys = pop[None, :] + rng.gumbel(size=(T, E))
    idx_np = np.argsort(-keys, axis=1)[:, :k].astype(np.int32)
    C = moe.Config(T=T, d=d, E=E, k=k, H=128, n_shared=0, H_shared=0, dtype="bf16",
                   gating="softmax_topk", residual="none")
    rows = gen.round_to_bf16(rng.standard_normal((T, d)).astype(np.float32))
    x = torch.from_numpy(rows).to(device="cuda", dtype=torch.bfloat16)
    out = moe.dispatch(C, x, torch.from_numpy(idx_np).cuda())
    torch.cuda.synchronize()
    counts, offsets, perm, slot_of = orc.dispatch(idx_np, E)
    assert (counts == 0).any()
    np.testing.assert_array_equal(_np(out["counts"]), counts)
    np.testing.assert_array_equal(_np(out["offsets"]), offsets)
    np.testing.assert_array_equal(_np(out["perm"])[: T * k], perm)
    np.testing.assert_array_equal(_np(out["slot_of"]), slot_of)
    assert torch.equal(out["x_perm"][: T * k], x.index_select(0, out["perm"][: T * k].long()))
    _status_ok(moe)
