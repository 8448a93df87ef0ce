"""Pins for the fp64 oracle: each check compares it with something other than itself.

Brute force on tiny inputs, library routines (sorted, scipy.special,
torch.nn.functional), closed forms, invariants and hand-derived worked
examples (tests/golden).  All run on the CPU.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import scipy.special as sp

from oracle import moe_oracle as orc
from routing_expert_ffn_gb300 import inputs as gen
from tests import harness

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ router
def _brute_topk(key_row, k):
    """The unique k-subset whose every member outranks every non-member, members ranked."""
    E = len(key_row)
    rank = lambda e: (float(key_row[e]), -e)  # larger is better; tie -> lower e
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if not rest or min(rank(e) for e in S) > max(rank(e) for e in rest):
            found.append(sorted(S, key=rank, reverse=True))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 2), (8, 8), (7, 6)])
def test_topk_matches_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # small integer logits make exact ties common
    l = rng.integers(-3, 4, size=(64, E)).astype(np.float64)
    idx = orc.select_topk(l, k)
    for t in range(64):
        assert list(idx[t]) == _brute_topk(l[t].astype(np.float32), k)


def test_topk_matches_brute_force_continuous():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((64, 8))
    idx = orc.select_topk(l, 3)
    for t in range(64):
        assert list(idx[t]) == _brute_topk(l[t].astype(np.float32), 3)


def test_topk_golden_ties():
    for c in _golden("topk_ties.json")["cases"]:
        idx = orc.select_topk(np.array([c["logits"]]), c["k"])
        assert list(idx[0]) == c["idx"]


def test_logits_against_python_loop():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 7))
    W = rng.standard_normal((7, 4))
    b = rng.standard_normal(4)
    l = orc.router_logits(x, W, b)
    for t in range(5):
        for e in range(4):
            ref = math.fsum(float(x[t, i]) * float(W[i, e]) for i in range(7)) + float(b[e])
            assert abs(l[t, e] - ref) < 1e-12


def test_gates_against_scipy():
    rng = np.random.default_rng(11)
    l = rng.standard_normal((32, 16)) * 3
    idx = orc.select_topk(l, 4)
    g = orc.gate_values(l, idx, "softmax_topk")
    full = sp.softmax(l, axis=1)
    np.testing.assert_allclose(g, np.take_along_axis(full, idx.astype(np.int64), 1), rtol=1e-13)
    assert np.all(g.sum(axis=1) < 1.0)
    gr = orc.gate_values(l, idx, "softmax_topk_renorm")
    sel = np.take_along_axis(l, idx.astype(np.int64), 1)
    np.testing.assert_allclose(gr, sp.softmax(sel, axis=1), rtol=1e-13)
    np.testing.assert_allclose(gr.sum(axis=1), 1.0, rtol=1e-14)
    gs = orc.gate_values(l, idx, "sigmoid_topk")
    np.testing.assert_allclose(gs, sp.expit(sel), rtol=1e-14)
    # softmax over all experts sums to one; sigmoid(l)+sigmoid(-l) = 1
    np.testing.assert_allclose(orc.gate_values(l, orc.select_topk(l, 16), "softmax_topk").sum(1), 1.0,
                               rtol=1e-13)


def test_gate_ratios_follow_logit_differences():
    l = np.array([[2.0, 0.0, 1.0, -1.0]])
    idx = orc.select_topk(l, 2)
    assert list(idx[0]) == [0, 2]
    g = orc.gate_values(l, idx, "softmax_topk_renorm")
    assert abs(g[0, 0] / g[0, 1] - math.e) < 1e-14
    assert abs(orc.gate_values(np.zeros((1, 3)), np.array([[0]]), "sigmoid_topk")[0, 0] - 0.5) < 1e-16


# ------------------------------------------------------------------ dispatch
def test_dispatch_golden():
    g = _golden("dispatch_small.json")
    counts, offsets, perm, slot_of = orc.dispatch(np.array(g["idx"]), g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm"]
    assert slot_of.tolist() == g["slot_of"]


@pytest.mark.parametrize("T,E,k", [(50, 6, 2), (200, 16, 4), (33, 5, 5), (1, 4, 1), (0, 4, 2)])
def test_dispatch_is_stable_sort_of_pairs(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.array([rng.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
    counts, offsets, perm, slot_of = orc.dispatch(idx, E)
    pairs = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(k))  # library sort
    assert perm.tolist() == [t for (_, t, _) in pairs]
    for s, (e, t, j) in enumerate(pairs):
        assert slot_of[t, j] == s
        assert offsets[e] <= s < offsets[e + 1]
    assert counts.sum() == T * k
    assert np.all(np.diff(offsets) >= 0) and offsets[0] == 0
    assert np.all(np.bincount(perm, minlength=T) == k) if T else True


def test_dispatch_skewed_load_of_zipf_workload():
    cfg, inp = harness.workload("qwen3_30b_a3b")
    l, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    counts, _, _, _ = orc.dispatch(idx, cfg.E)
    mean = cfg.T * cfg.k / cfg.E
    assert (counts == 0).sum() >= 1
    assert counts.max() > 4 * mean


# ------------------------------------------------------------------ experts
def test_silu_against_scipy_and_limits():
    z = np.array([-50.0, -3.0, -0.5, 0.0, 0.25, 2.0, 40.0, 800.0, -800.0])
    np.testing.assert_allclose(orc.silu(z), z * sp.expit(z), rtol=1e-14, atol=1e-300)
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(40.0) - 40.0) < 1e-15 * 40
    assert orc.silu(-800.0) == 0.0 or abs(orc.silu(-800.0)) < 1e-300


def test_swiglu_expert_against_torch_functional():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(5)
    d, H = 24, 40
    x = rng.standard_normal((9, d))
    W_gu = rng.standard_normal((2 * H, d)) * 0.3
    W_down = rng.standard_normal((d, H)) * 0.3
    got = orc.swiglu_expert(x, W_gu, W_down)
    tx, tgu, td = (torch.from_numpy(a) for a in (x, W_gu, W_down))
    ref = F.linear(F.silu(F.linear(tx, tgu[:H])) * F.linear(tx, tgu[H:]), td).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_swiglu_hidden_permutation_and_linearity():
    rng = np.random.default_rng(6)
    d, H = 8, 12
    x = rng.standard_normal((4, d))
    W_gu = rng.standard_normal((2 * H, d))
    W_down = rng.standard_normal((d, H))
    y = orc.swiglu_expert(x, W_gu, W_down)
    p = rng.permutation(H)
    W_gu_p = np.concatenate([W_gu[:H][p], W_gu[H:][p]])
    np.testing.assert_allclose(orc.swiglu_expert(x, W_gu_p, W_down[:, p]), y, rtol=1e-12)
    np.testing.assert_allclose(orc.swiglu_expert(x, W_gu, 2 * W_down), 2 * y, rtol=1e-14)
    # swapping gate and up changes the result (SiLU sits on the gate only)
    W_sw = np.concatenate([W_gu[H:], W_gu[:H]])
    assert np.max(np.abs(orc.swiglu_expert(x, W_sw, W_down) - y)) > 1e-3


def test_shared_experts_concatenation_identity():
    rng = np.random.default_rng(8)
    d, Hs = 6, 5
    x = rng.standard_normal((7, d))
    Ws_gu = rng.standard_normal((2, 2 * Hs, d))
    Ws_down = rng.standard_normal((2, d, Hs))
    two = orc.shared_experts(x, Ws_gu, Ws_down)
    cat_gu = np.concatenate([Ws_gu[0][:Hs], Ws_gu[1][:Hs], Ws_gu[0][Hs:], Ws_gu[1][Hs:]])
    cat_down = np.concatenate([Ws_down[0], Ws_down[1]], axis=1)
    np.testing.assert_allclose(two, orc.swiglu_expert(x, cat_gu, cat_down), rtol=1e-12)


# ------------------------------------------------------------------ combine / round trip
def test_round_trip_identity_experts_returns_x():
    """Dispatch, identity experts, combine with gates summing to one: out == x."""
    rng = np.random.default_rng(9)
    T, d, E, k = 40, 12, 6, 3
    x = rng.standard_normal((T, d))
    W_r = rng.standard_normal((d, E))
    l, idx, g = orc.route(x, W_r, None, k, "softmax_topk_renorm")
    counts, offsets, perm, slot_of = orc.dispatch(idx, E)
    x_perm = x[perm]
    y_pairs = x_perm[slot_of]              # identity expert on every dispatched row
    out = orc.combine(y_pairs, g, orc.residual_base(x, None, "none"))
    np.testing.assert_allclose(out, x, rtol=0, atol=1e-14)


def test_k_equals_E_with_identical_experts_is_one_dense_ffn():
    rng = np.random.default_rng(10)
    T, d, E, H = 16, 10, 4, 14
    x = rng.standard_normal((T, d))
    W_r = rng.standard_normal((d, E))
    W_gu1 = rng.standard_normal((2 * H, d)) * 0.4
    W_dn1 = rng.standard_normal((d, H)) * 0.4
    W_gu = np.repeat(W_gu1[None], E, axis=0)
    W_dn = np.repeat(W_dn1[None], E, axis=0)
    empty_gu, empty_dn = np.zeros((0, 2, d)), np.zeros((0, d, 1))
    r = orc.layer_forward(x, W_r, None, W_gu, W_dn, empty_gu, empty_dn, E, "softmax_topk_renorm",
                          residual_mode="none")
    np.testing.assert_allclose(r["out"], orc.swiglu_expert(x, W_gu1, W_dn1), rtol=1e-12, atol=1e-13)
    # softmax over all E with k = E also sums to one
    r2 = orc.layer_forward(x, W_r, None, W_gu, W_dn, empty_gu, empty_dn, E, "softmax_topk",
                           residual_mode="none")
    np.testing.assert_allclose(r2["out"], r["out"], rtol=1e-12, atol=1e-13)


def test_residual_modes_and_zero_experts():
    cfg, inp = harness.workload("tiny_fp32")
    args = (inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
            inp["Ws_down"], cfg.k, cfg.gating)
    ext = orc.layer_forward(*args, residual_mode="external", residual=inp["residual"])["out"]
    both = orc.layer_forward(*args, residual_mode="input_plus_external", residual=inp["residual"])["out"]
    none = orc.layer_forward(*args, residual_mode="none")["out"]
    np.testing.assert_allclose(both - ext, inp["x"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ext - none, inp["residual"], rtol=0, atol=1e-12)
    # zero routed-expert weights: out = residual + shared exactly
    z = orc.layer_forward(inp["x"], inp["W_r"], None, np.zeros_like(inp["W_gu"]), np.zeros_like(inp["W_down"]),
                          inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating,
                          residual_mode="external", residual=inp["residual"])["out"]
    shared = orc.shared_experts(inp["x"], inp["Ws_gu"], inp["Ws_down"])
    np.testing.assert_array_equal(z, inp["residual"].astype(np.float64) + shared)


def test_partial_activation_is_the_output_without_routed_experts():
    """FarSkip's partial activation: what the layer outputs when the routed experts
    contribute nothing, and independent of the routed experts' weights."""
    cfg, inp = harness.workload("tiny_fp32")
    common = dict(residual_mode="external", residual=inp["residual"])
    zero = orc.layer_forward(inp["x"], inp["W_r"], None, np.zeros_like(inp["W_gu"]),
                             np.zeros_like(inp["W_down"]), inp["Ws_gu"], inp["Ws_down"], cfg.k,
                             cfg.gating, **common)
    np.testing.assert_array_equal(zero["partial"], zero["out"])
    full = orc.layer_forward(inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"], inp["Ws_down"], cfg.k, cfg.gating, **common)
    np.testing.assert_array_equal(full["partial"], zero["partial"])
    assert np.max(np.abs(full["out"] - full["partial"])) > 1e-3
    # no shared experts and no residual: nothing is left
    none = orc.layer_forward(inp["x"], inp["W_r"], None, inp["W_gu"], inp["W_down"],
                             inp["Ws_gu"][:0], inp["Ws_down"][:0], cfg.k, cfg.gating,
                             residual_mode="none")
    assert not np.any(none["partial"])


def test_layer_subset_equals_full():
    cfg, inp = harness.workload("tiny_fp32")
    args = (inp["x"], inp["W_r"], inp["bias"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
            inp["Ws_down"], cfg.k, cfg.gating)
    full = orc.layer_forward(*args, residual_mode="external", residual=inp["residual"])
    sub = orc.layer_forward(*args, residual_mode="external", residual=inp["residual"],
                            tokens=[3, 77, 255, 0])
    np.testing.assert_allclose(sub["out"], full["out"][[3, 77, 255, 0]], rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------ condensation
def test_condense_golden_angles():
    for c in _golden("condense_angles.json")["cases"]:
        rows = harness.angle_rows(c["angles"], c["norms"])
        tau = c["tau"] if "tau" in c else math.cos(math.radians(c["tau_deg"]))
        assert orc.condense_bucket(rows, tau).tolist() == c["rep"], c["name"]


def test_condense_zero_rows():
    rows = np.array([[0.0, 0.0], [1.0, 0.0], [0.0, 0.0], [2.0, 0.0]])
    assert orc.condense_bucket(rows, 0.5).tolist() == [0, 1, 0, 1]
    assert orc.condense_bucket(rows, 1.0).tolist() == [0, 1, 0, 1]


def test_condense_tau_above_one_is_identity():
    cfg, inp = harness.workload("luffy_condense", T=1024)
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    for tau in (1.0000001, 2.0, float("nan")):
        np.testing.assert_array_equal(orc.condense(inp["x"][perm], offsets, tau), np.arange(len(perm)))


def test_exact_duplicates_collapse_at_tau_one():
    cfg, inp = harness.workload("luffy_condense", T=1024, x_kind="duplicates")
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    rep_of = orc.condense(inp["x"][perm], offsets, 1.0)
    lab = inp["labels"][perm]
    for e in range(cfg.E):
        a, b = offsets[e], offsets[e + 1]
        seen = {}
        for s in range(a, b):
            if lab[s] < 0:
                assert rep_of[s] == s            # i.i.d. tokens never reach similarity 1
            elif lab[s] in seen:
                assert rep_of[s] == seen[lab[s]]  # later copy -> first copy of the bucket
            else:
                seen[lab[s]] = s
                assert rep_of[s] == s


def _condensation_from_labels(cfg, inp):
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    lab = inp["labels"][perm]
    expected = 0
    for e in range(cfg.E):
        l = lab[offsets[e]:offsets[e + 1]]
        l = l[l >= 0]
        expected += len(l) - len(np.unique(l))
    return expected, offsets, perm, lab


def test_condensation_count_matches_centroid_labels():
    cfg, inp = harness.workload("luffy_condense", T=4096)
    expected, offsets, perm, lab = _condensation_from_labels(cfg, inp)
    for tau in cfg.taus:
        rep_of = orc.condense(inp["x"][perm], offsets, tau)
        condensed = rep_of != np.arange(len(perm))
        assert condensed.sum() == expected
        assert np.all(lab[condensed] >= 0)
        assert np.all(lab[rep_of[condensed]] == lab[condensed])
    # tau = 0.95 and tau = h_t(-3) give the same assignment, and so does the
    # [0,1]-normalised reading (1 + cos)/2 >= tau, i.e. cos >= 2 tau - 1.
    a = orc.condense(inp["x"][perm], offsets, cfg.taus[0])
    b = orc.condense(inp["x"][perm], offsets, cfg.taus[1])
    c = orc.condense(inp["x"][perm], offsets, 2 * cfg.taus[0] - 1)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


def test_similarity_margins_of_condensation_workload():
    cfg, inp = harness.workload("luffy_condense", T=4096)
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    xp = inp["x"][perm]
    for e in range(cfg.E):
        S = orc.cosine_similarity_matrix(xp[offsets[e]:offsets[e + 1]])
        off = ~np.eye(len(S), dtype=bool)
        for tau in cfg.taus:
            assert np.min(np.abs(S[off] - tau)) > 1e-3


def test_adaptive_tau_closed_forms():
    vals = {"0": 0.0, "ln 3": math.log(3), "-ln 3": -math.log(3), "ln 9": math.log(9)}
    fr = {"1/2": 0.5, "1/4": 0.25, "3/4": 0.75, "1/10": 0.1}
    for c in _golden("adaptive_tau.json")["cases"]:
        assert abs(orc.adaptive_tau(vals[c["l_norm"]]) - fr[c["h"]]) < 1e-15
    # decreasing in l_norm, in (0, 1)
    ls = np.linspace(-10, 10, 101)
    h = orc.adaptive_tau(ls)
    assert np.all(np.diff(h) < 0) and np.all((h > 0) & (h < 1))
    assert abs(orc.adaptive_tau(-3.0) - gen.adaptive_tau_l_norm_minus_3()) < 1e-16


# ------------------------------------------------------------------ full layer with condensation
def test_condensed_pairs_reuse_representative_output():
    cfg, inp = harness.workload("luffy_condense", T=512)
    small = dict(inp)
    H = 64
    small["W_gu"] = inp["W_gu"][:, np.r_[0:H, cfg.H:cfg.H + H], :]
    small["W_down"] = inp["W_down"][:, :, :H]
    args = (inp["x"], inp["W_r"], inp["bias"], small["W_gu"], small["W_down"], inp["Ws_gu"],
            inp["Ws_down"], cfg.k, cfg.gating)
    r = orc.layer_forward(*args, residual_mode="none", tau=cfg.taus[0])
    plain = orc.layer_forward(*args, residual_mode="none")
    assert (r["rep_of"] != np.arange(len(r["perm"]))).sum() > 0
    # recompute by hand: each pair uses the representative token's row
    for t in range(0, cfg.T, 37):
        acc = np.zeros(cfg.d)
        for j in range(cfg.k):
            e = r["idx"][t, j]
            src = r["perm"][r["rep_of"][r["slot_of"][t, j]]]
            acc += r["gates"][t, j] * orc.swiglu_expert(inp["x"][src][None], small["W_gu"][e],
                                                        small["W_down"][e])[0]
        np.testing.assert_allclose(r["out"][t], acc, rtol=1e-12, atol=1e-14)
    # tokens that are their own representative get the plain result
    own = np.all(r["rep_of"][r["slot_of"]] == r["slot_of"], axis=1)
    np.testing.assert_allclose(r["out"][own], plain["out"][own], rtol=1e-13, atol=1e-15)


def test_conditioned_workloads_have_routing_margins():
    for name in ("tiny_fp32", "luffy_condense"):
        cfg, inp = harness.workload(name, T=2048 if name == "luffy_condense" else None)
        assert len(harness.near_tie_tokens(inp, cfg.k)) == 0


# ------------------------------------------------------------------ backward
def _fd_case(gating, residual_mode, tau=None, x_kind=None, T=32):
    if x_kind is None:
        cfg, inp = harness.workload("tiny_fp32", T)
    else:
        # near-duplicate tokens: half the tokens are copies of 4 centroids plus 2 % noise
        from dataclasses import replace
        cfg = replace(gen.CONFIGS["tiny_fp32"], name="tiny_fp32_near_dup", T=T, x_kind=x_kind,
                      copy_fraction=0.5, n_centroids=4, noise_rel=0.02)
        inp = harness.condition(cfg, gen.make_inputs(cfg))
    rng = np.random.default_rng(7)
    E = cfg.E
    bias = rng.standard_normal(E) * 0.3 if gating != "sigmoid_topk" else rng.standard_normal(E) * 0.1
    params = dict(x=inp["x"].astype(np.float64), W_r=inp["W_r"].astype(np.float64), bias=bias,
                  W_gu=inp["W_gu"].astype(np.float64), W_down=inp["W_down"].astype(np.float64),
                  Ws_gu=inp["Ws_gu"].astype(np.float64), Ws_down=inp["Ws_down"].astype(np.float64),
                  residual=inp["residual"].astype(np.float64))
    d_out = rng.standard_normal((T, cfg.d))
    return cfg, params, d_out


def _loss(cfg, p, d_out, gating, residual_mode, tau):
    f = orc.layer_forward(p["x"], p["W_r"], p["bias"], p["W_gu"], p["W_down"], p["Ws_gu"],
                          p["Ws_down"], cfg.k, gating, residual_mode=residual_mode,
                          residual=p["residual"], tau=tau)
    return float(np.sum(d_out * f["out"])), f


@pytest.mark.parametrize("gating,residual_mode", [("softmax_topk", "input"),
                                                  ("softmax_topk_renorm", "external"),
                                                  ("sigmoid_topk", "input_plus_external")])
def test_backward_matches_finite_differences(gating, residual_mode):
    """Every gradient against the central difference of the forward's loss <d_out, out> along
    a random direction (h = 1e-6 moves no routing decision on the margin-conditioned inputs)."""
    cfg, p, d_out = _fd_case(gating, residual_mode)
    g = orc.layer_backward(p["x"], p["W_r"], p["bias"], p["W_gu"], p["W_down"], p["Ws_gu"],
                           p["Ws_down"], cfg.k, gating, d_out, residual_mode=residual_mode,
                           residual=p["residual"])
    grads = dict(x=g["dx"], W_r=g["dW_r"], bias=g["d_bias"], W_gu=g["dW_gu"], W_down=g["dW_down"],
                 Ws_gu=g["dWs_gu"], Ws_down=g["dWs_down"], residual=g["d_residual"])
    rng = np.random.default_rng(11)
    h = 1e-6
    _, f0 = _loss(cfg, p, d_out, gating, residual_mode, None)
    for name, grad in grads.items():
        v = rng.standard_normal(p[name].shape)
        plus = dict(p); plus[name] = p[name] + h * v
        minus = dict(p); minus[name] = p[name] - h * v
        lp, fp = _loss(cfg, plus, d_out, gating, residual_mode, None)
        lm, fm = _loss(cfg, minus, d_out, gating, residual_mode, None)
        assert np.array_equal(fp["idx"], f0["idx"]) and np.array_equal(fm["idx"], f0["idx"])
        fd = (lp - lm) / (2 * h)
        an = 0.0 if grad is None else float(np.sum(grad * v))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (gating, name, fd, an)


def test_backward_with_condensation_matches_finite_differences():
    """Near-duplicate tokens condensed at tau = 0.95: the finite difference of the forward
    (which feeds a condensed pair its representative's input) agrees with the gradient,
    including for the condensed tokens' own inputs."""
    cfg, p, d_out = _fd_case("softmax_topk", "input", x_kind="centroids", T=48)
    tau = 0.95
    g = orc.layer_backward(p["x"], p["W_r"], p["bias"], p["W_gu"], p["W_down"], p["Ws_gu"],
                           p["Ws_down"], cfg.k, "softmax_topk", d_out, residual_mode="input",
                           tau=tau)
    assert np.any(g["rep_of"] != np.arange(len(g["rep_of"])))  # something is condensed
    rng = np.random.default_rng(3)
    h = 1e-7
    _, f0 = _loss(cfg, p, d_out, "softmax_topk", "input", tau)
    for name, grad in dict(x=g["dx"], W_gu=g["dW_gu"], W_down=g["dW_down"], W_r=g["dW_r"]).items():
        v = rng.standard_normal(p[name].shape)
        plus = dict(p); plus[name] = p[name] + h * v
        minus = dict(p); minus[name] = p[name] - h * v
        lp, fp = _loss(cfg, plus, d_out, "softmax_topk", "input", tau)
        lm, fm = _loss(cfg, minus, d_out, "softmax_topk", "input", tau)
        assert np.array_equal(fp["rep_of"], f0["rep_of"]) and np.array_equal(fm["rep_of"], f0["rep_of"])
        fd = (lp - lm) / (2 * h)
        assert abs(fd - float(np.sum(grad * v))) <= 1e-5 * max(1.0, abs(fd)), name


def test_backward_condensed_token_gets_no_expert_gradient():
    """With W_r = 0 (no router gradient reaches x) and no shared experts, a token whose every
    pair is condensed onto another token's slot receives only the residual's gradient."""
    cfg, p, d_out = _fd_case("softmax_topk", "input", x_kind="centroids", T=48)
    W_r = np.zeros_like(p["W_r"])
    g = orc.layer_backward(p["x"], W_r, None, p["W_gu"], p["W_down"], p["Ws_gu"][:0],
                           p["Ws_down"][:0], cfg.k, "softmax_topk", d_out, residual_mode="input",
                           tau=0.95)
    counts, offsets, perm, slot_of = orc.dispatch(g["idx"], cfg.E)
    condensed_all = [t for t in range(d_out.shape[0])
                     if all(g["rep_of"][slot_of[t, j]] != slot_of[t, j] for j in range(cfg.k))]
    assert condensed_all, "the near-duplicate workload condenses some token in every bucket it visits"
    checked = 0
    for t in condensed_all:
        own = [perm[g["rep_of"][s]] for s in range(len(perm)) if perm[g["rep_of"][s]] == t]
        if not own:  # t is nobody's representative
            np.testing.assert_array_equal(g["dx"][t], d_out[t])
            checked += 1
    assert checked > 0


def test_backward_dense_case_matches_autograd():
    """k = E identical experts with renormalised gates is one dense SwiGLU FFN: its input
    gradient and the summed expert weight gradients equal torch autograd's (float64)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    cfg, inp = harness.workload("tiny_fp32", 40)
    E = 4
    x = inp["x"].astype(np.float64)
    W_gu = np.repeat(inp["W_gu"][:1], E, axis=0).astype(np.float64)
    W_down = np.repeat(inp["W_down"][:1], E, axis=0).astype(np.float64)
    W_r = inp["W_r"][:, :E].astype(np.float64)
    d_out = np.random.default_rng(5).standard_normal(x.shape)
    g = orc.layer_backward(x, W_r, None, W_gu, W_down, np.zeros((0, 2, cfg.d)),
                           np.zeros((0, cfg.d, 1)), E, "softmax_topk_renorm", d_out,
                           residual_mode="none")
    H = cfg.H
    xt = torch.tensor(x, requires_grad=True)
    wg = torch.tensor(W_gu[0], requires_grad=True)
    wd = torch.tensor(W_down[0], requires_grad=True)
    y = F.linear(F.silu(F.linear(xt, wg[:H])) * F.linear(xt, wg[H:]), wd)
    (y * torch.tensor(d_out)).sum().backward()
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dW_gu"].sum(axis=0), wg.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dW_down"].sum(axis=0), wd.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dW_r"], 0.0, atol=1e-9)


# ------------------------------------------------------------------ condensation with history
def _history_block(angles, buckets):
    """x_perm, offsets, perm of one block whose buckets list token indices in slot order."""
    rows = harness.angle_rows(angles, [1.0] * len(angles))
    perm = np.array([t for b in buckets for t in b], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum([len(b) for b in buckets])]).astype(np.int64)
    return rows[perm], offsets, perm


def test_condense_history_golden_two_blocks():
    g = _golden("condense_history.json")
    for c in g["cases"]:
        hist = None
        for bi, blk in enumerate(c["blocks"]):
            xp, offsets, perm = _history_block(blk["angles"], blk["buckets"])
            rep_of, hist = orc.condense_with_history(xp, offsets, perm, g["tau"], g["s1"], g["s2"], hist)
            got = [[int(perm[rep_of[s]]) for s in range(offsets[e], offsets[e + 1])]
                   for e in range(len(blk["buckets"]))]
            assert got == blk["rep"], (c["name"], bi)
            want = {(u, t): cls for u, t, cls in blk["history"]}
            assert hist == want, (c["name"], bi)


def test_condense_history_disabled_is_plain_condensation():
    """S1 > 1 and S2 < -1 classify nothing, so every block is plain condensation and the
    history stays empty; an empty history with S1 = 0.8, S2 = 0.2 also leaves the first
    block's assignment unchanged."""
    cfg, inp = harness.workload("luffy_condense", T=512)
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    xp = inp["x"][perm]
    plain = orc.condense(xp, offsets, 0.95)
    rep, hist = orc.condense_with_history(xp, offsets, perm, 0.95, 2.0, -2.0, None)
    np.testing.assert_array_equal(rep, plain)
    assert hist == {}
    rep2, hist2 = orc.condense_with_history(xp, offsets, perm, 0.95, 2.0, -2.0, hist)
    np.testing.assert_array_equal(rep2, plain)
    rep3, hist3 = orc.condense_with_history(xp, offsets, perm, 0.95, 0.8, 0.2, {})
    np.testing.assert_array_equal(rep3, plain)
    assert len(hist3) > 0


def test_condense_history_classes_of_first_block():
    """From an empty history the classes are exactly the co-routed pairs whose cosine (here
    from the 2-D angle difference, not from the oracle's similarity matrix) is >= S1 or <= S2."""
    rng = np.random.default_rng(3)
    angles = rng.uniform(0, 360, size=24)
    buckets = [sorted(rng.choice(24, size=9, replace=False).tolist()) for _ in range(3)]
    xp, offsets, perm = _history_block(angles, buckets)
    _, hist = orc.condense_with_history(xp, offsets, perm, 0.95, 0.8, 0.2, None)
    want = {}
    for b in buckets:
        for i in range(len(b)):
            for j in range(i):
                c = math.cos(math.radians(angles[b[i]] - angles[b[j]]))
                if abs(c - 0.8) < 1e-6 or abs(c - 0.2) < 1e-6:
                    continue
                if c >= 0.8:
                    want[(b[j], b[i])] = True
                elif c <= 0.2:
                    want[(b[j], b[i])] = False
    assert hist == want


def test_condense_history_repeated_block_keeps_assignment():
    """The same block twice (same rows, same buckets).  On this workload every co-routed
    cosine lies below S2 or at or above tau (i.i.d. rows are near orthogonal, copies of a
    centroid near 1; checked here), so each class the first block records says what the
    cosine says: the second block repeats the assignment and its history is the first's."""
    cfg, inp = harness.workload("luffy_condense", T=512)
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    _, offsets, perm, _ = orc.dispatch(idx, cfg.E)
    xp = inp["x"][perm]
    for e in range(cfg.E):
        S = orc.cosine_similarity_matrix(xp[offsets[e]:offsets[e + 1]])
        low = S[np.tril_indices(len(S), -1)]
        assert np.all((low <= 0.2) | (low >= 0.95))
    rep1, h1 = orc.condense_with_history(xp, offsets, perm, 0.95, 0.8, 0.2, None)
    rep2, h2 = orc.condense_with_history(xp, offsets, perm, 0.95, 0.8, 0.2, h1)
    np.testing.assert_array_equal(rep1, rep2)
    assert h1 == h2
    np.testing.assert_array_equal(rep1, orc.condense(xp, offsets, 0.95))
