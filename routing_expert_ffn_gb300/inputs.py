"""Seeded synthetic inputs for the routed-expert MoE layer.

This module only draws random numbers and lays them out; it computes nothing
of the layer itself (no logits, no routing, no similarity).  Both the CUDA
path and the fp64 oracle consume what it returns.

Every tensor comes from its own counter-keyed stream
``np.random.default_rng([seed, tensor_id, chunk])`` so that

* the first ``T'`` rows of a ``T``-token draw equal a ``T'``-token draw
  (token rows are drawn in order from one stream), and
* weights do not change when the token count changes.

bf16 tensors are returned as float32 arrays whose values are exactly
representable in bf16 (round-to-nearest-even of an fp32 draw), so either side
can consume them without a conversion step of its own.

Workload shapes follow the five MoE-layer shapes the routed-expert pages are
measured on: a tiny fp32 layer, a DeepSeek-V2-Lite-shaped layer, a
Qwen3-30B-A3B-shaped layer with Zipf-skewed expert popularity, a
Llama-4-Scout-shaped layer with FarSkip-Collective wiring (the MoE reads the
previous layer's full output, the residual base is the attention-partial
stream; FarSkip-Collective review, "Core claim"), and a layer whose tokens are
near-duplicates of a few centroids, for Luffy token condensation ("What
carries the argument" on the Luffy review page).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

# Stream ids, one per tensor kind.
_S_X, _S_WR, _S_BIAS, _S_WGU, _S_WDOWN, _S_WSGU, _S_WSDOWN, _S_RES, _S_CENT = range(9)


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    H: int
    n_shared: int
    H_shared: int
    dtype: str                 # "f32" or "bf16": activations, weights and outputs
    gating: str                # "softmax_topk" | "softmax_topk_renorm" | "sigmoid_topk"
    residual: str              # "none" | "input" | "external" | "input_plus_external"
    router_bias: str = "none"  # "none" | "zipf"
    zipf_s: float = 1.1
    x_kind: str = "gaussian"   # "gaussian" | "centroids" | "duplicates"
    residual_std: float = 1.0
    weight_std: float = 0.02
    copy_fraction: float = 0.0
    n_centroids: int = 0
    noise_rel: float = 0.0
    taus: tuple = field(default_factory=tuple)  # condensation thresholds the workload runs at
    seed: int = 1000

    @property
    def P(self) -> int:
        """Routed (token, expert) pairs."""
        return self.T * self.k

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)


def adaptive_tau_l_norm_minus_3() -> float:
    """Luffy's adaptive threshold evaluated at l_norm = -3, as a plain float.

    Luffy review, "What carries the argument": h_t = 1/(1+exp(l_norm)).  This
    is a workload constant (the second threshold the condensation workload
    runs at), not part of either implementation.
    """
    return 1.0 / (1.0 + math.exp(-3.0))


CONFIGS: dict[str, MoEConfig] = {
    "tiny_fp32": MoEConfig(
        name="tiny_fp32", T=256, d=128, E=8, k=2, H=256, n_shared=1, H_shared=256,
        dtype="f32", gating="softmax_topk", residual="external", residual_std=1.0,
        seed=1001),
    "dsv2_lite": MoEConfig(
        name="dsv2_lite", T=4096, d=2048, E=64, k=6, H=1408, n_shared=2, H_shared=1408,
        dtype="bf16", gating="softmax_topk", residual="input", seed=1002),
    "qwen3_30b_a3b": MoEConfig(
        name="qwen3_30b_a3b", T=8192, d=2048, E=128, k=8, H=768, n_shared=0, H_shared=0,
        dtype="bf16", gating="softmax_topk_renorm", residual="input", router_bias="zipf",
        zipf_s=1.1, seed=1003),
    "llama4_scout_farskip": MoEConfig(
        name="llama4_scout_farskip", T=8192, d=5120, E=16, k=1, H=8192, n_shared=1,
        H_shared=8192, dtype="bf16", gating="sigmoid_topk", residual="external",
        residual_std=0.5, seed=1004),
    "luffy_condense": MoEConfig(
        name="luffy_condense", T=16384, d=1024, E=16, k=2, H=4096, n_shared=0, H_shared=0,
        dtype="bf16", gating="softmax_topk", residual="input", x_kind="centroids",
        copy_fraction=0.4, n_centroids=512, noise_rel=0.02,
        taus=(0.95, adaptive_tau_l_norm_minus_3()), seed=1005),
}

# Decode-shaped layer: the DeepSeek-V2-Lite shapes and weights with one decode step of 64
# tokens, where the expert GEMMs are bound by streaming the weights from HBM
# (FarSkip-Collective review, Figure 7: decoding is memory-bandwidth bound).
CONFIGS["dsv2_lite_decode"] = replace(CONFIGS["dsv2_lite"], name="dsv2_lite_decode", T=64)

# Order used by tests and the bench: the small fp32 case first, then the bf16 shapes.
CONFIG_ORDER = ["tiny_fp32", "dsv2_lite", "qwen3_30b_a3b", "llama4_scout_farskip", "luffy_condense"]
DECODE_CONFIGS = ["dsv2_lite_decode"]


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([seed, *key])


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 value (ties to even), returned as fp32.  In place when possible."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    u += bias
    u &= np.uint32(0xFFFF0000)
    return a


def _normal(seed: int, key: tuple, shape: tuple, std: float) -> np.ndarray:
    a = _rng(seed, *key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _expert_stack(cfg: MoEConfig, stream: int, n: int, rows: int, cols: int,
                  bf16: bool, threads: int) -> np.ndarray:
    """[n, rows, cols] weights, one stream per expert, drawn in parallel."""
    out = np.empty((n, rows, cols), dtype=np.float32)

    def fill(e: int) -> None:
        w = _normal(cfg.seed, (stream, e), (rows, cols), cfg.weight_std)
        out[e] = round_to_bf16(w) if bf16 else w

    if n == 0:
        return out
    with ThreadPoolExecutor(max_workers=max(1, min(threads, n))) as ex:
        list(ex.map(fill, range(n)))
    return out


def _token_rows(cfg: MoEConfig) -> tuple[np.ndarray, np.ndarray]:
    """x [T, d] and the centroid label of every token (-1 for an i.i.d. token)."""
    T, d = cfg.T, cfg.d
    labels = np.full(T, -1, dtype=np.int32)
    x = _normal(cfg.seed, (_S_X, 0), (T, d), 1.0)
    if cfg.x_kind == "gaussian":
        return x, labels
    # Near-duplicate tokens: copies of unit centroids plus a noise vector whose
    # norm is noise_rel * ||c|| on average (per-component std noise_rel/sqrt(d)).
    cents = _centroids(cfg)
    r = _rng(cfg.seed, _S_CENT, 2)
    # Which tokens are copies is a property of the full-size workload, so that a
    # prefix of it is also a prefix of the full draw.
    T_full = CONFIGS[cfg.name].T if cfg.name in CONFIGS else T
    n_copy_full = int(round(cfg.copy_fraction * T_full))
    pos_full = np.sort(r.choice(T_full, size=n_copy_full, replace=False))
    cid_full = r.integers(0, cfg.n_centroids, size=n_copy_full)
    keep = pos_full < T
    pos, cid = pos_full[keep], cid_full[keep]
    noise = _normal(cfg.seed, (_S_CENT, 1), (n_copy_full, d), 1.0)[keep].astype(np.float64)
    if cfg.x_kind == "centroids":
        noise *= cfg.noise_rel / math.sqrt(d)
    else:  # "duplicates": exact copies of the centroid
        noise[:] = 0.0
    x[pos] = (cents[cid] + noise).astype(np.float32)
    labels[pos] = cid
    return x, labels


def make_inputs(cfg: MoEConfig, threads: int = 8) -> dict:
    """All inputs of one layer call, as numpy arrays.

    Keys: x [T,d], W_r [d,E] (fp32), bias [E] or None, W_gu [E,2H,d]
    (gate rows 0..H-1, up rows H..2H-1), W_down [E,d,H], Ws_gu [S,2Hs,d],
    Ws_down [S,d,Hs], residual [T,d] or None, labels [T] (centroid id or -1).
    """
    bf16 = cfg.dtype == "bf16"
    x, labels = _token_rows(cfg)
    if bf16:
        x = round_to_bf16(x)
    W_r = _normal(cfg.seed, (_S_WR, 0), (cfg.d, cfg.E), 1.0 / math.sqrt(cfg.d))
    bias = None
    if cfg.router_bias == "zipf":
        # Zipf(s) popularity p_i ~ i^-s over a seeded permutation of the experts;
        # the router adds ln p to the logits of the matching expert.
        r = _rng(cfg.seed, _S_BIAS, 0)
        perm = r.permutation(cfg.E)
        p = np.arange(1, cfg.E + 1, dtype=np.float64) ** (-cfg.zipf_s)
        p /= p.sum()
        bias = np.log(p[perm]).astype(np.float32)
    W_gu = _expert_stack(cfg, _S_WGU, cfg.E, 2 * cfg.H, cfg.d, bf16, threads)
    W_down = _expert_stack(cfg, _S_WDOWN, cfg.E, cfg.d, cfg.H, bf16, threads)
    Ws_gu = _expert_stack(cfg, _S_WSGU, cfg.n_shared, 2 * cfg.H_shared, cfg.d, bf16, threads)
    Ws_down = _expert_stack(cfg, _S_WSDOWN, cfg.n_shared, cfg.d, cfg.H_shared, bf16, threads)
    residual = None
    if cfg.residual in ("external", "input_plus_external"):
        residual = _normal(cfg.seed, (_S_RES, 0), (cfg.T, cfg.d), cfg.residual_std)
        if bf16:
            residual = round_to_bf16(residual)
    return dict(x=x, W_r=W_r, bias=bias, W_gu=W_gu, W_down=W_down, Ws_gu=Ws_gu,
                Ws_down=Ws_down, residual=residual, labels=labels)


def _centroids(cfg: MoEConfig) -> np.ndarray:
    r = _rng(cfg.seed, _S_CENT, 0)
    cents = r.standard_normal((cfg.n_centroids, cfg.d))
    return cents / np.linalg.norm(cents, axis=1, keepdims=True)


def redraw_token_rows(cfg: MoEConfig, x: np.ndarray, labels: np.ndarray,
                      rows: np.ndarray, attempt: int) -> None:
    """Replace the given token rows of x with fresh draws from a dedicated stream.

    An i.i.d. token gets a fresh N(0,1) row; a centroid copy keeps its centroid
    and gets fresh noise, so the token keeps its label.  An exact duplicate
    (no noise) cannot move away from its centroid's logits, so it becomes an
    i.i.d. token and its label is set to -1 in place.  Which rows to redraw
    is decided by the caller (the test harness moves tokens away from routing
    ties); this function only draws.
    """
    rows = np.asarray(rows, dtype=np.int64)
    if len(rows) == 0:
        return
    r = _rng(cfg.seed, _S_X, 1000 + attempt)
    fresh = r.standard_normal((len(rows), cfg.d)).astype(np.float64)
    if cfg.x_kind == "duplicates":
        labels[rows] = -1
    lab = labels[rows]
    if (lab >= 0).any():
        cents = _centroids(cfg)
        cp = lab >= 0
        scale = cfg.noise_rel / math.sqrt(cfg.d) if cfg.x_kind == "centroids" else 0.0
        fresh[cp] = cents[lab[cp]] + scale * fresh[cp]
    fresh = fresh.astype(np.float32)
    if cfg.dtype == "bf16":
        fresh = round_to_bf16(fresh)
    x[rows] = fresh
