"""fp64 CPU oracle for the routed-expert path of a Mixture-of-Experts layer.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA path computes.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it.  It shares no code with the CUDA path (no kernels,
helpers, tables or pre/post-processing) and imports nothing from the package.

Sources.  The pages that define the subject are the Pith reviews of
"FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
Models" (arXiv 2511.11505) and of "Communication-Efficient Sparsely-Activated
Model Training via Sequence Migration and Token Condensation" (Luffy, arXiv
2411.15419).  Neither prints the router, the expert or the combine formula;
they describe the layer as router -> Dispatch -> routed experts -> Combine,
with a shared expert, the FarSkip residual wiring and Luffy's in-bucket
token condensation.  Where they are silent this oracle takes the plainest
reading (listed with each function).

Arithmetic.  Everything is float64 on the exact values of the stored inputs.
Where floating point decides an integer (top-k selection, sim >= tau) the
decision is taken in float32, the precision the CUDA kernels decide in: the
fp64 value is rounded to float32 and compared.

Pins.  Every function here is checked by ``tests/test_oracle_pins.py``
against something other than itself: brute-force enumeration on tiny inputs,
library routines (``np.lexsort``/``sorted``, ``scipy.special``,
``torch.nn.functional``), closed forms, invariants (round trip with identity
experts, k = E with identical experts = one dense FFN, shared-expert
concatenation, tau > 1 no-op, exact duplicates at tau = 1), hand-derived
worked examples under ``tests/golden/`` and the centroid labels of the
condensation workload.
"""
from __future__ import annotations

import numpy as np

GATINGS = ("softmax_topk", "softmax_topk_renorm", "sigmoid_topk")
RESIDUALS = ("none", "input", "external", "input_plus_external")


# --------------------------------------------------------------------------- router
def router_logits(x, W_r, bias=None):
    """l[t, e] = sum_i x[t, i] * W_r[i, e] (+ bias[e]), float64.

    The pages name the router only through its cited prior work (the
    sparsely-gated MoE layer and Switch Transformers in the FarSkip-Collective
    review's reference list).  Reading: a linear router with no noise, no
    temperature and no capacity limit; a per-expert bias, when present, is
    added to every token's logits before selection and gating.
    """
    l = np.asarray(x, dtype=np.float64) @ np.asarray(W_r, dtype=np.float64)
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def select_topk(logits, k):
    """idx[t, :] = the k experts with the largest logits, largest first.

    Decided in float32 (the CUDA router's precision): the key is float32(l);
    experts are ordered by (-key, e), so an exact tie goes to the lower expert
    index.  Selecting on logits equals selecting on softmax or sigmoid
    probabilities, both being increasing in l.
    """
    key = np.asarray(logits, dtype=np.float64).astype(np.float32)
    order = np.argsort(-key, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :k]).astype(np.int32)


def gate_values(logits, idx, gating):
    """Combine weights of the selected experts, float64.

    * softmax_topk:        g = softmax over all E logits, taken at the k selected
                            experts (not renormalised: the k gates sum to < 1).
    * softmax_topk_renorm: g = softmax over the k selected logits only.
    * sigmoid_topk:        g = 1 / (1 + exp(-l_e)) of each selected expert.
    """
    l = np.asarray(logits, dtype=np.float64)
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    if gating == "softmax_topk":
        m = l.max(axis=1, keepdims=True)
        p = np.exp(l - m)
        p /= p.sum(axis=1, keepdims=True)
        return np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if gating == "softmax_topk_renorm":
        m = sel.max(axis=1, keepdims=True)
        p = np.exp(sel - m)
        return p / p.sum(axis=1, keepdims=True)
    if gating == "sigmoid_topk":
        return 1.0 / (1.0 + np.exp(-sel))
    raise ValueError(f"unknown gating {gating!r}")


def route(x, W_r, bias, k, gating):
    """Router step: (logits, idx, gates)."""
    l = router_logits(x, W_r, bias)
    idx = select_topk(l, k)
    return l, idx, gate_values(l, idx, gating)


# --------------------------------------------------------------------------- dispatch
def dispatch(idx, E):
    """Expert-contiguous permutation of the routed (token, expert) pairs.

    The single-GPU analogue of the expert-parallel Dispatch all-to-all
    (FarSkip-Collective review, "The reading" and the overlap condition of
    Eq. 9 in the ledger).  Bucket e is the list of tokens t whose selection
    contains e, in ascending t.  Buckets are laid end to end in expert order.

    Returns counts [E], offsets [E+1] (exclusive prefix of counts),
    perm [T*k] (slot -> token) and slot_of [T, k] (pair -> slot).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    perm = np.empty(T * k, dtype=np.int64)
    slot_of = np.full((T, k), -1, dtype=np.int64)
    for e in range(E):
        hit = idx == e
        tokens = np.nonzero(hit.any(axis=1))[0]            # ascending token index
        j = np.argmax(hit[tokens], axis=1)                  # the pair's position in idx[t]
        base = offsets[e]
        slot_of[tokens, j] = base + np.arange(len(tokens))
        perm[base:base + len(tokens)] = tokens
        counts[e] = len(tokens)
        offsets[e + 1] = base + len(tokens)
    return counts, offsets, perm, slot_of


# --------------------------------------------------------------------------- condensation
def cosine_similarity_matrix(rows):
    """sim[i, j] = cos(x_i, x_j) on float64 values, clamped to [-1, 1].

    The Luffy review leaves "normalized cosine similarity" undefined (referee
    minor comment 2).  Reading: the raw cosine of the dispatched input rows;
    bitwise-identical rows have similarity exactly 1 (including two zero
    rows); a zero row is otherwise dissimilar (similarity 0) to everything.
    """
    X = np.asarray(rows, dtype=np.float64)
    n = np.sqrt((X * X).sum(axis=1))
    G = X @ X.T
    with np.errstate(divide="ignore", invalid="ignore"):
        S = G / np.outer(n, n)
    zero = n == 0.0
    S[zero, :] = 0.0
    S[:, zero] = 0.0
    S = np.clip(S, -1.0, 1.0)
    # exact duplicates
    groups: dict[bytes, list[int]] = {}
    raw = np.ascontiguousarray(rows)
    for i in range(raw.shape[0]):
        groups.setdefault(raw[i].tobytes(), []).append(i)
    for members in groups.values():
        if len(members) > 1:
            m = np.asarray(members)
            S[np.ix_(m, m)] = 1.0
    return S


def condense_bucket(rows, tau):
    """Greedy in-bucket representative assignment.  rep[j] = local index of j's representative.

    Luffy review, "What carries the argument": tokens routed to the same
    expert are compared (only co-routed tokens, via expert activation), similar
    tokens are grouped in a token graph, and one representative's expert
    output is reused for the group; referee major comment 1: a condensed
    token's forward uses its representative's expert output.

    Reading: walk the bucket in slot order keeping the set R of
    representatives; slot j is condensed onto the earliest r in R with
    sim(x_j, x_r) >= tau, otherwise j joins R (and is its own
    representative).  Comparisons are against representatives only (no
    chaining through condensed tokens).  The comparison is taken in float32.
    """
    n = len(rows)
    rep = np.arange(n, dtype=np.int64)
    if n == 0:
        return rep
    S32 = cosine_similarity_matrix(rows).astype(np.float32)
    tau32 = np.float32(tau)
    reps = np.empty(0, dtype=np.int64)
    for j in range(n):
        hits = np.nonzero(S32[j, reps] >= tau32)[0] if len(reps) else ()
        if len(hits):
            rep[j] = reps[hits[0]]
        else:
            reps = np.append(reps, j)
    return rep


def condense(x_perm, offsets, tau):
    """rep_of[slot] = the representative slot (global slot index) of every routed slot.

    tau > 1 (or NaN) disables condensation: rep_of is the identity.
    """
    P = int(offsets[-1])
    rep_of = np.arange(P, dtype=np.int64)
    if not (tau <= 1.0):
        return rep_of
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            rep_of[a:b] = a + condense_bucket(x_perm[a:b], tau)
    return rep_of


def condense_with_history(x_perm, offsets, perm, tau, s1, s2, history=None):
    """Condensation that reuses the previous block's similarity of a token pair.

    Luffy review: the fast similarity measurement "uses expert activation and
    historical similarity to skip most pair-wise comparisons" ("What carries the
    argument"); the ledger's free parameters S1 and S2 (e.g. 0.8 and 0.2) decide
    which pairs are classified similar or dissimilar without a cosine, and its
    domain assumption is that historical similarity persists across consecutive
    blocks (Figure 7).

    Reading (the pages give no more): the history is a set of token pairs, each
    with a class, carried from one block (one call) to the next and keyed by the
    two token indices, so it does not depend on which buckets the tokens share.
    At this block every pair of slots in one bucket (expert activation: only
    co-routed tokens are compared) is decided as follows, for the token pair
    (u, t) of its two slots:

    * the pair is in the history: its class decides (similar = the pair counts
      as sim >= tau; dissimilar = it does not), no cosine is taken;
    * otherwise: sim(x_u, x_t) >= tau, with sim as in ``cosine_similarity_matrix``,
      decided in float32.

    The greedy representative walk is then the one of ``condense_bucket`` on
    these decisions.  The history handed to the next block holds exactly the
    pairs compared at this block: a pair decided by its history keeps its class;
    a pair with a cosine gets class similar if float32(sim) >= float32(s1),
    dissimilar if float32(sim) <= float32(s2), and no entry otherwise.  Pairs not
    compared at this block (no shared bucket) are not carried on.

    history: dict {(u, t): bool} with u < t token indices, True = similar; None
    or {} for the first block.  Returns (rep_of [P], new_history dict).
    """
    P = int(offsets[-1])
    rep_of = np.arange(P, dtype=np.int64)
    hist = {} if history is None else history
    new_hist: dict = {}
    tau32, s1_32, s2_32 = np.float32(tau), np.float32(s1), np.float32(s2)
    perm = np.asarray(perm)
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        n = b - a
        if n == 0:
            continue
        S32 = cosine_similarity_matrix(x_perm[a:b]).astype(np.float32)
        toks = perm[a:b]
        similar = np.zeros((n, n), dtype=bool)
        for i in range(n):
            for j in range(i):
                u, t = sorted((int(toks[j]), int(toks[i])))
                if (u, t) in hist:
                    cls = bool(hist[(u, t)])
                    similar[i, j] = cls
                    new_hist[(u, t)] = cls
                else:
                    similar[i, j] = bool(S32[i, j] >= tau32)
                    if S32[i, j] >= s1_32:
                        new_hist[(u, t)] = True
                    elif S32[i, j] <= s2_32:
                        new_hist[(u, t)] = False
        reps: list[int] = []
        for i in range(n):
            hit = next((r for r in reps if similar[i, r]), None)
            if hit is None:
                reps.append(i)
            else:
                rep_of[a + i] = a + hit
    return rep_of, new_hist


def adaptive_tau(l_norm):
    """Luffy's adaptive condensation threshold h_t = 1 / (1 + exp(l_norm)).

    Luffy review, "What carries the argument" (Eq. 2); referee minor comment 1
    notes the paper's wording calls it exponential while the form is logistic.
    l_norm is the normalised loss decrease of the previous iteration; its
    normalisation is not given, so it is taken as an input.
    """
    return 1.0 / (1.0 + np.exp(np.float64(l_norm)))


# --------------------------------------------------------------------------- experts
def silu(z):
    """SiLU(z) = z / (1 + exp(-z)), float64."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_expert(xrows, W_gu, W_down):
    """One SwiGLU expert: W_down (SiLU(W_gate x) * (W_up x)), no biases.

    W_gu is [2H, d] with the gate projection in rows 0..H-1 and the up
    projection in rows H..2H-1; W_down is [d, H].  The pages name "routed
    experts" and a "shared expert" without printing the expert; the SwiGLU
    form is the layer statement's.
    """
    X = np.asarray(xrows, dtype=np.float64)
    W = np.asarray(W_gu, dtype=np.float64)
    H = W.shape[0] // 2
    g = X @ W[:H].T
    u = X @ W[H:].T
    return (silu(g) * u) @ np.asarray(W_down, dtype=np.float64).T


def shared_experts(x, Ws_gu, Ws_down):
    """Sum of the shared experts' outputs, each applied to every token."""
    out = np.zeros((x.shape[0], Ws_down.shape[1] if len(Ws_down) else x.shape[1]))
    for s in range(len(Ws_gu)):
        out += swiglu_expert(x, Ws_gu[s], Ws_down[s])
    return out


def residual_base(x, residual, mode):
    """The residual the combine adds, per FarSkip-Collective wiring.

    FarSkip-Collective review, "Core claim": the MoE sub-block reads the
    previous layer's full output (x here), not the post-attention stream;
    referee minor comment 1: Eq. 6 needs the base residual o_0 added once.
    Modes: none -> 0; input -> x (standard wiring); external -> r (the
    attention-partial stream, given separately); input_plus_external -> x + r.
    """
    x = np.asarray(x, dtype=np.float64)
    if mode == "none":
        return np.zeros_like(x)
    if mode == "input":
        return x.copy()
    r = np.asarray(residual, dtype=np.float64)
    if mode == "external":
        return r.copy()
    if mode == "input_plus_external":
        return x + r
    raise ValueError(f"unknown residual mode {mode!r}")


def combine(y_pairs, gates, base, shared=None):
    """out[t] = base[t] + shared[t] + sum_j gates[t, j] * y_pairs[t, j].

    The single-GPU analogue of the Combine all-to-all followed by the gated
    sum of the k expert outputs and the shared expert (FarSkip-Collective
    review, "Core claim": the partial activation includes the shared-expert
    output).
    """
    out = np.asarray(base, dtype=np.float64).copy()
    if shared is not None:
        out += shared
    out += np.einsum("tk,tkd->td", np.asarray(gates, np.float64), np.asarray(y_pairs, np.float64))
    return out


# --------------------------------------------------------------------------- layer
def layer_forward(x, W_r, bias, W_gu, W_down, Ws_gu, Ws_down, k, gating,
                  residual_mode="input", residual=None, tau=None, tokens=None):
    """The whole routed-expert layer on the host.

    Steps: route (logits, top-k, gates) -> dispatch -> optional condensation
    (tau <= 1) -> per (token, expert) pair the expert's SwiGLU output on the
    input row of the pair's representative -> out = base + shared + gated sum.

    ``tokens`` restricts the expert and combine work to a subset of tokens
    (routing, dispatch and condensation always run over all T tokens, since
    slots and representatives depend on every token).  Returns a dict with
    logits, idx, gates, counts, offsets, perm, slot_of, rep_of, tokens, out,
    partial.

    ``partial`` = base + shared: FarSkip-Collective review, "Core claim" -- the
    attention sub-block under FarSkip wiring reads a partial activation that
    already holds the shared-expert output but none of the routed experts.
    """
    x = np.asarray(x)
    T = x.shape[0]
    E = W_gu.shape[0]
    logits, idx, g = route(x, W_r, bias, k, gating)
    counts, offsets, perm, slot_of = dispatch(idx, E)
    use_tau = tau is not None and tau <= 1.0
    if use_tau:
        rep_of = condense(x[perm], offsets, tau)
    else:
        rep_of = np.arange(len(perm), dtype=np.int64)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    d = x.shape[1]
    y_pairs = np.zeros((len(tok), k, d))
    # source token of every selected pair: the token of the pair's representative slot
    src = perm[rep_of[slot_of[tok]]]                         # [n, k]
    sel = idx[tok]
    for e in range(E):
        where = np.nonzero(sel == e)
        if len(where[0]) == 0:
            continue
        y_pairs[where[0], where[1]] = swiglu_expert(x[src[where]], W_gu[e], W_down[e])
    shared = shared_experts(x[tok], Ws_gu, Ws_down) if len(Ws_gu) else None
    base = residual_base(x[tok], None if residual is None else residual[tok], residual_mode)
    out = combine(y_pairs, g[tok], base, shared)
    partial = base + shared if shared is not None else base
    return dict(logits=logits, idx=idx, gates=g, counts=counts, offsets=offsets, perm=perm,
                slot_of=slot_of, rep_of=rep_of, tokens=tok, out=out, partial=partial)


# --------------------------------------------------------------------------- backward
def sigmoid(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def swiglu_expert_backward(xrows, W_gu, W_down, dy):
    """Gradients of one SwiGLU expert y = W_down (SiLU(a) * u), a = W_gate x, u = W_up x.

    Given dL/dy for every row: returns (dL/dx [n, d], dL/dW_gu [2H, d], dL/dW_down [d, H]),
    by the chain rule with SiLU'(a) = s(a) (1 + a (1 - s(a))), s the logistic function.
    """
    X = np.asarray(xrows, dtype=np.float64)
    W = np.asarray(W_gu, dtype=np.float64)
    Wd = np.asarray(W_down, dtype=np.float64)
    DY = np.asarray(dy, dtype=np.float64)
    H = W.shape[0] // 2
    a = X @ W[:H].T
    u = X @ W[H:].T
    s = sigmoid(a)
    h = a * s * u
    dh = DY @ Wd
    da = dh * u * (s * (1.0 + a * (1.0 - s)))
    du = dh * a * s
    dx = da @ W[:H] + du @ W[H:]
    dW_gu = np.concatenate([da.T @ X, du.T @ X], axis=0)
    dW_down = DY.T @ h
    return dx, dW_gu, dW_down


def gate_backward(logits, idx, gating, dg):
    """dL/dlogits [T, E] from dL/dgates [T, k] (the top-k selection itself is piecewise
    constant and passes no gradient).

    * softmax_topk:        g_j = p[e_j], p = softmax(l): dl = p * (dp - <dp, p>), dp[e_j] = dg_j.
    * softmax_topk_renorm: g = softmax(l[sel]): dl[e_j] = g_j (dg_j - sum_i dg_i g_i).
    * sigmoid_topk:        g_j = s(l[e_j]): dl[e_j] = dg_j s (1 - s).
    """
    l = np.asarray(logits, dtype=np.float64)
    ix = idx.astype(np.int64)
    dg = np.asarray(dg, dtype=np.float64)
    T, E = l.shape
    dl = np.zeros((T, E))
    if gating == "softmax_topk":
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dp = np.zeros((T, E))
        np.put_along_axis(dp, ix, dg, axis=1)
        return p * (dp - np.sum(dp * p, axis=1, keepdims=True))
    g = gate_values(l, idx, gating)
    if gating == "softmax_topk_renorm":
        sel = g * (dg - np.sum(dg * g, axis=1, keepdims=True))
    elif gating == "sigmoid_topk":
        sel = dg * g * (1.0 - g)
    else:
        raise ValueError(f"unknown gating {gating!r}")
    np.put_along_axis(dl, ix, sel, axis=1)
    return dl


def layer_backward(x, W_r, bias, W_gu, W_down, Ws_gu, Ws_down, k, gating, d_out,
                   residual_mode="input", residual=None, tau=None, grad_experts=None):
    """Gradients of layer_forward's output for an output gradient d_out [T, d].

    Plain chain rule through the forward's own definition: the residual base, the shared
    experts on every token, and for every routed pair (t, j) the term g[t, j] * E_e(x[src])
    where src is the token of the pair's representative slot.  A condensed pair therefore
    sends its expert gradient to its representative's input, never to its own token: Luffy
    review, referee major comment 1 -- for a condensed token the gradient in that path is
    zero.  Its gate still receives dg = <d_out[t], E_e(x[src])>.

    Returns dx, d_residual (None unless the mode reads r), dW_r, d_bias (None without a
    bias), dW_gu, dW_down, dWs_gu, dWs_down, all float64.  ``grad_experts`` (a list of
    expert ids) limits dW_gu / dW_down to those experts, returned as dicts keyed by
    expert (every other output is complete); None returns full arrays.
    """
    x = np.asarray(x, dtype=np.float64)
    dO = np.asarray(d_out, dtype=np.float64)
    T, d = x.shape
    E = W_gu.shape[0]
    logits, idx, g = route(x, W_r, bias, k, gating)
    counts, offsets, perm, slot_of = dispatch(idx, E)
    use_tau = tau is not None and tau <= 1.0
    rep_of = condense(x[perm], offsets, tau) if use_tau else np.arange(len(perm))
    src = perm[rep_of[slot_of]]                               # [T, k] input token of each pair
    dx = np.zeros((T, d))
    if residual_mode in ("input", "input_plus_external"):
        dx += dO
    d_residual = dO.copy() if residual_mode in ("external", "input_plus_external") else None
    dWs_gu = np.zeros(np.shape(Ws_gu))
    dWs_down = np.zeros(np.shape(Ws_down))
    for s in range(len(Ws_gu)):
        gx, gW, gD = swiglu_expert_backward(x, Ws_gu[s], Ws_down[s], dO)
        dx += gx
        dWs_gu[s] = gW
        dWs_down[s] = gD
    if grad_experts is None:
        dW_gu = np.zeros(np.shape(W_gu))
        dW_down = np.zeros(np.shape(W_down))
    else:
        dW_gu = {e: np.zeros(np.shape(W_gu)[1:]) for e in grad_experts}
        dW_down = {e: np.zeros(np.shape(W_down)[1:]) for e in grad_experts}
    dg = np.zeros((T, k))
    for e in range(E):
        t_sel, j_sel = np.nonzero(idx == e)
        if len(t_sel) == 0:
            continue
        rows = src[t_sel, j_sel]
        y = swiglu_expert(x[rows], W_gu[e], W_down[e])
        dg[t_sel, j_sel] = np.sum(dO[t_sel] * y, axis=1)
        dy = g[t_sel, j_sel][:, None] * dO[t_sel]
        gx, gW, gD = swiglu_expert_backward(x[rows], W_gu[e], W_down[e], dy)
        np.add.at(dx, rows, gx)
        if grad_experts is None or e in dW_gu:
            dW_gu[e] = gW
            dW_down[e] = gD
    dl = gate_backward(logits, idx, gating, dg)
    Wr = np.asarray(W_r, dtype=np.float64)
    dx += dl @ Wr.T
    dW_r = x.T @ dl
    d_bias = dl.sum(axis=0) if bias is not None else None
    return dict(dx=dx, d_residual=d_residual, dW_r=dW_r, d_bias=d_bias, dW_gu=dW_gu,
                dW_down=dW_down, dWs_gu=dWs_gu, dWs_down=dWs_down, idx=idx, rep_of=rep_of)
