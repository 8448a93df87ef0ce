"""Luffy condensation with historical similarity on the GPU (moe_condense_hist) against the
oracle's condense_with_history, through the C ABI.

Bit for bit: the representative of every slot, and the pair classes the call hands to the
next one (decoded from the history record's documented layout).  Two consecutive calls
("blocks"): the first without history, the second with the first one's record.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as orc
from routing_expert_ffn_gb300 import inputs as gen
from tests import harness

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "condense_history.json")
MAGIC = 0x48697374


@pytest.fixture(scope="module")
def moe():
    from routing_expert_ffn_gb300 import build
    build.build()
    from routing_expert_ffn_gb300 import moe as m
    m.lib()
    return m


def _align(x):
    return (x + 255) & ~255


def decode_history(rec: np.ndarray, T: int, k: int, E: int) -> dict:
    """{(u, t): similar} from a history record (layout of include/moe.h)."""
    P = T * k
    words = P * ((min(T, P) + 31) // 32)  # a bucket holds each token at most once
    o = 0
    at = []
    for nbytes in (4 * 5, 4 * (E + 1), 4 * P, 8 * E, 8 * words):
        at.append(o)
        o = _align(o + nbytes)
    b = rec.tobytes()
    header = np.frombuffer(b, np.int32, 5, at[0])
    assert header.tolist() == [MAGIC, T, k, E, P]
    offsets = np.frombuffer(b, np.int32, E + 1, at[1])
    slot_of = np.frombuffer(b, np.int32, P, at[2])
    base = np.frombuffer(b, np.int64, E, at[3])
    planes = np.frombuffer(b, np.uint32, 2 * words, at[4])
    known, simc = np.ascontiguousarray(planes[0::2]), np.ascontiguousarray(planes[1::2])
    tok_of = np.full(P, -1, np.int64)
    for p, s in enumerate(slot_of):
        if s >= 0:
            tok_of[s] = p // k
    out: dict = {}
    for e in range(E):
        a, n = int(offsets[e]), int(offsets[e + 1] - offsets[e])
        if n < 2:
            continue
        W = (n + 31) // 32
        kn = known[base[e]: base[e] + n * W].reshape(n, W)
        sm = simc[base[e]: base[e] + n * W].reshape(n, W)
        kb = np.unpackbits(kn.view(np.uint8).reshape(n, -1), axis=1, bitorder="little")[:, :n]
        sb = np.unpackbits(sm.view(np.uint8).reshape(n, -1), axis=1, bitorder="little")[:, :n]
        low = np.tril(np.ones((n, n), bool), -1)
        assert not (sb.astype(bool) & ~kb.astype(bool) & low).any(), "similar without a class"
        ii, jj = np.nonzero(kb.astype(bool) & low)
        for i, j in zip(ii.tolist(), jj.tolist()):
            u, t = sorted((int(tok_of[a + j]), int(tok_of[a + i])))
            cls = bool(sb[i, j])
            assert out.setdefault((u, t), cls) == cls, "one pair, two classes"
    return out


def _gpu_block(moe, C, x_perm_np, offsets, perm, slot_of, tau, s1, s2, hist_in):
    xp = torch.from_numpy(np.ascontiguousarray(x_perm_np, np.float32)).to("cuda", torch.bfloat16)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    rep_of, n_rep, n_cond, n_cos, rec = moe.condense_hist(C, xp, t(offsets), t(perm), t(slot_of),
                                                          tau, s1, s2, hist_in=hist_in)
    torch.cuda.synchronize()
    assert moe.get_device_status() == 0
    return rep_of.cpu().numpy(), int(n_cond.item()), int(n_cos.item()), rec


def test_history_golden_blocks(moe):
    """The hand-derived two-block cases: rows are the unit 2-D vectors padded to d = 256 and
    rounded to bf16 (the oracle runs on the same stored values)."""
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        T = len(c["blocks"][0]["angles"])
        k = max(sum(t in b for b in blk["buckets"]) for blk in c["blocks"] for t in range(T))
        E = max(len(blk["buckets"]) for blk in c["blocks"])
        C = moe.Config(T=T, d=256, E=E, k=k, H=128, dtype="bf16")
        hist_gpu, hist_orc = None, None
        for bi, blk in enumerate(c["blocks"]):
            rows = np.zeros((T, 256), np.float32)
            for t, a in enumerate(blk["angles"]):
                rows[t, 0], rows[t, 1] = math.cos(math.radians(a)), math.sin(math.radians(a))
            rows = gen.round_to_bf16(rows)
            buckets = blk["buckets"] + [[]] * (E - len(blk["buckets"]))
            perm = np.array([t for b in buckets for t in b], np.int32)
            offsets = np.concatenate([[0], np.cumsum([len(b) for b in buckets])]).astype(np.int32)
            slot_of = np.full((T, k), -1, np.int32)
            for s, t in enumerate(perm):
                j = int(np.sum(slot_of[t] >= 0))
                slot_of[t, j] = s
            xp = rows[perm]
            rep_o, hist_orc = orc.condense_with_history(xp, offsets, perm, g["tau"], g["s1"],
                                                        g["s2"], hist_orc)
            got = [[int(perm[rep_o[s]]) for s in range(offsets[e], offsets[e + 1])]
                   for e in range(len(blk["buckets"]))]
            assert got == blk["rep"], (c["name"], bi, "oracle on bf16 rows")
            rep_g, _, n_cos, rec = _gpu_block(moe, C, xp, offsets, perm, slot_of, g["tau"],
                                              g["s1"], g["s2"], hist_gpu)
            np.testing.assert_array_equal(rep_g[: offsets[-1]], rep_o[: offsets[-1]])
            assert decode_history(rec.cpu().numpy(), T, k, E) == hist_orc, (c["name"], bi)
            hist_gpu = rec


def _luffy_block2_routing(cfg, labels, seed=11):
    """A second block's routing: every centroid keeps one expert pair for all its copies
    (near-duplicate tokens route together), every other token a seeded pair of its own."""
    rng = np.random.default_rng(seed)
    T, E, k = len(labels), cfg.E, cfg.k
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    cent = {}
    for t, c in enumerate(labels):
        if c >= 0:
            idx[t] = cent.setdefault(int(c), idx[t])
    return idx


def _perturb(x, eps=0.02, seed=12):
    """Rows moved by a small relative step (a block's residual update): x + eps |x| n / sqrt(d)."""
    rng = np.random.default_rng(seed)
    n = rng.standard_normal(x.shape)
    scale = eps * np.linalg.norm(x, axis=1, keepdims=True) / math.sqrt(x.shape[1])
    return gen.round_to_bf16((x + scale * n).astype(np.float32))


@pytest.mark.parametrize("scenario", ["repeat", "next_block"])
def test_history_luffy_two_blocks(moe, scenario):
    """luffy_condense at T = 2048: block 1 without history, block 2 with block 1's record.
    'repeat': the same rows and routing again -- every co-routed pair already has a class,
    so no Gram tile needs the tensor cores.  'next_block': rows perturbed, a fresh routing."""
    cfg, inp = harness.workload("luffy_condense", T=2048)
    C = moe.Config.from_workload(cfg)
    tau, s1, s2 = cfg.taus[0], 0.8, 0.2
    _, idx1, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    blocks = [(inp["x"], idx1)]
    if scenario == "repeat":
        blocks.append((inp["x"], idx1))
    else:
        blocks.append((_perturb(inp["x"]), _luffy_block2_routing(cfg, inp["labels"])))
    hist_gpu, hist_orc = None, None
    for bi, (x, idx) in enumerate(blocks):
        counts, offsets, perm, slot_of = orc.dispatch(idx, cfg.E)
        xp = x[perm]
        rep_o, hist_orc = orc.condense_with_history(xp, offsets, perm, tau, s1, s2, hist_orc)
        rep_g, n_cond, n_cos, rec = _gpu_block(moe, C, xp, offsets, perm, slot_of, tau, s1, s2,
                                               hist_gpu)
        np.testing.assert_array_equal(rep_g[: cfg.P], rep_o)
        assert n_cond == int(np.sum(rep_o != np.arange(cfg.P)))
        assert decode_history(rec.cpu().numpy(), cfg.T, cfg.k, cfg.E) == hist_orc, bi
        if bi == 1 and scenario == "repeat":
            assert n_cos == 0
        hist_gpu = rec


def test_history_top8_two_blocks(moe):
    """The lookup searches each token pair's k previous buckets for a common one: top-8 of 16
    experts (each token in half the buckets) on 512 tokens of the condensation workload; the
    second block keeps the rows and draws a fresh top-8 per token (copies of one centroid
    still route together), so pairs meet again in other buckets than before."""
    from dataclasses import replace
    base = gen.CONFIGS["luffy_condense"]
    cfg = replace(base, name="luffy_top8", k=8)
    inp = harness.condition(cfg, gen.make_inputs(cfg.with_tokens(512)))
    cfg = cfg.with_tokens(512)
    C = moe.Config.from_workload(cfg)
    _, idx1, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    idx2 = _luffy_block2_routing(cfg, inp["labels"], seed=21)
    hist_gpu, hist_orc = None, None
    for bi, idx in enumerate((idx1, idx2)):
        counts, offsets, perm, slot_of = orc.dispatch(idx, cfg.E)
        xp = inp["x"][perm]
        rep_o, hist_orc = orc.condense_with_history(xp, offsets, perm, 0.95, 0.8, 0.2, hist_orc)
        rep_g, n_cond, n_cos, rec = _gpu_block(moe, C, xp, offsets, perm, slot_of, 0.95, 0.8,
                                               0.2, hist_gpu)
        np.testing.assert_array_equal(rep_g[: cfg.P], rep_o)
        assert decode_history(rec.cpu().numpy(), cfg.T, cfg.k, cfg.E) == hist_orc, bi
        hist_gpu = rec


def test_history_of_another_shape_is_ignored(moe):
    """A record written for another token count counts as no history: the call equals the
    first block's."""
    cfg, inp = harness.workload("luffy_condense", T=1024)
    C = moe.Config.from_workload(cfg)
    _, idx, _ = orc.route(inp["x"], inp["W_r"], inp["bias"], cfg.k, cfg.gating)
    counts, offsets, perm, slot_of = orc.dispatch(idx, cfg.E)
    xp = inp["x"][perm]
    rep0, _, _, rec0 = _gpu_block(moe, C, xp, offsets, perm, slot_of, 0.95, 0.8, 0.2, None)
    # a record of the 512-token layer, written into a buffer of this layer's record size
    cfg_s, inp_s = harness.workload("luffy_condense", T=512)
    C_s = moe.Config.from_workload(cfg_s)
    _, idx_s, _ = orc.route(inp_s["x"], inp_s["W_r"], inp_s["bias"], cfg_s.k, cfg_s.gating)
    _, off_s, perm_s, so_s = orc.dispatch(idx_s, cfg_s.E)
    other = torch.zeros(moe.condense_history_bytes(C), dtype=torch.uint8, device="cuda")
    xps = torch.from_numpy(inp_s["x"][perm_s]).to("cuda", torch.bfloat16)
    ti = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    moe.condense_hist(C_s, xps, ti(off_s), ti(perm_s), ti(so_s), 0.95, 0.8, 0.2, hist_out=other)
    rep1, _, n_cos, rec1 = _gpu_block(moe, C, xp, offsets, perm, slot_of, 0.95, 0.8, 0.2, other)
    np.testing.assert_array_equal(rep1, rep0)
    assert decode_history(rec1.cpu().numpy(), cfg.T, cfg.k, cfg.E) == \
        decode_history(rec0.cpu().numpy(), cfg.T, cfg.k, cfg.E)
