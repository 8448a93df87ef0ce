"""The seeded input generators (shared by the oracle and the CUDA path): prefix property,
bf16 rounding and the Zipf router bias, each against something independent."""
from __future__ import annotations

import math
from dataclasses import replace

import numpy as np
import pytest

from routing_expert_ffn_gb300 import inputs as gen


@pytest.mark.parametrize("name", gen.CONFIG_ORDER)
def test_token_prefix_equals_smaller_draw(name):
    """A T'-token workload is the first T' tokens of the full one (x, labels, residual)."""
    cfg = gen.CONFIGS[name]
    full_x, full_lab = gen._token_rows(cfg)
    for Tp in (1, 37, min(1000, cfg.T)):
        small = replace(cfg, T=Tp)
        x, lab = gen._token_rows(small)
        np.testing.assert_array_equal(x, full_x[:Tp])
        np.testing.assert_array_equal(lab, full_lab[:Tp])
    if cfg.residual in ("external", "input_plus_external"):
        a = gen._normal(cfg.seed, (gen._S_RES, 0), (cfg.T, cfg.d), cfg.residual_std)
        b = gen._normal(cfg.seed, (gen._S_RES, 0), (37, cfg.d), cfg.residual_std)
        np.testing.assert_array_equal(b, a[:37])


def test_round_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    a = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 20000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3e38, -3e38], np.float32)])
    # halfway cases: the low 16 bits exactly 0x8000 (ties go to the even bf16 value)
    # (bit 16, the bf16 LSB, drawn too, so ties round both down and up)
    ties = (rng.integers(0, 2 ** 16, 2000, dtype=np.uint32) << np.uint32(16) | np.uint32(0x8000)) & np.uint32(0x7F7FFFFF)
    a = np.concatenate([a.astype(np.float32), ties.view(np.float32)])
    assert a.dtype == np.float32
    want = torch.from_numpy(a.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    got = gen.round_to_bf16(a.copy())
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_zipf_bias_is_a_normalised_power_law():
    cfg = gen.CONFIGS["qwen3_30b_a3b"]
    small = replace(cfg, T=8)
    inp = gen.make_inputs(replace(small, d=256, H=128))
    p = np.exp(inp["bias"].astype(np.float64))
    assert math.isclose(p.sum(), 1.0, rel_tol=1e-5)
    ranked = np.sort(p)[::-1]
    i = np.arange(1, cfg.E + 1, dtype=np.float64)
    np.testing.assert_allclose(ranked / ranked[0], i ** -cfg.zipf_s, rtol=1e-5)
