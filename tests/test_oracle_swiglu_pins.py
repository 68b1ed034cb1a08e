"""Pins for the oracle's gated FFN input h = silu(W_gate x) * (W_up x), the
epilogue of the fused gate/up call (the FFN of a decode layer, "wgpu-llm"
README, Architecture at a Glance).

SiLU is pinned at points where it has a closed form: silu(0) = 0,
silu(ln 3) = (3/4) ln 3 (the logistic function is 3/4 there), the odd part
silu(t) - silu(-t) = t, silu(t) -> t and -> 0 at the ends; the composition is
pinned to the pinned products: h[n] = silu(g[n]) * u[n] with g, u the
oracle's own (separately pinned) products, and to closed forms of hand-built
blocks.
"""
import math

import numpy as np
import pytest

import oracle
from block_quantized_weight_dot_gb300 import synthetic as syn
from test_oracle_pins import enc_q4_0, f16_bits, mat


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    for t in (0.1, 1.0, 2.5, 17.0):
        assert abs((oracle.silu(t) - oracle.silu(-t)) - t) < 1e-13 * max(1.0, t)
    assert oracle.silu(60.0) == 60.0
    assert 0.0 > oracle.silu(-60.0) > -1e-24
    # slope 1/2 at 0
    h = 1e-6
    assert abs((oracle.silu(h) - oracle.silu(-h)) / (2 * h) - 0.5) < 1e-9


def test_swiglu_composes_the_products():
    fmt, N, K = syn.Q4_0, 40, 256
    Wg, x = syn.make_problem(fmt, N, K, 1, seed=(120,))
    Wu, _ = syn.make_problem(fmt, N, K, 1, seed=(121,))
    h, g, u, bg, bu = oracle.swiglu(fmt, Wg, Wu, x, N, K)
    g2, bg2 = oracle.qmatmul(fmt, Wg, x, N, K)
    u2, bu2 = oracle.qmatmul(fmt, Wu, x, N, K)
    assert np.array_equal(g, g2[0]) and np.array_equal(u, u2[0])
    assert np.array_equal(bg, bg2[0]) and np.array_equal(bu, bu2[0])
    assert np.array_equal(h, np.array([oracle.silu(a) for a in g]) * u)


def test_swiglu_hand_built_blocks():
    """gate = all q = 9 (w = d) and up = all q = 15 (w = 7d) times ones:
    g = K d, u = 7 K d, h = silu(K d) * 7 K d; and gate at q = 8 (w = 0) gives
    h = 0 whatever up is."""
    K = 64
    d = f16_bits(0.01)
    dv = float(np.float16(0.01))
    ones = np.ones(K, np.float32)
    Wg = mat([[enc_q4_0(d, [9] * 32)] * 2])
    Wu = mat([[enc_q4_0(d, [15] * 32)] * 2])
    h, g, u, _, _ = oracle.swiglu(syn.Q4_0, Wg, Wu, ones, 1, K)
    assert g[0] == K * dv and u[0] == 7 * K * dv
    assert h[0] == (K * dv / (1.0 + math.exp(-K * dv))) * (7 * K * dv)
    Wz = mat([[enc_q4_0(d, [8] * 32)] * 2])
    h, _, _, _, _ = oracle.swiglu(syn.Q4_0, Wz, Wu, ones, 1, K)
    assert h[0] == 0.0
