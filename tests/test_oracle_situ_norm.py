"""Pins for SiTU-GLU and RMSNorm in the oracle (CPU only).

SiTU-GLU (kimi-k3-in-c README section 9, k3_situ_glu; colibri "Stable
LatentMoE"): zeros, the analytic cap b1*b2 = 100 that the page's fixture hits,
the sweep 0.1..1000 staying under it, the small-input limit where it reduces
to SiLU(g)*u (scipy's expit), odd symmetry in u, and the sigma-of-uncapped-gate
rule. RMSNorm (README section 5): closed forms for constant and two-element
vectors, eps inside the square root, gain applied after.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bound():
    with open(os.path.join(GOLD, "situ_bound.json")) as f:
        return json.load(f)


def test_situ_zeros():
    for v in (0.1, 1.0, -3.0, 1000.0):
        assert oracle.situ(0.0, v) == 0.0
        assert oracle.situ(v, 0.0) == 0.0


def test_situ_reaches_cap():
    g = _bound()
    # saturated inputs: tanh -> 1 and sigmoid -> 1 in double precision
    assert oracle.situ(1000.0, 1000.0, g["b1"], g["b2"]) == g["cap"]
    assert oracle.situ(1000.0, -1000.0, g["b1"], g["b2"]) == -g["cap"]


def test_situ_sweep_stays_below_cap():
    g = _bound()
    mags = np.geomspace(g["sweep_min"], g["sweep_max"], 61)
    vals = np.concatenate([mags, -mags])
    worst = max(abs(oracle.situ(a, b, g["b1"], g["b2"])) for a in vals for b in vals)
    assert worst <= g["cap"]
    assert worst > 0.999 * g["cap"]


@pytest.mark.parametrize("g,u", [(1e-4, 2e-4), (-3e-4, 1e-4), (5e-4, -5e-4)])
def test_situ_small_input_is_silu_times_u(g, u):
    """For |g|,|u| << b1, b2 the tanh caps are the identity and SiTU-GLU is
    SiLU(g) * u (library expit for the sigmoid)."""
    ref = g * expit(g) * u
    assert oracle.situ(g, u) == pytest.approx(ref, rel=1e-7)


def test_situ_odd_in_u_and_monotone():
    for gv in (-5.0, -0.5, 0.7, 9.0):
        for uv in (0.3, 4.0, 60.0):
            assert oracle.situ(gv, -uv) == -oracle.situ(gv, uv)
        us = np.linspace(-80, 80, 41)
        ys = [oracle.situ(gv, uu) for uu in us]
        s = np.sign(gv * expit(gv))
        assert all(s * (b - a) >= 0 for a, b in zip(ys, ys[1:]))


def test_situ_sigmoid_reads_uncapped_gate():
    """At g = 8 the two readings differ by about 2%: sigma(8) vs
    sigma(4*tanh(8/4)). With the up factor saturated (u = 1000 -> 25)."""
    uncapped = 4 * math.tanh(2.0) * expit(8.0) * 25.0
    capped = 4 * math.tanh(2.0) * expit(4 * math.tanh(2.0)) * 25.0
    got = oracle.situ(8.0, 1000.0)
    assert got == pytest.approx(uncapped, rel=1e-14)
    assert abs(got - capped) > 1.0


def test_situ_large_gate_limits():
    # g -> +inf: sigma -> 1, b1*tanh -> b1;  g -> -inf: sigma -> 0
    assert oracle.situ(200.0, 10.0) == pytest.approx(4.0 * 25 * math.tanh(0.4), rel=1e-15)
    assert abs(oracle.situ(-200.0, 10.0)) < 1e-80


def test_rmsnorm_constant_vector():
    for c in (0.5, -2.0, 3e-3):
        for n in (1, 7, 128):
            for eps in (1e-5, 0.0, 0.25):
                out = oracle.rmsnorm(np.full(n, c), None, eps)
                np.testing.assert_allclose(out, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_two_element_and_gain():
    out = oracle.rmsnorm(np.array([3.0, 4.0]), np.array([2.0, -1.0]), 0.0)
    # mean of squares 12.5
    np.testing.assert_allclose(out, [2 * 3 / math.sqrt(12.5), -4 / math.sqrt(12.5)], rtol=1e-15)


def test_rmsnorm_eps_inside_sqrt():
    x = np.array([1e-3, -1e-3])
    eps = 1e-5
    out = oracle.rmsnorm(x, None, eps)
    # eps inside the root: x / sqrt(1e-6 + 1e-5); outside would be x / (1e-3 + 1e-5)
    np.testing.assert_allclose(out, x / math.sqrt(1e-6 + eps), rtol=1e-15)
    assert abs(out[0] - x[0] / (1e-3 + eps)) > 0.1


def test_rmsnorm_scale_invariant_without_eps():
    x = np.linspace(-2, 3, 37)
    np.testing.assert_allclose(oracle.rmsnorm(7.0 * x, None, 0.0), oracle.rmsnorm(x, None, 0.0),
                               rtol=1e-14)


# ---- the layer input made from the residual stream ---------------------------------

def test_round_bf16_exact_values():
    """Round to nearest, ties to even, at bf16's 8 significant bits."""
    cases = [
        (1.0, 0x3F80), (-1.5, 0xBFC0), (3.0, 0x4040), (0.0, 0x0000), (-0.0, 0x8000),
        (1.0 + 2.0 ** -8, 0x3F80),              # tie between 0x3F80 and 0x3F81: the even one
        (1.0 + 3 * 2.0 ** -8, 0x3F82),          # tie between 0x3F81 and 0x3F82: the even one
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81), # just above the tie
        (1.0 - 2.0 ** -10, 0x3F80),             # below 1: ulp 2^-8, rounds up to 1
        (2.0 ** -130, 0x0008),                  # subnormal: 8 * 2^-133
        (2.0 ** -134, 0x0000),                  # half of the smallest subnormal, tie to even 0
        (3 * 2.0 ** -134, 0x0002),              # 1.5 * 2^-133: tie between 1 and 2, even
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F), # the largest finite bf16
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80), # tie above it: the even neighbour is infinity
    ]
    got = oracle.round_bf16(np.array([v for v, _ in cases], np.float64))
    for (v, want), g in zip(cases, got):
        assert int(g) == want, (v, hex(int(g)), hex(want))


def test_round_bf16_is_nearest_on_a_sweep():
    """Every rounded value is a nearest bf16 neighbour (checked by widening the
    two candidates around it), over a sweep of magnitudes and signs."""
    v = np.concatenate([np.linspace(-7.3, 9.1, 2001), np.geomspace(1e-30, 1e30, 301)])
    bits = oracle.round_bf16(v).astype(np.uint32)
    w = (bits << 16).view(np.float32).astype(np.float64)
    up = ((bits + 1) << 16).view(np.float32).astype(np.float64)
    dn = ((bits - 1) << 16).view(np.float32).astype(np.float64)
    err = np.abs(w - v)
    assert np.all(err <= np.abs(up - v)) and np.all(err <= np.abs(dn - v))


def test_residual_input_closed_form():
    """x = h / sqrt(mean(h^2) + eps) * gain per row."""
    h = np.array([[3.0, 4.0, 0.0, 0.0], [1.0, 1.0, 1.0, 1.0]], np.float32)
    g = np.array([0x3F80, 0x4000, 0xBF80, 0x3F00], np.uint16)   # 1, 2, -1, 0.5
    eps = 1e-5
    x = oracle.residual_input(h, g, eps)
    inv0 = 1 / math.sqrt(25 / 4 + eps)
    inv1 = 1 / math.sqrt(1 + eps)
    np.testing.assert_allclose(x[0], [3 * inv0, 8 * inv0, 0.0, 0.0], rtol=1e-15)
    np.testing.assert_allclose(x[1], [inv1, 2 * inv1, -inv1, 0.5 * inv1], rtol=1e-15)

