"""Pins of the oracle's SiTU: closed-form values derived by hand, zeros,
limits, oddness, and the reduction to SwiGLU (SiLU(g) * u) for large betas."""
import math
import os

import numpy as np

from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(expr):
    return float(eval(expr, {"ln2": math.log(2.0), "ln3": math.log(3.0)}))


def test_closed_form_points():
    for line in open(os.path.join(GOLDEN, "situ_points.txt")):
        if line.startswith("#") or not line.strip():
            continue
        g, u, ref = line.split()
        got = float(moe.situ(np.array([_ev(g)]), np.array([_ev(u)]), 4.0, 25.0)[0])
        assert abs(got - float(ref)) <= 1e-13 * max(1.0, abs(float(ref))), (g, u, got, ref)


def test_limits_and_symmetry():
    big = np.array([1e3])
    assert moe.situ(big, big)[0] == 100.0 or 100.0 - moe.situ(big, big)[0] < 1e-12
    v = moe.situ(np.array([60.0]), np.array([400.0]))[0]
    assert 99.99 < v <= 100.0
    assert abs(moe.situ(np.array([-80.0]), np.array([50.0]))[0]) < 1e-30
    g = np.linspace(-30, 30, 101)
    u = np.linspace(-300, 300, 101)
    a = moe.situ(g[:, None], u[None, :])
    b = moe.situ(g[:, None], -u[None, :])
    assert np.array_equal(a, -b)                           # odd in up
    assert np.all(np.abs(a) < 100.0)                       # |SiTU| < beta * beta_lin


def test_reduces_to_swiglu_for_large_beta():
    g = np.linspace(-6, 6, 41)
    u = np.linspace(-3, 3, 41)
    a = moe.situ(g, u, 1e7, 1e7)
    silu_u = g / (1.0 + np.exp(-g)) * u
    assert np.allclose(a, silu_u, rtol=1e-9, atol=1e-12)
    # small-argument behaviour at the real betas: SiLU(g)*u to third order
    gs, us = 1e-3, 2e-3
    a = moe.situ(np.array([gs]), np.array([us]))[0]
    ref = gs / (1 + math.exp(-gs)) * us
    assert abs(a - ref) < 1e-6 * abs(ref)
