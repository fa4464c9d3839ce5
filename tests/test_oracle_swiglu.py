"""Pins of the oracle's SwiGLU control activation: closed-form values derived
by hand (sigmoid(ln 3) = 3/4), the clamps, the zero, and the reduction to the
textbook SwiGLU (SiLU(g) * u) when the clamp and offset are lifted."""
import math
import os

import numpy as np

from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_closed_form_points():
    n = 0
    for line in open(os.path.join(GOLDEN, "swiglu_points.txt")):
        if line.startswith("#") or not line.strip():
            continue
        g, u, ref = line.split()
        gv = float(eval(g, {"ln3": math.log(3.0)}))
        got = float(moe.swiglu(np.array([gv]), np.array([float(u)]))[0])
        assert abs(got - float(ref)) <= 1e-13 * max(1.0, abs(float(ref))), (g, u, got, ref)
        n += 1
    assert n == 7


def test_clamps():
    u = np.linspace(-20, 20, 81)
    assert np.array_equal(moe.swiglu(np.full_like(u, 10.0), u), moe.swiglu(np.full_like(u, 7.0), u))
    g = np.linspace(-20, 20, 81)
    assert np.array_equal(moe.swiglu(g, np.full_like(g, 100.0)), moe.swiglu(g, np.full_like(g, 7.0)))
    assert np.array_equal(moe.swiglu(g, np.full_like(g, -100.0)), moe.swiglu(g, np.full_like(g, -7.0)))
    # u' = -beta gives exactly zero; large negative gates decay to zero
    assert np.all(moe.swiglu(g, np.full_like(g, -1.0)) == 0.0)
    assert abs(moe.swiglu(np.array([-200.0]), np.array([3.0]))[0]) < 1e-100


def test_reduces_to_textbook_swiglu():
    g = np.linspace(-6, 6, 41)
    u = np.linspace(-3, 3, 41)
    a = moe.swiglu(g, u, alpha=1.0, beta=0.0, limit=np.inf)
    assert np.allclose(a, g / (1.0 + np.exp(-g)) * u, rtol=1e-14, atol=0.0)
