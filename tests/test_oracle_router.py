"""Pins of the oracle's router GEMM (logits = fp32(x @ W_g^T), bf16 operands)
and of its bfloat16 decode, against things other than the oracle itself:
torch's bfloat16 conversion, exact rational sums, exactly rounded double sums
(math.fsum) and exact scaling / permutation invariants."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O


def test_bf16_decode_all_codes_match_torch():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = F.bf16_decode(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the smallest subnormal, the largest finite value, one
    assert F.bf16_decode(np.uint16(0x0001)) == 2.0 ** -133
    assert F.bf16_decode(np.uint16(0x7F7F)) == (2 - 2 ** -7) * 2.0 ** 127
    assert F.bf16_decode(np.uint16(0x3F80)) == 1.0


def _fp32_nearest(fr: Fraction) -> np.float32:
    """The fp32 value nearest to the rational `fr` (ties to the even code)."""
    c = np.float32(float(fr))
    best = None
    for v in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d = abs(Fraction(float(v)) - fr)
        key = (d, int(np.array(v).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, v)
    return best[1]


def _random_bf16(rng, shape, emin, emax):
    """bf16 bit patterns with random signs, exponents in [emin, emax] and fractions."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint32) << 15
    ex = (rng.integers(emin, emax + 1, size=shape) + 127).astype(np.uint32) << 7
    fr = rng.integers(0, 128, size=shape, dtype=np.uint32)
    return (sign | ex | fr).astype(np.uint16)


def test_router_logits_equal_correctly_rounded_exact_sums():
    """Tiny shapes: every logit is the exact rational dot product rounded once to fp32."""
    rng = np.random.default_rng(5)
    x = _random_bf16(rng, (3, 40), -12, 12)
    g = _random_bf16(rng, (6, 40), -12, 12)
    got = O.router_logits(x, g)
    xv, gv = F.bf16_decode(x), F.bf16_decode(g)
    for t in range(3):
        for e in range(6):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xv[t], gv[e]))
            assert got[t, e] == _fp32_nearest(exact), (t, e)


def test_router_logits_full_width_against_exactly_rounded_sums():
    """H = 7168 with the workload's distributions: the BLAS double sums agree
    with math.fsum (the exactly rounded sum of the exact products) after the
    fp32 rounding, to within one fp32 ulp and almost always exactly."""
    w = W.WORKLOADS["decode"]
    s = W.gen_small_inputs(w)
    xb, gb = s["x"][:4], W.gen_gate_weight(w)[:64]
    got = O.router_logits(xb, gb)
    xv, gv = F.bf16_decode(xb), F.bf16_decode(gb)
    same = 0
    for t in range(4):
        for e in range(64):
            ref = np.float32(math.fsum((xv[t] * gv[e]).tolist()))
            assert abs(int(np.array(got[t, e]).view(np.int32)) - int(np.array(ref).view(np.int32))) <= 1
            same += got[t, e] == ref
    assert same >= 255


def test_router_logits_invariants():
    rng = np.random.default_rng(9)
    x = _random_bf16(rng, (5, 256), -6, 3)
    g = _random_bf16(rng, (12, 256), -9, -3)
    base = O.router_logits(x, g)
    # doubling x (exponent + 1, no overflow here) doubles every logit exactly
    x2 = (x.astype(np.uint32) + (1 << 7)).astype(np.uint16)
    assert np.array_equal(O.router_logits(x2, g), 2 * base)
    # permuting the experts (rows of W_g) permutes the columns
    perm = rng.permutation(12)
    assert np.array_equal(O.router_logits(x, g[perm]), base[:, perm])
    # a token's logits depend on that token only
    assert np.array_equal(O.router_logits(x[[3, 1]], g), base[[3, 1]])
    # negating W_g negates the logits
    assert np.array_equal(O.router_logits(x, g ^ np.uint16(0x8000)), -base)
    with pytest.raises(O.ShapeError):
        O.router_logits(x, g[:, :128])


def test_router_logits_match_the_generated_logits():
    """The logits the input generator hands to the logits-input path are the
    router GEMM of its x and W_g."""
    w = W.WORKLOADS["tiny"]
    s = W.gen_small_inputs(w)
    assert np.array_equal(O.router_logits(s["x"], s["wg"]), s["logits"])
