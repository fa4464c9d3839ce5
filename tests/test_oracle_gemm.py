"""Pins of the oracle's block-scaled FC1/FC2: exact rational sums over
independently decoded operands (torch's float8 decode for E4M3, the OCP table
for E2M1, 2^(b-127) as an exact Fraction), [gate; up] ordering, and
order-independence of the double result."""
import os
from fractions import Fraction

import numpy as np
import torch

from oracle import formats as F
from oracle import moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = [Fraction(v) for _, v in (l.split() for l in open(os.path.join(GOLDEN, "e2m1_values.txt")) if l[0] != "#")]


def _e4m3_exact(codes):
    vals = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return [[Fraction(float(v)) for v in row] for row in vals]


def _fp4_row(packed_row, sf_row):
    out = []
    for kk in range(len(packed_row) * 2):
        byte = int(packed_row[kk // 2])
        code = (byte >> 4) if kk % 2 else (byte & 0xF)
        out.append(E2M1[code] * Fraction(2) ** (int(sf_row[kk // 32]) - 127))
    return out


def _rand_case(rng, n, H, I):
    xq = rng.integers(0, 256, (n, H), dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x3C                       # no NaN codes
    xs = rng.integers(118, 132, (n, H // 32), dtype=np.uint8)
    w13 = rng.integers(0, 256, (2 * I, H // 2), dtype=np.uint8)
    w13s = rng.integers(121, 128, (2 * I, H // 32), dtype=np.uint8)
    return xq, xs, w13, w13s


def test_fc1_equals_exact_rational_sum():
    rng = np.random.default_rng(5)
    n, H, I = 3, 64, 32
    xq, xs, w13, w13s = _rand_case(rng, n, H, I)
    gate, up = moe.expert_fc1(xq, xs, w13, w13s, I)
    a = _e4m3_exact(xq)
    for r in range(n):
        arow = [a[r][kk] * Fraction(2) ** (int(xs[r, kk // 32]) - 127) for kk in range(H)]
        for c in range(2 * I):
            brow = _fp4_row(w13[c], w13s[c])
            exact = sum(x * y for x, y in zip(arow, brow))
            got = gate[r, c] if c < I else up[r, c - I]
            assert Fraction(got) == exact, (r, c)


def test_fc2_equals_exact_rational_sum():
    rng = np.random.default_rng(6)
    n, H, I = 2, 32, 64
    iq = rng.integers(0, 256, (n, I), dtype=np.uint8)
    iq[(iq & 0x7F) == 0x7F] = 0x41
    isf = rng.integers(120, 126, (n, I // 32), dtype=np.uint8)
    w2 = rng.integers(0, 256, (H, I // 2), dtype=np.uint8)
    w2s = rng.integers(121, 128, (H, I // 32), dtype=np.uint8)
    y = moe.expert_fc2(iq, isf, w2, w2s)
    a = _e4m3_exact(iq)
    for r in range(n):
        arow = [a[r][kk] * Fraction(2) ** (int(isf[r, kk // 32]) - 127) for kk in range(I)]
        for h in range(H):
            assert Fraction(y[r, h]) == sum(x * b for x, b in zip(arow, _fp4_row(w2[h], w2s[h])))


def test_gate_rows_come_first():
    rng = np.random.default_rng(7)
    n, H, I = 2, 64, 32
    xq, xs, w13, w13s = _rand_case(rng, n, H, I)
    w13z = w13.copy()
    w13z[I:] = 0                                          # up half = +0 codes
    gate, up = moe.expert_fc1(xq, xs, w13z, w13s, I)
    assert np.all(up == 0) and np.any(gate != 0)


def test_fc1_is_order_independent_at_workload_scales():
    # products span ~2^-24..2^5 and |sums| < 2^18 at the workloads' distributions,
    # so the double result is exact and any summation order gives the same bits
    rng = np.random.default_rng(8)
    n, H, I = 4, 1024, 64
    xf = rng.standard_normal((n, H))
    xq, xs = F.quantize_mx(xf, "e4m3")
    w13 = rng.integers(0, 256, (2 * I, H // 2), dtype=np.uint8)
    w13s = rng.integers(121, 128, (2 * I, H // 32), dtype=np.uint8)
    gate, up = moe.expert_fc1(xq, xs, w13, w13s, I)
    a = F.dequant_mxfp8(xq, xs)
    b = F.dequant_mxfp4(w13, w13s)
    prod = a[:, None, :] * b[None, :, :]
    s1 = np.sum(prod, axis=2)
    s2 = np.sum(prod[:, :, ::-1], axis=2)
    assert np.array_equal(np.concatenate([gate, up], 1), s1)
    assert np.array_equal(s1, s2)
