"""Pins of the oracle's microscaling formats against things other than itself:
a library's float8 decode and rounding, the OCP E2M1 value table, exact
closed forms of the scale rule, round trips and the pages' NaN/Inf rules."""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_lut_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    lut = F.e4m3_lut()
    assert np.array_equal(np.isnan(ref), np.isnan(lut))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], lut[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(lut[ok]))
    assert lut[0x7E] == 448.0 and lut[0x01] == 2.0 ** -9


def test_e2m1_lut_matches_ocp_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_values.txt")) if l[0] != "#"]
    table = np.array([float(v) for _, v in rows])
    lut = F.e2m1_lut()
    assert np.array_equal(table, lut)
    assert np.array_equal(np.signbit(table), np.signbit(lut))
    # every E2M1 value is exactly an E4M3 value (FP4 widens to FP8 losslessly)
    e4 = F.e4m3_lut()
    assert all(v in e4 for v in lut)


def test_e4m3_rounding_matches_torch_rne():
    rng = np.random.default_rng(1)
    lut = F.e4m3_lut()[:127]
    mids = (lut[1:] + lut[:-1]) / 2                       # exact ties
    vals = np.concatenate([
        rng.uniform(-448, 448, 20000),
        np.exp(rng.uniform(-14, 6, 20000)) * rng.choice([-1, 1], 20000),
        mids, -mids, lut, -lut, [0.0, -0.0, 2.0 ** -10, -2.0 ** -10, 2.0 ** -11],
    ])
    vals = vals.astype(np.float32).astype(np.float64)      # representable in fp32: no double rounding in torch
    ours = F.round_to_code(vals, "e4m3")
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_saturation_and_nonfinite_rules():
    # beyond 448 saturates (the pages: saturating-finite conversion, payload always finite)
    assert F.round_to_code(np.array([1e30, -1e30, np.inf, -np.inf]), "e4m3").tolist() == [0x7E, 0xFE, 0x7E, 0xFE]
    assert F.round_to_code(np.array([np.nan]), "e4m3").tolist() == [0x00]
    assert F.round_to_code(np.array([7.0, 100.0, -5.1, -4.9]), "e2m1").tolist() == [0x7, 0x7, 0xF, 0xE]
    x = np.zeros((1, 64))
    x[0, 3] = np.inf
    x[0, 40] = np.nan
    x[0, 41] = 1.0
    codes, scales = F.quantize_mx(x, "e4m3")
    assert scales[0, 0] == 0xFE                # inf group: largest finite scale
    assert scales.max() < 0xFF                 # never the NaN scale
    assert codes[0, 3] == 0x7E
    assert codes[0, 40] == 0x00                # NaN -> +0
    lut = F.e4m3_lut()
    assert np.all(np.isfinite(lut[codes]))


def test_scale_rule_is_minimal_exponent():
    rng = np.random.default_rng(2)
    for qmax in (448.0, 6.0):
        amax = np.exp(rng.uniform(-60, 60, 5000))
        e = F.scale_exponent(amax, qmax)
        assert np.all(amax <= qmax * 2.0 ** e)
        assert np.all(amax > qmax * 2.0 ** (e - 1))
        r = amax * 2.0 ** -e                   # normalised amax lands in (qmax/2, qmax]
        assert np.all((r > qmax / 2) & (r <= qmax))
    # boundaries
    assert F.scale_exponent(np.array([448.0, 448.0 * (1 + 2 ** -50), 0.0]), 448.0).tolist() == [0, 1, -127]
    assert F.scale_exponent(np.array([2.0 ** -200, 2.0 ** 300]), 448.0).tolist() == [-127, 127]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_quantize_round_trip(fmt):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 256)) * np.exp(rng.uniform(-5, 5, (8, 1)))
    q, s = F.quantize_mx(x, fmt)
    lut = F._LUTS[fmt]
    deq = lut[q] * np.repeat(F.ue8m0_decode(s), 32, axis=1)
    q2, s2 = F.quantize_mx(deq, fmt)
    deq2 = lut[q2] * np.repeat(F.ue8m0_decode(s2), 32, axis=1)
    # grid values re-quantise to the same values (the scale may drop by one
    # when rounding brought a group's max down to exactly qmax/2)
    assert np.array_equal(deq, deq2)
    assert np.all((s2 == s) | (s2 == s - 1))
    # each element is the nearest grid point: error at most half a step of the
    # coarsest spacing of its group (qmax step: 32 for e4m3 at the top, 2 for e2m1)
    step = {"e4m3": 32.0, "e2m1": 2.0}[fmt]
    err = np.abs(deq - x) / np.repeat(F.ue8m0_decode(s), 32, axis=1)
    assert np.all(err <= step / 2 + 1e-12)


def test_fp4_nibble_order_and_int32_scale_packing():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = F.pack_e2m1(codes)
    assert packed.tolist() == [[0x21, 0x43]]            # element 2j in the low nibble
    assert np.array_equal(F.unpack_e2m1(packed), codes)
    s = np.arange(8, dtype=np.uint8).reshape(1, 8) + 120
    w = F.pack_scales_int32(s)
    assert np.array_equal(w, s.view("<i4"))             # a little-endian int32 view of the bytes
    # the pages' x_sf shape: [T, H/128] int32 for H = 7168
    assert F.pack_scales_int32(np.zeros((3, 7168 // 32), np.uint8)).shape == (3, 56)


def test_checkpoint_shapes_from_pages():
    import json
    g = json.load(open(os.path.join(GOLDEN, "checkpoint_shapes.json")))
    K, I = g["K_latent"], g["I"]
    # two E2M1 codes per byte; one scale byte per 32 along K
    assert g["w1.weight_packed"] == [I, K // 2] and g["w1.weight_scale"] == [I, K // 32]
    assert g["w2.weight_packed"] == [K, I // 2] and g["w2.weight_scale"] == [K, I // 32]
    from workloads import Workload, weight_shapes
    sh = weight_shapes(Workload("ckpt", T=1, H=K, I=I, E=1, k=1))
    # the loader stacks w1 (gate) and w3 (up) into the [gate; up] halves of w13
    assert sh["w13"][1:] == (2 * g["w1.weight_packed"][0], g["w1.weight_packed"][1])
    assert sh["w13_sf"][1:] == (2 * g["w1.weight_scale"][0], g["w1.weight_scale"][1])
    assert list(sh["w2"][1:]) == g["w2.weight_packed"]
    assert list(sh["w2_sf"][1:]) == g["w2.weight_scale"]
