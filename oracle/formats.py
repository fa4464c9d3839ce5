"""Microscaling formats, written out from their definitions (float64).

TEST INFRASTRUCTURE ONLY: this oracle is imported by tests, by the smoke
check and by the CPU-baseline leg of the benchmark; the product path never
uses it.

Sources
- Kimi-K3 SM120 FlashInfer MXFP4 page, "real checkpoint contract": weights
  are packed MXFP4 (two E2M1 values per byte) with one E8M0 scale per group
  of 32 along K.
- Same page, "NaN/Inf decision record": E8M0 bytes 0x00..0xFE are finite
  powers of two, only 0xFF is NaN; conversion is saturating-finite, so a
  quantised MXFP8 payload is always finite and no scale byte is 0xFF.
- Kimi-K3 MoE path analysis page (SM100 section): activations are quantised
  per 32 elements (absmax -> UE8M0 scale -> FP8 E4M3 codes); four UE8M0 bytes
  are packed into one int32.

Readings where the pages are silent (each is one switch here):
- scale rule: e = smallest integer with amax <= qmax * 2^e, clamped to
  [-127, 127]; byte = e + 127.  amax ignores NaN; amax = 0 gives byte 0x00.
- element rounding: round-to-nearest, ties to the even code, saturating at
  +-qmax; NaN elements become +0; the sign of zero is kept.
- FP4 packing: element 2j in the low nibble, element 2j+1 in the high nibble.
"""
from __future__ import annotations

import math
import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def bf16_decode(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64, from the format's definition: sign bit
    15, 8 exponent bits (bias 127), 7 fraction bits; exponent 0 is subnormal
    (2^-126 * f/128), exponent 255 is Inf (f = 0) or NaN."""
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    ex = (b >> 7) & 0xFF
    fr = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + fr / 128.0, (ex - 127).astype(np.int64))
    sub = np.ldexp(fr / 128.0, -126)
    v = np.where(ex == 0, sub, normal)
    v = np.where(ex == 255, np.where(fr == 0, np.inf, np.nan), v)
    return sign * v


def e2m1_lut() -> np.ndarray:
    """Value of each of the 16 E2M1 codes (1 sign, 2 exponent (bias 1), 1 mantissa bit)."""
    out = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        ex = (c >> 1) & 0x3
        man = c & 0x1
        if ex == 0:
            mag = man * 0.5                      # subnormal: man * 2^(1-1) * 2^-1
        else:
            mag = (1.0 + man / 2.0) * 2.0 ** (ex - 1)
        out[c] = sign * mag
    return out


def e4m3_lut() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (1 sign, 4 exponent (bias 7), 3 mantissa bits;
    no infinities; S.1111.111 is NaN)."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        ex = (c >> 3) & 0xF
        man = c & 0x7
        if ex == 0xF and man == 0x7:
            out[c] = np.nan
            continue
        if ex == 0:
            mag = (man / 8.0) * 2.0 ** -6
        else:
            mag = (1.0 + man / 8.0) * 2.0 ** (ex - 7)
        out[c] = sign * mag
    return out


def ue8m0_decode(b) -> np.ndarray:
    """UE8M0 byte -> 2^(b-127); 0xFF -> NaN."""
    b = np.asarray(b, dtype=np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 0xFF, np.nan, v)


_FORMATS = {
    "e4m3": (e4m3_lut, E4M3_MAX),
    "e2m1": (e2m1_lut, E2M1_MAX),
}
_LUTS = {"e4m3": e4m3_lut(), "e2m1": e2m1_lut()}


def scale_exponent(amax, qmax: float) -> np.ndarray:
    """Smallest integer e with amax <= qmax * 2^e, clamped to [-127, 127].

    Vectorised over `amax`.  NaN counts as 0 (NaN is ignored by the absmax),
    amax = 0 gives -127 and amax = inf gives 127.  The search starts below
    the answer and steps up while the bound is violated; every comparison
    is exact because qmax * 2^e is a scaled power of two."""
    a = np.asarray(amax, dtype=np.float64)
    a = np.where(np.isnan(a), 0.0, a)
    finite_pos = np.isfinite(a) & (a > 0)
    safe = np.where(finite_pos, a, 1.0)
    _, ex_a = np.frexp(safe)          # safe = m * 2^ex_a, m in [0.5, 1)
    _, ex_q = math.frexp(qmax)
    e = (ex_a - ex_q - 1).astype(np.int64)       # qmax*2^e < amax here
    for _ in range(4):
        e = e + (safe > np.ldexp(qmax, e))
    e = np.where(a == 0, -127, e)
    e = np.where(np.isinf(a), 127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def round_to_code(v: np.ndarray, fmt: str) -> np.ndarray:
    """Code of the nearest representable value (ties -> even code), saturating
    at +-qmax; NaN -> +0; the sign of zero is kept.  One code per byte."""
    lut_fn, qmax = _FORMATS[fmt]
    lut = _LUTS[fmt]
    npos = 127 if fmt == "e4m3" else 8           # positive finite codes 0..npos-1
    sign_bit = 0x80 if fmt == "e4m3" else 0x8
    grid = lut[:npos]                              # increasing
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    mag = np.where(nan, 0.0, np.abs(v))
    mag = np.minimum(mag, qmax)                    # saturating finite
    lo = np.searchsorted(grid, mag, side="right") - 1   # grid[lo] <= mag
    lo = np.clip(lo, 0, npos - 1)
    hi = np.minimum(lo + 1, npos - 1)
    dlo = mag - grid[lo]
    dhi = grid[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    neg = np.signbit(v) & ~nan
    code = np.where(neg, code | sign_bit, code).astype(np.uint8)
    return code


def quantize_mx(x: np.ndarray, fmt: str = "e4m3"):
    """Per-32-column microscaling quantisation of a 2-D array.

    Returns (codes uint8 [rows, cols] (one code per byte, not packed),
             scales uint8 [rows, cols/32])."""
    x = np.asarray(x, dtype=np.float64)
    rows, cols = x.shape
    assert cols % 32 == 0, "cols must be a multiple of 32"
    _, qmax = _FORMATS[fmt]
    g = x.reshape(rows, cols // 32, 32)
    absg = np.where(np.isnan(g), 0.0, np.abs(g))
    amax = absg.max(axis=2)
    e = scale_exponent(amax, qmax)
    scales = (e + 127).astype(np.uint8)
    scaled = np.ldexp(g, -e[..., None])          # exact: power-of-two scaling
    codes = round_to_code(scaled, fmt)
    return codes.reshape(rows, cols), scales


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[.., K] 4-bit codes -> [.., K/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def dequant_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 codes [rows, K] + UE8M0 scales [rows, K/32] -> float64."""
    v = _LUTS["e4m3"][np.asarray(codes, dtype=np.uint8)]
    s = ue8m0_decode(scales)
    return v * np.repeat(s, 32, axis=-1)


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed E2M1 [.., K/2] + UE8M0 [.., K/32] -> float64 [.., K]."""
    v = _LUTS["e2m1"][unpack_e2m1(packed)]
    s = ue8m0_decode(scales)
    return v * np.repeat(s, 32, axis=-1)


def pack_scales_int32(scales: np.ndarray) -> np.ndarray:
    """[rows, K/32] bytes -> [rows, K/128] int32, byte i of word p = group 4p+i."""
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    assert s.shape[-1] % 4 == 0
    b = s.reshape(s.shape[:-1] + (s.shape[-1] // 4, 4)).astype(np.uint32)
    w = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    return w.astype(np.uint32).view(np.int32)
