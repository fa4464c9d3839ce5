"""Seeded synthetic inputs for the Kimi-K3 routed-expert MoE layer.

This module only *draws* inputs. It holds none of the layer's arithmetic
(no routing, no quantisation, no GEMM); both the CPU oracle and the CUDA
path consume what it produces.

Workloads (all seeded with seed 0, one independent stream per tensor):

  tiny      T=16,   H=128,  I=128,  E=8,   k=2
  reduced   T=128,  H=7168, I=3584, E=64,  k=16
  decode    T=16,   H=7168, I=3584, E=896, k=16
  prefill   T=8192, H=7168, I=3584, E=896, k=16
  skewed    T=2048, H=7168, I=3584, E=896, k=16, Zipf-skewed correction bias

Distributions (Kimi-K3 SM120 FlashInfer MXFP4 page, "real checkpoint
contract": packed MXFP4 weights, group-32 E8M0 scales, [gate; up] halves):

  x        bf16 N(0,1)                       numpy PCG64 stream 0
  W_g      bf16 N(0,0.02) router gate [E,H]  numpy PCG64 stream 1
  bias     fp32 N(0,0.1)                     numpy PCG64 stream 2
           (skewed: bias[perm[r-1]] = 3.0 * r**-1.2, perm from stream 7)
  w13      packed E2M1 bytes [E, 2I, H/2], uniform over 256     counter stream 3
  w13_sf   UE8M0 bytes      [E, 2I, H/32], uniform in 121..127  counter stream 4
  w2       packed E2M1 bytes [E, H, I/2]                        counter stream 5
  w2_sf    UE8M0 bytes      [E, H, I/32]                        counter stream 6
  logits   fp32 [T,E] = fp32(double(x) @ double(W_g)^T)  (router GEMM is
           upstream of the routed-expert path; it is an input here)

The expert weights of the 896-expert workloads are 36.7 GB, so they come
from a counter-based generator (below) that gives the same bytes whether it
runs in numpy on the host (for any slice of experts) or in torch on the
device (for the whole tensor).
"""
from __future__ import annotations

import dataclasses
import numpy as np

SEED = 0

# stream ids (one per tensor)
S_X, S_WG, S_BIAS, S_W13, S_W13SF, S_W2, S_W2SF, S_PERM = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    skewed: bool = False
    situ_beta: float = 4.0
    situ_linear_beta: float = 25.0
    activation: str = "situ"  # or "swiglu": the clamped SwiGLU control below
    swiglu_alpha: float = 1.702
    swiglu_beta: float = 1.0
    swiglu_limit: float = 7.0
    routed_scaling_factor: float = 1.0
    sf_lo: int = 121  # UE8M0 byte range of the weight scales: 2^-6 .. 2^0
    sf_hi: int = 127

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops(self) -> float:
        """Algorithmic FLOPs of the two expert GEMMs (FC1: 2I wide, FC2: H wide)."""
        return 6.0 * self.R * self.H * self.I

    def expert_weight_bytes(self) -> float:
        """Bytes of one expert's packed weights + scales (w13 and w2)."""
        w13 = 2 * self.I * self.H // 2 + 2 * self.I * self.H // 32
        w2 = self.H * self.I // 2 + self.H * self.I // 32
        return float(w13 + w2)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=16, H=128, I=128, E=8, k=2),
    "reduced": Workload("reduced", T=128, H=7168, I=3584, E=64, k=16),
    "decode": Workload("decode", T=16, H=7168, I=3584, E=896, k=16),
    "prefill": Workload("prefill", T=8192, H=7168, I=3584, E=896, k=16),
    "skewed": Workload("skewed", T=2048, H=7168, I=3584, E=896, k=16, skewed=True),
}

# The real Kimi-K3 checkpoint runs its routed experts in a 3584-wide latent
# with I = 3072 (SM120 FlashInfer MXFP4 page, real checkpoint contract); same
# input distributions.
NEXT_WORKLOADS = {
    "real_prefill": Workload("real_prefill", T=8192, H=3584, I=3072, E=896, k=16),
    "real_decode": Workload("real_decode", T=16, H=3584, I=3072, E=896, k=16),
}

# Smaller cases of the same kernels, sized for profiler captures (a few GB on
# the device, still larger than L2): a prefill-like layer with hundreds of rows
# per touched expert, and a decode-like layer with one or two.
PROFILE_WORKLOADS = {
    "ncu_prefill": Workload("ncu_prefill", T=1536, H=7168, I=3584, E=64, k=16),
    "ncu_decode": Workload("ncu_decode", T=16, H=7168, I=3584, E=64, k=16),
}


# ----------------------------------------------------------------------------
# bf16 helpers (storage as uint16 bit patterns)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even), return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(a)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rng(stream: int, seed: int = SEED) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


# ----------------------------------------------------------------------------
# Small tensors: numpy PCG64
# ----------------------------------------------------------------------------

def gen_x(w: Workload, seed: int = SEED) -> np.ndarray:
    """bf16 activations [T, H] as uint16 bits."""
    return f32_to_bf16_bits(_rng(S_X, seed).standard_normal((w.T, w.H), dtype=np.float32))


def gen_gate_weight(w: Workload, seed: int = SEED) -> np.ndarray:
    """bf16 router gate weight [E, H] as uint16 bits."""
    g = _rng(S_WG, seed).standard_normal((w.E, w.H), dtype=np.float32) * np.float32(0.02)
    return f32_to_bf16_bits(g)


def gen_bias(w: Workload, seed: int = SEED) -> np.ndarray:
    """fp32 e_score_correction_bias [E]."""
    if not w.skewed:
        return (_rng(S_BIAS, seed).standard_normal(w.E) * 0.1).astype(np.float32)
    perm = _rng(S_PERM, seed).permutation(w.E)
    ranks = np.arange(1, w.E + 1, dtype=np.float64)
    b = np.empty(w.E, dtype=np.float64)
    b[perm] = 3.0 * ranks ** -1.2
    return b.astype(np.float32)


def gen_logits(w: Workload, x_bits: np.ndarray, wg_bits: np.ndarray) -> np.ndarray:
    """Router logits fp32 [T, E] = fp32(double(x) @ double(W_g)^T)."""
    return (bf16_bits_to_f64(x_bits) @ bf16_bits_to_f64(wg_bits).T).astype(np.float32)


# ----------------------------------------------------------------------------
# Expert weights: counter-based generator (numpy and torch give the same bytes)
# ----------------------------------------------------------------------------
# A 32-bit integer mixer (xorshift-multiply, constants from the public
# "lowbias32" hash) keyed by (seed, stream) and applied to the 64-bit word
# counter in two rounds (high word, then low word).

_M32 = 0xFFFFFFFF
_C1 = 0x7FEB352D
_C2 = 0x846CA68B


def _mix32_np(x: np.ndarray) -> np.ndarray:
    x = x & _M32
    x = x ^ (x >> 16)
    x = (x * _C1) & _M32
    x = x ^ (x >> 15)
    x = (x * _C2) & _M32
    x = x ^ (x >> 16)
    return x


def _key(stream: int, seed: int) -> int:
    k = np.array([(seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x165667B1) & _M32], dtype=np.uint64)
    return int(_mix32_np(_mix32_np(k))[0])


def _words_np(stream: int, start: int, count: int, seed: int) -> np.ndarray:
    """32-bit random words for counters [start, start+count) as uint64."""
    key = _key(stream, seed)
    c = np.arange(start, start + count, dtype=np.uint64)
    hi = _mix32_np((c >> np.uint64(32)) ^ np.uint64(key))
    return _mix32_np((c & np.uint64(_M32)) ^ hi ^ np.uint64((key * 0x9E3779B1) & _M32))


def _bytes_np(stream: int, start: int, count: int, seed: int) -> np.ndarray:
    """Uniform random bytes for flat byte offsets [start, start+count)."""
    w0, w1 = start // 4, (start + count + 3) // 4
    words = _words_np(stream, w0, w1 - w0, seed).astype(np.uint32)
    b = words.view(np.uint8)  # little-endian: byte i of word w is offset 4w+i
    off = start - 4 * w0
    return b[off:off + count].copy()


def _scales_np(stream: int, start: int, count: int, lo: int, hi: int, seed: int) -> np.ndarray:
    words = _words_np(stream, start, count, seed)
    return (lo + (words % np.uint64(hi - lo + 1))).astype(np.uint8)


def weight_shapes(w: Workload):
    return {
        "w13": (w.E, 2 * w.I, w.H // 2),
        "w13_sf": (w.E, 2 * w.I, w.H // 32),
        "w2": (w.E, w.H, w.I // 2),
        "w2_sf": (w.E, w.H, w.I // 32),
    }


def gen_expert_weights_np(w: Workload, experts, seed: int = SEED):
    """Host copy of the packed weights of the listed experts.

    Returns dict name -> array [len(experts), ...] (uint8)."""
    shp = weight_shapes(w)
    out = {}
    streams = {"w13": S_W13, "w13_sf": S_W13SF, "w2": S_W2, "w2_sf": S_W2SF}
    for name, (E, a, b) in shp.items():
        per = a * b
        arr = np.empty((len(experts), a, b), dtype=np.uint8)
        for i, e in enumerate(experts):
            if name.endswith("_sf"):
                v = _scales_np(streams[name], int(e) * per, per, w.sf_lo, w.sf_hi, seed)
            else:
                v = _bytes_np(streams[name], int(e) * per, per, seed)
            arr[i] = v.reshape(a, b)
        out[name] = arr
    return out


# ---- torch (device) version of the same generator --------------------------

def _mulmod32_t(x, c: int):
    # (x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow
    return (x * (c & 0xFFFF) + (((x * (c >> 16)) & 0xFFFF) << 16)) & _M32


def _mix32_t(x):
    x = x & _M32
    x = x ^ (x >> 16)
    x = _mulmod32_t(x, _C1)
    x = x ^ (x >> 15)
    x = _mulmod32_t(x, _C2)
    x = x ^ (x >> 16)
    return x


def _words_t(stream: int, start: int, count: int, seed: int, device):
    import torch
    key = _key(stream, seed)
    c = torch.arange(start, start + count, dtype=torch.int64, device=device)
    hi = _mix32_t((c >> 32) ^ key)
    return _mix32_t((c & _M32) ^ hi ^ ((key * 0x9E3779B1) & _M32))


def gen_expert_weights_torch(w: Workload, device, seed: int = SEED, chunk_bytes: int = 1 << 28):
    """Whole packed weight tensors generated on `device` (torch uint8)."""
    import torch
    shp = weight_shapes(w)
    streams = {"w13": S_W13, "w13_sf": S_W13SF, "w2": S_W2, "w2_sf": S_W2SF}
    out = {}
    for name, s in shp.items():
        total = s[0] * s[1] * s[2]
        t = torch.empty(total, dtype=torch.uint8, device=device)
        if name.endswith("_sf"):
            for b0 in range(0, total, chunk_bytes):
                n = min(chunk_bytes, total - b0)
                v = _words_t(streams[name], b0, n, seed, device)
                t[b0:b0 + n] = (w.sf_lo + torch.remainder(v, w.sf_hi - w.sf_lo + 1)).to(torch.uint8)
        else:
            assert total % 4 == 0 and chunk_bytes % 4 == 0
            for b0 in range(0, total, chunk_bytes):
                n = min(chunk_bytes, total - b0)
                v = _words_t(streams[name], b0 // 4, n // 4, seed, device)
                # little-endian split of each 32-bit word into 4 bytes
                by = torch.stack([(v >> (8 * i)) & 0xFF for i in range(4)], dim=1)
                t[b0:b0 + n] = by.reshape(-1).to(torch.uint8)
        out[name] = t.view(*s)
    return out


def gen_small_inputs(w: Workload, seed: int = SEED):
    """x bits, gate weight bits, bias, logits (all numpy)."""
    x = gen_x(w, seed)
    wg = gen_gate_weight(w, seed)
    bias = gen_bias(w, seed)
    logits = gen_logits(w, x, wg)
    return {"x": x, "wg": wg, "bias": bias, "logits": logits}
