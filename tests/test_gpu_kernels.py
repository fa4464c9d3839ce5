"""GPU parity of the routing and quantisation kernels against the oracle,
through the C ABI: bit-exact ids, codes and scales; weights to fp32
rounding; edge cases; the bounded-wait self-test and device error reporting."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


def test_check_device(K):
    assert K.kmoe_check_device(0) == 0


@pytest.mark.parametrize("name", ["tiny", "reduced", "decode", "prefill", "skewed"])
def test_route_bit_exact(K, name):
    w = W.WORKLOADS[name]
    s = W.gen_small_inputs(w)
    ids_ref, w_ref, _ = O.route(s["logits"], s["bias"], w.k)
    ids, wts = K.kmoe_route(torch.from_numpy(s["logits"]).cuda(), torch.from_numpy(s["bias"]).cuda(), w.k)
    ids = ids.cpu().numpy()
    wts = wts.cpu().numpy().astype(np.float64)
    assert np.array_equal(ids, ids_ref), f"{(ids != ids_ref).sum()} routing ids differ"
    assert np.allclose(wts, w_ref, rtol=1e-6, atol=0)
    assert np.allclose(wts.sum(1), 1.0, atol=1e-6)


def test_route_ties_and_k_equals_e(K):
    T, E = 5, 64
    logits = np.zeros((T, E), np.float32)
    logits[1, [3, 40, 41]] = 2.0                  # exact ties
    logits[2] = np.linspace(-3, 3, E, dtype=np.float32)
    bias = np.zeros(E, np.float32)
    bias[7] = 0.5
    for k in (1, 3, 16, 32):
        ref, wref, _ = O.route(logits, bias, k)
        ids, wts = K.kmoe_route(torch.from_numpy(logits).cuda(), torch.from_numpy(bias).cuda(), k)
        assert np.array_equal(ids.cpu().numpy(), ref)
        assert np.allclose(wts.cpu().numpy(), wref, rtol=1e-6)
    E = 8
    lg = np.random.default_rng(0).standard_normal((7, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    ref, _, _ = O.route(lg, b, E)
    ids, _ = K.kmoe_route(torch.from_numpy(lg).cuda(), torch.from_numpy(b).cuda(), E)
    assert np.array_equal(ids.cpu().numpy(), ref)


def test_route_every_selection_path(K):
    """Tokens built to take each of the kernel's three selection paths (the
    lane-maximum bound, the radix select, the k rounds of arg-max) and edge
    keys: NaN logits, a 40-way tie at the top, keys concentrated in one lane."""
    E, k = 896, 16
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((6, E)).astype(np.float32)
    lg[1, ::32] = 5.0 + 0.01 * rng.standard_normal(E // 32).astype(np.float32)  # all in lane 0's experts
    lg[2] = 0.0                                                                   # every key equal
    lg[3, rng.choice(E, 40, replace=False)] = 4.0                                 # 40 equal keys on top
    lg[4, rng.choice(E, 100, replace=False)] = np.nan                             # NaN -> never chosen
    lg[5] = -30.0 + 0.001 * rng.standard_normal(E).astype(np.float32)             # tiny scores
    for bias in (np.zeros(E, np.float32), (0.01 * rng.standard_normal(E)).astype(np.float32)):
        ref, wref, _ = O.route(lg, bias, k)
        ids, wts = K.kmoe_route(torch.from_numpy(lg).cuda(), torch.from_numpy(bias).cuda(), k)
        assert np.array_equal(ids.cpu().numpy(), ref)
        assert np.allclose(wts.cpu().numpy(), wref, rtol=1e-6)


def _quant_check(K, xbits, fmt):
    x = torch.from_numpy(xbits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = K.kmoe_quantize_mx(x, fmt)
    xf = W.bf16_bits_to_f64(xbits)
    name = "e4m3" if fmt == K.KMOE_MXFP8_E4M3 else "e2m1"
    qref, sref = F.quantize_mx(xf, name)
    if name == "e2m1":
        qref = F.pack_e2m1(qref)
    c = codes.cpu().numpy()
    sc = scales.cpu().numpy()
    assert np.array_equal(sc, sref), f"{(sc != sref).sum()} scale bytes differ"
    assert np.array_equal(c, qref), f"{(c != qref).sum()} code bytes differ"


@pytest.mark.parametrize("name", ["tiny", "reduced", "decode", "prefill"])
def test_quantize_mxfp8_bit_exact(K, name):
    w = W.WORKLOADS[name]
    _quant_check(K, W.gen_x(w), K.KMOE_MXFP8_E4M3)


def test_quantize_edge_cases(K):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    x[0, :32] = 0.0                                   # all-zero group
    x[1, 5] = np.inf                                  # inf group
    x[2, 7] = -np.inf
    x[3, 9] = np.nan                                  # NaN ignored by the absmax, becomes +0
    x[4, :] = 1e-40                                   # bf16 subnormals
    x[5, :] = 448.0                                   # exactly qmax
    x[6, :] = -0.0
    x[7, :32] = 3.0e38                                # near the bf16 maximum
    x[8, 0] = 1.0
    x[8, 1:32] = 2.0 ** -20                           # tiny next to a large value
    bits = W.f32_to_bf16_bits(x)
    bits[3, 9] = 0x7FC0
    for fmt in (K.KMOE_MXFP8_E4M3, K.KMOE_MXFP4_E2M1):
        _quant_check(K, bits, fmt)


def test_quantize_mxfp4_bit_exact(K):
    w = W.WORKLOADS["reduced"]
    _quant_check(K, W.gen_x(w)[:64], K.KMOE_MXFP4_E2M1)


def test_bounded_wait_timeout_keeps_context(K):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    K.kmoe_selftest_wait_timeout(ws, 2000)
    st, word = K.kmoe_device_error(ws)
    assert st == 7 and (word & 1)
    st, word = K.kmoe_device_error(ws)     # cleared
    assert st == 0 and word == 0
    # the context still works
    ids, _ = K.kmoe_route(torch.zeros(2, 8, device="cuda"), torch.zeros(8, device="cuda"), 2)
    assert ids.cpu().tolist() == [[0, 1], [0, 1]]


def test_mma_peak_kernel_runs(K):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    flops = K.kmoe_mma_peak_run(2000, 224, ws)
    torch.cuda.synchronize()
    st, word = K.kmoe_device_error(ws)
    assert st == 0 and word == 0
    assert flops == torch.cuda.get_device_properties(0).multi_processor_count * 2000 * 4 * 2 * 128 * 224 * 32
    with pytest.raises(K.KmoeError):
        K.kmoe_mma_peak_run(10, 200, ws)   # N not a multiple of 16


# ---------------------------------------------------------------- the FC1 activation's error
# The FC1 epilogue evaluates SiTU (and the SwiGLU control) in fp32 from fast
# exponentials; the oracle evaluates the formula in double.  The relative
# error bound asserted here is what keeps intermediate-code flips rare: a
# value flips to the neighbouring E4M3 code only if it lies within that
# relative distance of a rounding midpoint (midpoints sit 2^-4 .. 2^-3 apart
# in relative terms), so a bound of 2^-18 allows flips on about 2^-18 * 2^4 =
# 6e-5 of the values at most.
ACT_REL_BOUND = 2.0 ** -18


# (g, u) points at the end of the activation inputs; the first three have an
# exact zero in g or u
SPECIAL_GU = [(0.0, 3.0), (-0.0, 3.0), (5.0, 0.0), (1e-30, 1e-30), (4.0, 25.0), (-4.0, 25.0), (25.0, -4.0),
              (-25.0, 4.0), (88.0, 1.0), (-88.0, 1.0), (1e30, 1e30), (-1e30, 1.0), (np.inf, 2.0),
              (-np.inf, np.inf)]


def _activation_inputs():
    rng = np.random.default_rng(11)
    parts = [rng.normal(0, 108, (2, 400000)), rng.normal(0, 14.5, (2, 400000)), rng.uniform(-40, 40, (2, 400000)),
             rng.uniform(-1, 1, (2, 200000)), rng.uniform(-1e-3, 1e-3, (2, 100000)),
             np.array(SPECIAL_GU).T]
    gu = np.concatenate(parts, axis=1).astype(np.float32)
    return gu[0], gu[1]


@pytest.mark.parametrize("act,params", [("situ", dict(situ_beta=4.0, situ_linear_beta=25.0)),
                                        ("situ", dict(situ_beta=2.0, situ_linear_beta=10.0)),
                                        ("swiglu", dict(swiglu_alpha=1.702, swiglu_beta=1.0, swiglu_limit=7.0))],
                         ids=["situ_4_25", "situ_2_10", "swiglu"])
def test_activation_error_bound(K, act, params):
    g, u = _activation_inputs()
    if act == "swiglu":
        # -Inf * sigmoid(-Inf) has no value (the forward maps such a NaN
        # activation to +0 when it requantises); finite inputs only here
        keep = np.isfinite(g) & np.isfinite(u)
        g, u = g[keep], u[keep]
    p = K.make_params(0, 128, 128, 1, 1, activation=act, **params)
    out = K.kmoe_selftest_activation(p, torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda()).cpu().numpy()
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    # the library receives the parameters as fp32 (kmoe_params): the oracle
    # evaluates the formula in double with those same values
    f32 = {n: float(np.float32(v)) for n, v in params.items()}
    if act == "situ":
        ref = O.situ(gd, ud, f32["situ_beta"], f32["situ_linear_beta"])
    else:
        ref = O.swiglu(gd, ud, f32["swiglu_alpha"], f32["swiglu_beta"], f32["swiglu_limit"])
    assert np.all(np.isfinite(out))
    big = np.abs(ref) > 1e-30
    rel = np.abs(out[big].astype(np.float64) - ref[big]) / np.abs(ref[big])
    tiny_abs = np.abs(out[~big].astype(np.float64) - ref[~big]).max(initial=0.0)
    print(f"{act} {params}: max relative error {rel.max():.3e} (= {rel.max() / 2 ** -24:.1f} x 2^-24), "
          f"mean {rel.mean():.3e}; |ref| <= 1e-30: max abs error {tiny_abs:.1e}")
    assert rel.max() <= ACT_REL_BOUND
    assert tiny_abs <= 1e-30
    # exact zeros stay zero (SiTU(0, u) = SiTU(g, 0) = 0)
    if act == "situ":
        n0 = len(out) - len(SPECIAL_GU)
        assert out[n0] == 0.0 and out[n0 + 1] == 0.0 and out[n0 + 2] == 0.0
