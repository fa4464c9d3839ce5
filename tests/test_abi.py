"""CPU checks of the C ABI library: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching a GPU.
Also: the workload generator gives identical bytes in numpy and torch."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    return K


def test_library_exports_every_declared_symbol(K):
    hdr = open(os.path.join(ROOT, "include", "kmoe.h")).read()
    declared = set(re.findall(r"^\s*(?:const char\*|int|size_t)\s+(kmoe_\w+)\s*\(", hdr, re.M))
    assert {"kmoe_route", "kmoe_quantize_mx", "kmoe_forward"} <= declared
    lib = ctypes.CDLL(K.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(K.EXPORTS) == declared


def test_status_strings_and_workspace(K):
    for s in range(9):
        assert K.kmoe_status_string(s)
    p = K.make_params(8192, 7168, 3584, 896, 16)
    L = K.kmoe_workspace_layout(p)
    assert (L.tile_rows, L.tile_rows_big, L.big_rows) == (64, 224, 64) and L.total == K.kmoe_workspace_size(p)
    offs = [L.err, L.topk_ids, L.topk_w, L.counts, L.seg_start, L.tile_start, L.row_of_slot, L.slot_of_row,
            L.xq, L.xsf, L.iq, L.isf, L.y]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.y + 8192 * 16 * 7168 * 4 <= L.total
    for args, rows in (((16, 7168, 3584, 896, 16), (32, 0)), ((128, 7168, 3584, 64, 16), (64, 224)),
                       ((64, 7168, 3584, 64, 16), (32, 0))):
        Ld = K.kmoe_workspace_layout(K.make_params(*args))
        assert (Ld.tile_rows, Ld.tile_rows_big) == rows
    assert L.isf < L.tile_start_big < L.xsf_big < L.isf_big < L.total


def test_host_side_argument_errors(K):
    lib = K.lib()
    bad = [K.make_params(16, 100, 128, 8, 2),      # H not a multiple of 128
           K.make_params(16, 128, 96, 8, 2),       # I not a multiple of 128
           K.make_params(16, 128, 128, 8, 9),      # k > E
           K.make_params(-1, 128, 128, 8, 2),
           K.make_params(16, 128, 128, 8, 2, situ_beta=0.0),                          # SiTU beta not > 0
           K.make_params(16, 128, 128, 8, 2, activation="swiglu", swiglu_limit=0.0),  # clamp not > 0
           K.make_params(16, 128, 128, 8, 2, activation="swiglu", swiglu_alpha=float("inf")),
           K.make_params(16, 128, 128, 8, 2, activation="swiglu", swiglu_beta=float("nan"))]
    p_flag = K.make_params(16, 128, 128, 8, 2)
    p_flag.flags = 2                                                                   # unknown flag bit
    bad.append(p_flag)
    assert K.kmoe_workspace_size(K.make_params(16, 128, 128, 8, 2, activation="swiglu")) > 0
    with pytest.raises(ValueError):
        K.make_params(16, 128, 128, 8, 2, activation="gelu")
    for p in bad:
        assert K.kmoe_workspace_size(p) == 0
        st = lib.kmoe_forward(ctypes.byref(p), None, None, None, None, None, None, None, None, None, 0, None)
        assert st in (1, 2)
    assert lib.kmoe_route(None, None, 4, 8, 9, None, None, None) == 1
    # the fused router: shapes, pointers, alignment and workspace are checked on the host
    nr = K.kmoe_router_workspace_size(300, 128, 8)
    assert nr >= 512 and K.kmoe_router_workspace_size(-1, 128, 8) == 0
    assert K.kmoe_router_workspace_size(16, 96, 8) == 0 and K.kmoe_router_workspace_size(16, 128, 2000) == 0
    # decode-sized routers split K: the partial sums are part of the workspace
    assert K.kmoe_router_workspace_size(16, 7168, 896) > 5 * 16 * 896 * 4
    r = lib.kmoe_router
    assert r(16, 16, 16, 4, 128, 6, 2, 16, 16, 16, 256, nr, None) == 2      # E not a multiple of 4
    assert r(16, 16, 16, 4, 96, 8, 2, 16, 16, 16, 256, nr, None) == 2       # H not a multiple of 64
    assert r(16, 16, 16, 4, 128, 8, 9, 16, 16, 16, 256, nr, None) == 1      # k > E
    assert r(None, 16, 16, 4, 128, 8, 2, 16, 16, 16, 256, nr, None) == 1    # no x
    assert r(8, 16, 16, 4, 128, 8, 2, 16, 16, 16, 256, nr, None) == 3       # x not 16-byte aligned
    assert r(16, 16, 16, 4, 128, 8, 2, 16, 16, 16, 256, 16, None) == 5      # workspace too small
    assert r(16, 16, 16, 4, 128, 8, 2, 16, 16, 16, 128, nr, None) == 3      # workspace not 256-byte aligned
    assert r(16, 16, 16, 4, 128, 8, 2, 8, 16, 16, 256, nr, None) == 3       # logits not 16-byte aligned
    pr = K.make_params(16, 128, 128, 6, 2)
    assert lib.kmoe_forward_router(ctypes.byref(pr), 16, 16, 16, 256, 256, 16, 256, 1 << 30, None, None) == 2
    assert lib.kmoe_quantize_mx(None, 4, 100, 0, None, None, None) == 2
    assert lib.kmoe_quantize_mx(None, 4, 128, 7, None, None, None) == 1
    p = K.make_params(16, 128, 128, 8, 2)
    n = K.kmoe_workspace_size(p)
    # workspace too small / misaligned pointers are rejected before any CUDA call
    assert lib.kmoe_forward(ctypes.byref(p), 16, 16, 16, 256, 256, None, None, 16, 256, n - 1, None) == 5
    assert lib.kmoe_forward(ctypes.byref(p), 16, 16, 16, 256, 256, None, None, 16, 258, n, None) == 3
    assert lib.kmoe_forward(ctypes.byref(p), 8, 16, 16, 256, 256, None, None, 16, 256, n, None) == 3
    assert lib.kmoe_forward(ctypes.byref(p), 16, 16, 16, 128, 256, None, None, 16, 256, n, None) == 3
    assert K.kmoe_prepared_weight_bytes(p, 0) == 8 * 2 * 1 * 8704 and K.kmoe_prepared_weight_bytes(p, 1) == 8 * 8704
    # tile 1, row 33, group 5 (K block 1) of K = 256 (2 K blocks), 32-row tiles
    assert lib.kmoe_tile_sf_offset(1, 33, 5, 32, 256, 10) == ((1 * 2 + 1) * 1 + 0) * 512 + 1 * 16 + 1 * 4 + 1


def test_weight_generator_numpy_equals_torch():
    w = W.WORKLOADS["tiny"]
    a = W.gen_expert_weights_np(w, range(w.E))
    b = W.gen_expert_weights_torch(w, "cpu", chunk_bytes=4096)
    for k in a:
        assert np.array_equal(a[k], b[k].numpy()), k
    big = W.WORKLOADS["decode"]
    sub = W.gen_expert_weights_np(big, [5])
    # the counter stream is position-addressed: expert 5 alone equals its slice of a longer draw
    per = 2 * big.I * big.H // 32
    words = W._scales_np(W.S_W13SF, 4 * per, 2 * per, big.sf_lo, big.sf_hi, W.SEED)
    assert np.array_equal(sub["w13_sf"][0].ravel(), words[per:])


def test_binding_rejects_mis_sized_tensors_before_the_library(K):
    """The C ABI sees plain pointers; the binding checks every caller tensor's
    dtype, shape or byte size before a pointer reaches the library (host
    tensors here: the size checks come before the device check)."""
    bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8

    def rejects(fn, needle):
        with pytest.raises(ValueError, match=needle):
            fn()

    lg = torch.zeros(4, 8)
    rejects(lambda: K.kmoe_route(lg, torch.zeros(7), 2), r"bias must have shape \(8,\)")
    rejects(lambda: K.kmoe_route(lg, torch.zeros(8), 2, topk_ids=torch.zeros(4, 3, dtype=i32)), "topk_ids")
    rejects(lambda: K.kmoe_route(lg, torch.zeros(8), 2, topk_ids=torch.zeros(4, 2)), "topk_ids must be torch.int32")
    rejects(lambda: K.kmoe_route(torch.zeros(8), torch.zeros(8), 2), "2-D")
    rejects(lambda: K.kmoe_route(lg, torch.zeros(8), 2), "CUDA tensor")   # sizes right, host memory
    x = torch.zeros(4, 128, dtype=bf)
    rejects(lambda: K.kmoe_quantize_mx(x, codes=torch.zeros(4, 64, dtype=u8)), "codes must have shape")
    rejects(lambda: K.kmoe_quantize_mx(x, K.KMOE_MXFP4_E2M1, codes=torch.zeros(4, 128, dtype=u8)), "codes")
    rejects(lambda: K.kmoe_quantize_mx(x, scales=torch.zeros(4, 2, dtype=u8)), "scales")

    p = K.make_params(4, 128, 128, 8, 2)
    w13 = torch.zeros(K.kmoe_prepared_weight_bytes(p, 0), dtype=u8)
    w2 = torch.zeros(K.kmoe_prepared_weight_bytes(p, 1), dtype=u8)
    b = torch.zeros(8)
    fwd = K.kmoe_forward
    rejects(lambda: fwd(p, torch.zeros(4, 256, dtype=bf), lg, b, w13, w2), r"x must have shape \(4, 128\)")
    rejects(lambda: fwd(p, x.float(), lg, b, w13, w2), "x must be torch.bfloat16")
    rejects(lambda: fwd(p, x, lg, b, w13[:-1], w2), "w13_k holds")
    rejects(lambda: fwd(p, x, lg, b, w13, w2[:-16]), "w2_k holds")
    rejects(lambda: fwd(p, x, torch.zeros(4, 9), b, w13, w2), "logits must have shape")
    rejects(lambda: fwd(p, x, None, None, w13, w2, topk_ids=torch.zeros(4, 3, dtype=i32),
                        topk_w=torch.zeros(4, 3)), "topk_ids")
    rejects(lambda: fwd(p, x, lg, b, w13, w2, out=torch.zeros(4, 128)), "out must be torch.bfloat16")
    rejects(lambda: fwd(p, x, lg, b, w13, w2, workspace=torch.zeros(K.kmoe_workspace_size(p), dtype=f32)),
            "workspace must be torch.uint8")
    rejects(lambda: fwd(p, x, lg, b, w13, w2, workspace=torch.zeros(K.kmoe_workspace_size(p) - 1, dtype=u8)),
            "workspace holds")
    rejects(lambda: K.kmoe_forward_noalloc(p, x, lg, b, w13, w2, device_error=torch.zeros(0, dtype=i32)),
            "device_error holds")
    # the fused router: gate weight [E, H], logits [T, E]
    wg = torch.zeros(8, 128, dtype=bf)
    rejects(lambda: K.kmoe_router(x, torch.zeros(8, 64, dtype=bf), b, 2), r"w_gate must have shape \(8, 128\)")
    rejects(lambda: K.kmoe_router(x, wg, b, 2, logits=torch.zeros(4, 7)), "logits")
    rejects(lambda: K.kmoe_router(x, wg, b, 2, workspace=torch.zeros(1, dtype=u8)), "workspace holds")
    rejects(lambda: K.kmoe_forward_router(p, x, torch.zeros(9, 128, dtype=bf), b, w13, w2), "w_gate")
    rejects(lambda: K.kmoe_device_error(torch.zeros(3, dtype=u8)), "workspace holds")


def _worst_tiles(T, E, k, BN, big_rows, big_tile_rows):
    """Adversarial per-expert row counts (each expert at most T rows, the sum
    R = T*k, at most E experts) that maximise the tile count of each class:
    small tiles favour many experts of 1, BN+1, 2BN+1, ... rows up to big_rows;
    big tiles favour experts of big_rows+1 rows.  Returns (small, big)."""
    R = T * k
    small_cap = min(T, big_rows) if big_rows else T
    # small class: one row per expert first, then BN more rows per extra tile
    counts = [0] * E
    left = R
    for e in range(min(E, left)):
        counts[e] = 1
    left -= min(E, R)
    grew = True
    while left >= BN and grew:
        grew = False
        for e in range(E):
            if left >= BN and counts[e] and counts[e] + BN <= small_cap:
                counts[e] += BN
                left -= BN
                grew = True
    small = sum(-(-c // BN) for c in counts if 0 < c <= (big_rows or T))
    # big class: as many experts of big_rows + 1 rows as the rows and the experts allow
    big = 0
    if big_rows and T > big_rows:
        n = min(E, R // (big_rows + 1))
        big = n
        extra = R - n * (big_rows + 1)
        # more tiles on those experts: the next boundary (big_tile_rows + 1
        # rows) first, then one tile per big_tile_rows, each expert at most T rows
        step1 = big_tile_rows + 1 - (big_rows + 1)
        if T >= big_tile_rows + 1 and step1 > 0:
            first = min(n, extra // step1)
            big += first
            extra -= first * step1
            per_expert = (T - (big_tile_rows + 1)) // big_tile_rows
            big += min(extra // big_tile_rows, first * per_expert)
    return small, big


@pytest.mark.parametrize("T,E,k", [(8192, 896, 16), (2048, 896, 16), (128, 64, 16), (16, 896, 16), (16, 8, 2),
                                   (65, 1024, 32), (300, 200, 8), (1, 1, 1), (64, 64, 16), (1000, 37, 5)])
def test_workspace_tile_capacity_covers_adversarial_routing(K, T, E, k):
    L = K.kmoe_workspace_layout(K.make_params(T, 128, 128, E, k))
    small, big = _worst_tiles(T, E, k, L.tile_rows, L.big_rows if L.tile_rows_big else 0, 224)
    assert small <= L.max_tiles, (small, L.max_tiles)
    assert big <= (L.max_tiles_big if L.tile_rows_big else 0), (big, L.max_tiles_big)
