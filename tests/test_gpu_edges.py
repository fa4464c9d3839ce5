"""Empty batches through every compute entry point of the C ABI.  T = 0 (no
tokens, e.g. an expert-parallel rank that received none) is a valid call:
it returns KMOE_OK, launches nothing, writes nothing, and the context and the
next non-empty call are unaffected."""
import numpy as np
import pytest
import torch

import workloads as W
from tests._moe_setup import assert_output_parity, device_weights, oracle_forward, params, run_forward

pytestmark = pytest.mark.gpu

TINY = W.WORKLOADS["tiny"]


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


def test_empty_batch_every_entry_point(K):
    w = TINY
    dev = "cuda"
    x0 = torch.empty((0, w.H), dtype=torch.bfloat16, device=dev)
    lg0 = torch.empty((0, w.E), dtype=torch.float32, device=dev)
    bias = torch.zeros(w.E, dtype=torch.float32, device=dev)
    wg = torch.zeros((w.E, w.H), dtype=torch.bfloat16, device=dev)

    ids, wts = K.kmoe_route(lg0, bias, w.k)
    assert ids.shape == (0, w.k) and wts.shape == (0, w.k)

    for fmt in (K.KMOE_MXFP8_E4M3, K.KMOE_MXFP4_E2M1):
        codes, scales = K.kmoe_quantize_mx(x0, fmt)
        assert codes.shape[0] == 0 and scales.shape == (0, w.H // 32)

    ids, wts, logits, ws = K.kmoe_router(x0, wg, bias, w.k)
    assert logits.shape == (0, w.E) and ids.shape == (0, w.k)
    assert K.kmoe_router_workspace_size(0, w.H, w.E) > 0

    wt = device_weights(w)
    p0 = params(w, T=0)
    # the output buffer keeps its contents: nothing is written
    sentinel = torch.full((1, w.H), 7.0, dtype=torch.bfloat16, device=dev)
    out, ws = K.kmoe_forward(p0, x0, lg0, bias, wt["w13_k"], wt["w2_k"], out=sentinel[:0])
    assert out.shape == (0, w.H)
    out, ws = K.kmoe_forward_router(p0, x0, wg, bias, wt["w13_k"], wt["w2_k"])
    assert out.shape == (0, w.H)
    out = K.kmoe_forward_noalloc(p0, x0, lg0, bias, wt["w13_k"], wt["w2_k"])
    assert out.shape == (0, w.H)
    torch.cuda.synchronize()
    assert torch.all(sentinel.float() == 7.0)

    # an empty batch through the no-allocation forward reports its own (empty)
    # error word, not the one an earlier call left in the shared scratch: the
    # earlier call routes a slot to expert 99 >= E (error bit 2)
    import ctypes
    p1 = params(w, T=1)
    x1 = torch.zeros((1, w.H), dtype=torch.bfloat16, device=dev)
    bad_ids = torch.tensor([[1, 99]], dtype=torch.int32, device=dev)
    bad_w = torch.tensor([[0.5, 0.5]], dtype=torch.float32, device=dev)
    o1 = torch.empty((1, w.H), dtype=torch.bfloat16, device=dev)
    err = torch.full((1,), -1, dtype=torch.int32, device=dev)
    lib = K.lib()
    cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.kmoe_forward_noalloc(ctypes.byref(p1), ctypes.c_void_p(x1.data_ptr()), None, None,
                                  ctypes.c_void_p(wt["w13_k"].data_ptr()), ctypes.c_void_p(wt["w2_k"].data_ptr()),
                                  ctypes.c_void_p(bad_ids.data_ptr()), ctypes.c_void_p(bad_w.data_ptr()),
                                  ctypes.c_void_p(o1.data_ptr()), ctypes.c_void_p(err.data_ptr()), cur)
    torch.cuda.synchronize()
    assert st == 0 and (int(err.item()) & 2)
    err.fill_(-1)
    st = lib.kmoe_forward_noalloc(ctypes.byref(p0), None, None, None, ctypes.c_void_p(wt["w13_k"].data_ptr()),
                                  ctypes.c_void_p(wt["w2_k"].data_ptr()), None, None, None,
                                  ctypes.c_void_p(err.data_ptr()), cur)
    torch.cuda.synchronize()
    assert st == 0 and int(err.item()) == 0

    # the next non-empty call is unaffected
    out, ws, p, s, _ = run_forward(w)
    tokens = np.arange(w.T)
    ref = oracle_forward(w, s, tokens)
    assert_output_parity(out, ref["out"], "after_empty_batches")
