"""The no-allocation forward (kmoe_forward_noalloc) against kmoe_forward.

Some hosts cannot allocate device memory (they own all of it, or receive a
stream and no allocator), so the library offers a forward that uses a fixed
scratch array built into it instead of a caller workspace.  These tests call
that entry point through the C ABI twice in a row, with different inputs, and
compare each result with kmoe_forward's on the same inputs, within the output
tolerance the parity tests use.  This file sorts last so that a run stopping at
the first failure has already run every other test; it also passes alone."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests._moe_setup import assert_output_parity, device_inputs, device_weights, params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


def _pair(K, w, seed):
    wt = device_weights(w)
    s = W.gen_small_inputs(w, seed=seed)
    inp, _ = device_inputs(w, s)
    p = params(w)
    ref, ws = K.kmoe_forward(p, inp["x"], inp["logits"], inp["bias"], wt["w13_k"], wt["w2_k"])
    out = torch.full((w.T, w.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lib = K.lib()
    st = lib.kmoe_forward_noalloc(ctypes.byref(p), ctypes.c_void_p(inp["x"].data_ptr()),
                                  ctypes.c_void_p(inp["logits"].data_ptr()), ctypes.c_void_p(inp["bias"].data_ptr()),
                                  ctypes.c_void_p(wt["w13_k"].data_ptr()), ctypes.c_void_p(wt["w2_k"].data_ptr()),
                                  None, None, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(err.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0, K.kmoe_status_string(st)
    assert int(err.item()) == 0
    return ref, out


@pytest.mark.parametrize("w", [W.WORKLOADS["tiny"], W.PROFILE_WORKLOADS["ncu_decode"]], ids=["tiny", "T16_E64"])
def test_noalloc_matches_forward_twice(K, w):
    first_ref, first = _pair(K, w, seed=0)
    second_ref, second = _pair(K, w, seed=1)       # second call, new inputs, same shared scratch
    for ref, got in ((first_ref, first), (second_ref, second)):
        r = ref.float().cpu().numpy().astype(np.float64)
        assert_output_parity(got, r, "noalloc vs forward")
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert not torch.equal(first.view(torch.int16), second.view(torch.int16))


def test_noalloc_rejects_layers_beyond_its_scratch(K):
    p = K.make_params(8192, 7168, 3584, 896, 16)
    assert K.kmoe_workspace_size(p) > K.NOALLOC_SCRATCH_BYTES
    st = K.lib().kmoe_forward_noalloc(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None)
    assert st == 5  # KMOE_ERR_WORKSPACE
