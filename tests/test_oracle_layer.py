"""Whole-layer invariants of the oracle on the tiny workload: the gated
width rule, k=1, identical experts, token-permutation equivariance, masked
slots, sub-sampling, and bf16 rounding against a library conversion."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe


@pytest.fixture(scope="module")
def tiny():
    w = W.WORKLOADS["tiny"]
    s = W.gen_small_inputs(w)
    wts = W.gen_expert_weights_np(w, range(w.E))
    return w, s, wts


def test_gated_width_rule(tiny):
    w, s, wts = tiny
    assert wts["w13"].shape[1] == 256 and wts["w2"].shape[2] * 2 == 128   # 2I = 256 vs I = 128
    moe.check_shapes(w.H, w.I, wts["w13"], wts["w2"])
    bad = dict(wts, w13=wts["w13"][:, :128])                              # an un-gated FC1
    with pytest.raises(moe.ShapeError, match="256"):
        moe.forward(w, s["x"], s["logits"], s["bias"], bad)


def test_k1_output_is_the_expert_output(tiny):
    w, s, wts = tiny
    w1 = w.with_(k=1)
    r = moe.forward(w1, s["x"], s["logits"], s["bias"], wts, want_stages=True)
    assert np.allclose(r["topk_w"], 1.0)
    assert np.array_equal(r["out"], r["y"][:, 0])


def test_identical_experts_give_routing_independent_output(tiny):
    w, s, wts = tiny
    same = {k: np.repeat(v[:1], w.E, axis=0) for k, v in wts.items()}
    r = moe.forward(w, s["x"], s["logits"], s["bias"], same, want_stages=True)
    assert np.allclose(r["out"], r["y"][:, 0], rtol=1e-13, atol=1e-9)
    r2 = moe.forward(w, s["x"], s["logits"][:, ::-1].copy(), s["bias"], same)
    assert np.allclose(r["out"], r2["out"], rtol=1e-13, atol=1e-9)


def test_token_permutation_equivariance(tiny):
    w, s, wts = tiny
    perm = np.random.default_rng(0).permutation(w.T)
    r = moe.forward(w, s["x"], s["logits"], s["bias"], wts)
    rp = moe.forward(w, s["x"][perm], s["logits"][perm], s["bias"], wts)
    assert np.array_equal(r["out"][perm], rp["out"])


def test_masked_slot_and_token_subset(tiny):
    w, s, wts = tiny
    r = moe.forward(w, s["x"], s["logits"], s["bias"], wts, want_stages=True)
    ids = r["ids"].copy()
    ids[:, 1] = -1
    rm = moe.forward(w, s["x"], s["logits"], s["bias"], wts, ids=ids, topk_w=r["topk_w"], want_stages=True)
    assert np.array_equal(rm["out"], r["topk_w"][:, :1] * r["y"][:, 0])
    sub = [3, 7, 11]
    rs = moe.forward(w, s["x"], s["logits"], s["bias"], wts, tokens=sub)
    assert np.array_equal(rs["out"], r["out"][sub])
    # an expert subset gives the same rows when it covers the routed experts
    ex = sorted(set(r["ids"][sub].ravel().tolist()))
    part = {k: v[ex] for k, v in wts.items()}
    rs2 = moe.forward(w, s["x"], s["logits"], s["bias"], part, experts_host=ex, tokens=sub)
    assert np.array_equal(rs2["out"], rs["out"])


def test_intermediate_scale_bound(tiny):
    w, s, wts = tiny
    r = moe.forward(w, s["x"], s["logits"], s["bias"], wts, want_stages=True)
    # |SiTU| < 4 * 25, so every intermediate scale exponent is <= -2 (byte <= 125)
    assert r["inter_s"].max() <= 125


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(9)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(moe.bf16_round(v), ref)
