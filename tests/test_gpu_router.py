"""GPU parity of the fused router (gate GEMM + top-k routing in one kernel,
kmoe_router / kmoe_forward_router through the C ABI) against the float64
oracle.

- logits: within the fp32 accumulation error of the exact dot products
  (per element below the worst-case bound H * 2^-23 * sum_h |x_h w_h|, and the
  largest error below 2e-5 x max|logit|);
- routing: decided in the kernel's precision, so the ids must equal the
  oracle's routing of the kernel's own logits exactly (weights to 1e-6), and
  the oracle's routing of the exact logits on every token whose k-th and
  (k+1)-th keys are further apart than the logit error can move them;
- the forward with the fused router equals the forward given the router's
  logits bit for bit, and matches the oracle on sampled tokens."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O
from tests._moe_setup import (assert_output_parity, bf16_to_torch, device_weights, params)

pytestmark = pytest.mark.gpu

# a ragged case: three token tiles (the last one partial), 200 experts (the
# last expert chunk partial), H of two 128-wide blocks
RAGGED = W.WORKLOADS["tiny"].with_(name="router_ragged", T=300, H=256, E=200, k=8)
CASES = {
    "tiny": W.WORKLOADS["tiny"],
    "tiny_k_eq_E": W.WORKLOADS["tiny"].with_(name="tiny_k8", k=8),
    "T1": W.WORKLOADS["tiny"].with_(name="router_T1", T=1, H=512, E=64, k=4),
    "ragged": RAGGED,
    # CTA pairs (prefill-sized plan) with an odd number of token tiles (the
    # last pair's second CTA has no tokens) and a partial last expert chunk
    "pair_odd_tiles": W.WORKLOADS["tiny"].with_(name="router_pair_odd", T=2100, H=512, E=900, k=16),
    "reduced": W.WORKLOADS["reduced"],
    "decode": W.WORKLOADS["decode"],
    "skewed": W.WORKLOADS["skewed"],
    "prefill": W.WORKLOADS["prefill"],
    # the real checkpoint's hidden size (H = 3584): CTA pairs at T = 8192, split K at T = 16
    "real_prefill": W.NEXT_WORKLOADS["real_prefill"],
    "real_decode": W.NEXT_WORKLOADS["real_decode"],
    # the largest expert count and top-k the routing supports
    "max_e_k": W.WORKLOADS["tiny"].with_(name="router_max_e_k", T=300, H=256, E=1024, k=32),
}


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


def _run_router(K, w, s):
    x = bf16_to_torch(s["x"], "cuda")
    wg = bf16_to_torch(s["wg"], "cuda")
    bias = torch.from_numpy(s["bias"]).cuda()
    ids, wts, logits, ws = K.kmoe_router(x, wg, bias, w.k)
    torch.cuda.synchronize()
    st, word = K.kmoe_device_error(ws)
    assert st == 0, f"device error word {word:#x}"
    return ids.cpu().numpy(), wts.cpu().numpy(), logits.cpu().numpy()


def _key_gaps(logits, bias, k):
    """Per token: the gap between the k-th and (k+1)-th largest keys (inf when
    k = E), and the smallest gap between neighbours among the k+1 largest."""
    key = O.sigmoid_fp32(logits).astype(np.float64) + bias.astype(np.float64)[None, :]
    srt = -np.sort(-key, axis=1)
    if k >= key.shape[1]:
        top = srt
        kth = np.full(key.shape[0], np.inf)
    else:
        top = srt[:, :k + 1]
        kth = srt[:, k - 1] - srt[:, k]
    order = np.min(top[:, :-1] - top[:, 1:], axis=1) if top.shape[1] > 1 else np.full(key.shape[0], np.inf)
    return kth, order


def check_router(w, s, ids, wts, logits):
    ref = O.router_logits(s["x"], s["wg"]).astype(np.float64)
    got = logits.astype(np.float64)
    err = np.abs(got - ref)
    absdot = np.abs(F.bf16_decode(s["x"])) @ np.abs(F.bf16_decode(s["wg"])).T
    bound = w.H * 2.0 ** -23 * absdot
    rel = err.max() / max(np.abs(ref).max(), 1e-30)
    print(f"{w.name}: logits max err {err.max():.3e} ({rel:.2e} of max|logit|), "
          f"max err / bound {np.max(err / np.maximum(bound, 1e-300)):.2e}")
    assert np.all(err <= bound)
    assert rel <= 5e-5
    # the routing decision in the kernel's precision: exactly the oracle's
    ids_k, w_k, _ = O.route(logits, s["bias"], w.k)
    assert np.array_equal(ids, ids_k)
    assert np.allclose(wts, w_k, rtol=1e-6, atol=1e-7)
    # against the exact logits: equal wherever the logit error cannot reorder the k-th key
    ids_x, _, _ = O.route(ref.astype(np.float32), s["bias"], w.k)
    # (a key moves by at most a quarter of its logit's error plus two fp32 roundings)
    delta = err.max() / 4 + 2 * 2.0 ** -23
    kth_gap, order_gap = _key_gaps(ref.astype(np.float32), s["bias"], w.k)
    safe_set = kth_gap > 2 * delta
    safe_order = safe_set & (order_gap > 2 * delta)
    same_set = np.all(np.sort(ids, axis=1) == np.sort(ids_x, axis=1), axis=1)
    same = np.all(ids == ids_x, axis=1)
    print(f"{w.name}: chosen set fixed by the exact logits on {safe_set.sum()} of {w.T} tokens "
          f"({same_set.sum()} equal), slot order on {safe_order.sum()} ({same.sum()} equal)")
    assert np.all(same_set[safe_set]) and np.all(same[safe_order])
    # the comparison is not vacuous (the skewed bias's saturated keys leave ~2.5 % in the band)
    assert safe_set.mean() >= 0.9


@pytest.mark.parametrize("name", list(CASES))
def test_router_parity(K, name):
    w = CASES[name]
    s = W.gen_small_inputs(w)
    ids, wts, logits = _run_router(K, w, s)
    check_router(w, s, ids, wts, logits)


def test_router_equal_logits_tie_to_lower_index(K):
    """x = 0: every logit is 0 and, with a flat bias, every key is equal; the
    k lowest expert indices win with equal weights."""
    w = W.WORKLOADS["tiny"].with_(name="router_ties", T=130, H=128, E=64, k=6)
    s = W.gen_small_inputs(w)
    s["x"] = np.zeros_like(s["x"])
    s["bias"] = np.full_like(s["bias"], 0.25)
    ids, wts, logits = _run_router(K, w, s)
    assert np.all(logits == 0)
    assert np.array_equal(ids, np.tile(np.arange(6, dtype=np.int32), (w.T, 1)))
    assert np.allclose(wts, 1.0 / 6)


def test_router_deterministic_and_graph_replay(K):
    w = W.WORKLOADS["skewed"]
    s = W.gen_small_inputs(w)
    x = bf16_to_torch(s["x"], "cuda")
    wg = bf16_to_torch(s["wg"], "cuda")
    bias = torch.from_numpy(s["bias"]).cuda()
    ids0, w0, l0, ws = K.kmoe_router(x, wg, bias, w.k)
    ids1, w1, l1, _ = K.kmoe_router(x, wg, bias, w.k, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(l0, l1) and torch.equal(ids0, ids1) and torch.equal(w0, w1)
    ids2 = torch.empty_like(ids0)
    w2 = torch.empty_like(w0)
    l2 = torch.empty_like(l0)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        K.kmoe_router(x, wg, bias, w.k, logits=l2, topk_ids=ids2, topk_w=w2, workspace=ws, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    l2.zero_()
    ids2.zero_()
    with torch.cuda.graph(g, stream=st):
        K.kmoe_router(x, wg, bias, w.k, logits=l2, topk_ids=ids2, topk_w=w2, workspace=ws, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(l0, l2) and torch.equal(ids0, ids2) and torch.equal(w0, w2)
    assert K.kmoe_device_error(ws)[0] == 0


@pytest.mark.parametrize("name,sample,activation", [("decode", 3, "situ"), ("prefill", 2, "situ"),
                                                    ("decode", 3, "swiglu")])
def test_forward_with_fused_router(K, name, sample, activation):
    """kmoe_forward_router = kmoe_forward on the router's logits, bit for bit;
    sampled tokens against the oracle routed on those logits."""
    w = W.WORKLOADS[name].with_(activation=activation)
    s = W.gen_small_inputs(w)
    wt = device_weights(w)
    p = params(w)
    x = bf16_to_torch(s["x"], "cuda")
    wg = bf16_to_torch(s["wg"], "cuda")
    bias = torch.from_numpy(s["bias"]).cuda()
    out_r, ws = K.kmoe_forward_router(p, x, wg, bias, wt["w13_k"], wt["w2_k"])
    torch.cuda.synchronize()
    assert K.kmoe_device_error(ws)[0] == 0
    logits = K.stage_views(p, ws)["logits"].clone()
    ids = K.stage_views(p, ws)["topk_ids"].cpu().numpy()
    out_l, ws2 = K.kmoe_forward(p, x, logits, bias, wt["w13_k"], wt["w2_k"])
    torch.cuda.synchronize()
    assert K.kmoe_device_error(ws2)[0] == 0
    assert torch.equal(out_r, out_l)
    lg = logits.cpu().numpy()
    ids_k, w_k, _ = O.route(lg, s["bias"], w.k)
    assert np.array_equal(ids, ids_k)
    rng = np.random.default_rng(11)
    tokens = np.sort(rng.choice(w.T, size=sample, replace=False))
    used = sorted(set(int(e) for e in ids_k[tokens].ravel()))
    ref = O.forward(w, s["x"], None, None, W.gen_expert_weights_np(w, used), experts_host=used, tokens=tokens,
                    ids=ids_k, topk_w=w_k)
    assert_output_parity(out_r[torch.from_numpy(tokens).cuda()], ref["out"], f"{name}_{activation}_router")
