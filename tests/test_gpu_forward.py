"""GPU parity of the whole forward (kmoe_forward through the C ABI) against
the float64 oracle: stage tensors (routing, MXFP8 codes and scales, expert
permutation) bit-exact, intermediate codes by agreement rate, outputs within
rel. Frobenius 2e-3 and max-abs 1e-2 x max|ref|.  Full-size workloads are
checked on sampled tokens (all their routing/quantisation on every token);
plus determinism, CUDA-graph replay, masked slots and edge cases."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O
from tests._moe_setup import (assert_output_parity, device_inputs, device_weights, gather_row_scales,
                              oracle_forward, oracle_forward_pool, params, run_forward, stage_numpy,
                              tile_position_tokens)

pytestmark = pytest.mark.gpu

TINY_UNSAT = W.WORKLOADS["tiny"].with_(name="tiny_unsaturated", sf_lo=117, sf_hi=121)
# 224-row token tiles (the CTA-pair GEMMs) at sizes the oracle checks on every
# token: 256 rows per expert on average, several work items per CTA pair,
# full and partial tiles; the skewed bias gives experts of 1 to ~1000 rows.
PAIR_EVEN = W.WORKLOADS["tiny"].with_(name="pair_tiles", T=4096, H=512, I=512, E=32, k=2)
PAIR_SKEW = PAIR_EVEN.with_(name="pair_tiles_skewed", skewed=True)
# SiTU with other beta values (the kernels specialise beta = 4)
TINY_BETA = TINY_UNSAT.with_(name="tiny_beta2_10", situ_beta=2.0, situ_linear_beta=10.0)
PAIR_BETA = PAIR_EVEN.with_(name="pair_tiles_beta3_20", situ_beta=3.0, situ_linear_beta=20.0, sf_lo=117, sf_hi=121)

# the clamped SwiGLU control in place of SiTU: with the default weight scales
# about half the gate/up values pass the clamp (|v| > 7), with the narrow ones
# none do; the pair case mixes both; one case with other parameters
TINY_SWIGLU = W.WORKLOADS["tiny"].with_(name="tiny_swiglu", activation="swiglu")
TINY_SWIGLU_UNSAT = TINY_UNSAT.with_(name="tiny_swiglu_unclamped", activation="swiglu")
TINY_SWIGLU_P = TINY_SWIGLU.with_(name="tiny_swiglu_a1_b05_l3", swiglu_alpha=1.0, swiglu_beta=0.5, swiglu_limit=3.0)
PAIR_SWIGLU = PAIR_EVEN.with_(name="pair_tiles_swiglu", activation="swiglu", sf_lo=119, sf_hi=124)


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


def _check_stages(w, p, ws, s, ref, tokens):
    st = stage_numpy(p, ws)
    ids_ref, w_ref, _ = O.route(s["logits"], s["bias"], w.k)
    assert np.array_equal(st["topk_ids"], ids_ref)
    assert np.allclose(st["topk_w"], w_ref, rtol=1e-6)
    # permutation: each slot owns exactly one row, rows of an expert are contiguous and token-ordered
    ros = st["row_of_slot"]
    R = w.T * w.k
    assert sorted(ros.tolist()) == list(range(R))
    assert np.array_equal(st["slot_of_row"][ros], np.arange(R))
    exp_of_row = np.empty(R, np.int64)
    exp_of_row[ros] = ids_ref.ravel()
    assert np.all(np.diff(exp_of_row) >= 0)
    counts = np.bincount(ids_ref.ravel(), minlength=w.E)
    assert np.array_equal(st["counts"], counts)
    # MXFP8 codes and scales of x, bit-exact on every token (tile layout for the scales)
    xq_ref, xs_ref = F.quantize_mx(W.bf16_bits_to_f64(s["x"]), "e4m3")
    slots = np.arange(R)
    rows = ros[slots]
    assert np.array_equal(st["xq"][rows], xq_ref[slots // w.k])
    got_sf = gather_row_scales(st, "x", rows, w.H)
    assert np.array_equal(got_sf, xs_ref[slots // w.k])
    # intermediate codes of the sampled tokens (masked slots excluded)
    tsl = np.array([t * w.k + j for t in tokens for j in range(w.k)])
    tsl = tsl[ids_ref.ravel()[tsl] >= 0]
    iq_gpu = st["iq"][ros[tsl]]
    iq_ref = ref["inter_q"].reshape(-1, w.I)[ids_ref[tokens].ravel() >= 0]
    isf_gpu = gather_row_scales(st, "i", ros[tsl], w.I)
    isf_ref = ref["inter_s"].reshape(-1, w.I // 32)[ids_ref[tokens].ravel() >= 0]
    check_intermediate_agreement(w.name, iq_gpu, iq_ref, isf_gpu, isf_ref)
    return st


def _e4m3_ordinal(c):
    """Position of E4M3 codes on the number line (+0 and -0 both 0; codes
    are monotonic in magnitude within a sign)."""
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def check_intermediate_agreement(name, iq_gpu, iq_ref, isf_gpu, isf_ref):
    """The GPU evaluates the activation in fp32, the oracle in double, so an
    activation within rounding of an E4M3 midpoint (or a group maximum within
    rounding of a power-of-two boundary) can quantise one step apart.  Bar:
    at least 99.99 % of scales and of codes agree (at most one disagreement
    in samples of fewer than 10^4), every differing scale is one step apart,
    and every differing code (in groups whose scales agree) is one E4M3 step
    apart.  No NaN code and no 0xFF scale anywhere."""
    assert not np.any((iq_gpu & 0x7F) == 0x7F), "NaN intermediate code"
    assert not np.any(isf_gpu == 0xFF), "0xFF intermediate scale"
    sf_bad = isf_gpu != isf_ref
    n_sf = sf_bad.size
    assert sf_bad.sum() <= max(1, int(1e-4 * n_sf)), f"{name}: {sf_bad.sum()} of {n_sf} scales differ"
    assert np.all(np.abs(isf_gpu[sf_bad].astype(int) - isf_ref[sf_bad].astype(int)) == 1)
    group_ok = np.repeat(~sf_bad, 32, axis=1)
    d = np.abs(_e4m3_ordinal(iq_gpu) - _e4m3_ordinal(iq_ref))[group_ok]
    n = d.size
    flips = int((d != 0).sum())
    rate = 1.0 - flips / max(n, 1)
    print(f"{name}: intermediate code agreement {rate:.7f} ({flips} of {n} differ), "
          f"scale agreement {1.0 - sf_bad.mean():.7f}")
    assert flips <= max(1, int(1e-4 * n)), f"{name}: {flips} of {n} intermediate codes differ"
    assert np.all(d <= 1), f"{name}: intermediate codes differ by more than one E4M3 step"


@pytest.mark.parametrize("wl", [W.WORKLOADS["tiny"], TINY_UNSAT, TINY_BETA, TINY_SWIGLU, TINY_SWIGLU_UNSAT, TINY_SWIGLU_P],
                         ids=["tiny", "tiny_unsaturated", "beta2", "swiglu", "swiglu_unclamped", "swiglu_params"])
def test_forward_tiny_full(K, wl):
    out, ws, p, s, _ = run_forward(wl)
    tokens = np.arange(wl.T)
    ref = oracle_forward(wl, s, tokens)
    _check_stages(wl, p, ws, s, ref, tokens)
    assert_output_parity(out, ref["out"], wl.name)


@pytest.mark.parametrize("wl", [PAIR_EVEN, PAIR_SKEW, PAIR_BETA, PAIR_SWIGLU], ids=["even", "skewed", "beta3", "swiglu"])
def test_forward_pair_tiles_every_token(K, wl):
    out, ws, p, s, _ = run_forward(wl)
    L = K.kmoe_workspace_layout(p)
    assert L.tile_rows_big == 224
    tokens = np.arange(wl.T)
    ref = oracle_forward(wl, s, tokens)
    st = _check_stages(wl, p, ws, s, ref, tokens)
    counts = st["counts"]
    big = counts > L.big_rows
    # multi-tile experts and partial tiles in the 224-row (CTA-pair) class
    assert counts.max() > 224 and (counts[big] % 224 != 0).any()
    assert_output_parity(out, ref["out"], wl.name)


@pytest.mark.parametrize("name", ["reduced", "decode", "prefill", "skewed"])
def test_forward_full_size_tile_positions(K, name):
    """Full-size layers, outputs and intermediate codes checked on at least
    32 tokens (all 16 at decode) chosen by tile position: the first row, both
    sides of the first tile boundary, a middle row and the last (partial-tile)
    row of the three most- and three least-loaded experts and of the last
    expert with rows (its work items are claimed last), plus random tokens.
    Routing, x codes/scales and the permutation are checked on every token."""
    w = W.WORKLOADS[name]
    out, ws, p, s, _ = run_forward(w)
    ids, tw, _ = O.route(s["logits"], s["bias"], w.k)
    L = K.kmoe_workspace_layout(p)
    tokens, experts = tile_position_tokens(ids, w.E, L.tile_rows, n=32, seed=123, big_rows=L.big_rows,
                                           BN_big=L.tile_rows_big)
    counts = np.bincount(ids.ravel(), minlength=w.E)
    print(f"{name}: {len(tokens)} tokens, tile rows {L.tile_rows} / {L.tile_rows_big} (experts with more than "
          f"{L.big_rows} rows), experts {experts} with rows {counts[experts].tolist()}")
    assert len(tokens) >= min(32, w.T)
    ref = oracle_forward_pool(w, s, tokens, ids, tw)
    _check_stages(w, p, ws, s, ref, tokens)
    assert_output_parity(out[torch.from_numpy(tokens).cuda()], ref["out"], name)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name,sample", [("real_decode", 3), ("real_prefill", 2)])
def test_forward_real_checkpoint_shape_sampled(K, name, sample):
    """The real checkpoint's expert shape (3584-wide latent, I = 3072)."""
    w = W.NEXT_WORKLOADS[name]
    out, ws, p, s, _ = run_forward(w)
    rng = np.random.default_rng(321)
    tokens = np.sort(rng.choice(w.T, size=sample, replace=False))
    ref = oracle_forward(w, s, tokens)
    _check_stages(w, p, ws, s, ref, tokens)
    assert_output_parity(out[torch.from_numpy(tokens).cuda()], ref["out"], name)


@pytest.mark.parametrize("name,sample", [("decode", 3), ("prefill", 2)])
def test_forward_swiglu_control_full_size_sampled(K, name, sample):
    """The SwiGLU control activation at the full layer sizes."""
    w = W.WORKLOADS[name].with_(name=name + "_swiglu", activation="swiglu")
    out, ws, p, s, _ = run_forward(w)
    assert p.flags == K.KMOE_FLAG_SWIGLU
    rng = np.random.default_rng(77)
    tokens = np.sort(rng.choice(w.T, size=sample, replace=False))
    ref = oracle_forward(w, s, tokens)
    _check_stages(w, p, ws, s, ref, tokens)
    assert_output_parity(out[torch.from_numpy(tokens).cuda()], ref["out"], w.name)


def test_forward_expert_parallel_local_slice(K):
    """One rank's slice of an expert-parallel layer: routing over all 896
    experts, this layer holds 28 of them (global 140..167); slots routed
    elsewhere are masked (-1) and contribute nothing."""
    g = W.NEXT_WORKLOADS["real_prefill"].with_(T=2048)
    s = W.gen_small_inputs(g)
    ids_g, wts, _ = O.route(s["logits"], s["bias"], g.k)
    e_loc, off = 28, 140
    ids = np.where((ids_g >= off) & (ids_g < off + e_loc), ids_g - off, -1).astype(np.int32)
    wl = g.with_(name="ep_local", E=e_loc)
    out, ws, p, _, _ = run_forward(wl, small=s, topk_ids=torch.from_numpy(ids).cuda(),
                                   topk_w=torch.from_numpy(wts.astype(np.float32)).cuda())
    assert K.kmoe_workspace_layout(p).tile_rows_big == 224
    o = out.float().cpu().numpy()
    none_local = np.all(ids < 0, axis=1)
    assert none_local.any() and np.all(o[none_local] == 0.0)
    rng = np.random.default_rng(99)
    local_tokens = np.flatnonzero(~none_local)
    tokens = np.sort(rng.choice(local_tokens, size=4, replace=False))
    used = sorted(set(int(e) for e in ids[tokens].ravel() if e >= 0))
    ref = O.forward(wl, s["x"], None, None, W.gen_expert_weights_np(wl, used), experts_host=used, tokens=tokens,
                    ids=ids, topk_w=wts.astype(np.float32).astype(np.float64))
    assert_output_parity(out[torch.from_numpy(tokens).cuda()], ref["out"], "ep_local")


@pytest.mark.parametrize("name", ["tiny", "reduced", "pair_tiles", "prefill"])
def test_determinism_and_graph_replay(K, name):
    """Three eager runs bitwise equal; a run with stage events (its kernels
    launched unchained) and a CUDA graph captured once and replayed twice
    bitwise equal to them.  pair_tiles and prefill run the CTA-pair GEMMs,
    whose FC1 work items are claimed dynamically (the order differs from run
    to run, the result may not)."""
    for w in [{"pair_tiles": PAIR_EVEN}.get(name) or W.WORKLOADS[name]]:
        wt = device_weights(w)
        inp, s = device_inputs(w)
        p = params(w)
        if name in ("pair_tiles", "prefill"):
            assert K.kmoe_workspace_layout(p).tile_rows_big == 224
        ws = torch.empty(K.kmoe_workspace_size(p), dtype=torch.uint8, device="cuda")
        outs = []
        for _ in range(3):
            o = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
            K.kmoe_forward(p, inp["x"], inp["logits"], inp["bias"], wt["w13_k"], wt["w2_k"], out=o, workspace=ws)
            outs.append(o)
        torch.cuda.synchronize()
        for o in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
        # stage events between the kernels: the forward launches them unchained
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
        for e in ev:
            e.record()  # creates the event
        o_ev = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
        K.kmoe_forward(p, inp["x"], inp["logits"], inp["bias"], wt["w13_k"], wt["w2_k"], out=o_ev, workspace=ws,
                       stage_events=ev)
        torch.cuda.synchronize()
        assert torch.equal(o_ev.view(torch.int16), outs[0].view(torch.int16))
        # CUDA graph: capture once, replay twice, bitwise equal to eager
        g_out = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                K.kmoe_forward(p, inp["x"], inp["logits"], inp["bias"], wt["w13_k"], wt["w2_k"], out=g_out,
                               workspace=ws, stream=stream)
        for _ in range(2):
            g_out.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(g_out.view(torch.int16), outs[0].view(torch.int16))
        st, word = K.kmoe_device_error(ws)
        assert st == 0


def test_given_routing_masked_slots_and_hot_expert(K):
    w = W.WORKLOADS["tiny"].with_(T=37)     # ragged: 37 tokens
    s = W.gen_small_inputs(w)
    ids, wts, _ = O.route(s["logits"], s["bias"], w.k)
    ids = ids.copy()
    ids[::3, 1] = -1                          # masked slots
    ids[5:30, 0] = 6                          # one hot expert: > 32 rows (several token tiles)
    wts = wts.astype(np.float32)
    out, ws, p, _, _ = run_forward(w, small=s, topk_ids=torch.from_numpy(ids).cuda(),
                                   topk_w=torch.from_numpy(wts).cuda())
    ref = O.forward(w, s["x"], s["logits"], s["bias"], W.gen_expert_weights_np(w, range(w.E)), ids=ids,
                    topk_w=wts.astype(np.float64))
    assert_output_parity(out, ref["out"], "masked")


def test_single_token_and_out_of_range_id(K):
    w = W.WORKLOADS["tiny"].with_(T=1)
    out, ws, p, s, _ = run_forward(w)
    ref = oracle_forward(w, s, np.arange(1))
    assert_output_parity(out, ref["out"], "T=1")
    # an expert id >= E is reported as a device error and treated as masked
    ids = torch.tensor([[1, 99]], dtype=torch.int32, device="cuda")
    wts = torch.tensor([[0.5, 0.5]], dtype=torch.float32, device="cuda")
    wt = device_weights(w)
    inp, _ = device_inputs(w, s)
    o, ws = K.kmoe_forward(p, inp["x"], None, None, wt["w13_k"], wt["w2_k"],
                           topk_ids=ids, topk_w=wts)
    st, word = K.kmoe_device_error(ws)
    assert st == 8 and (word & 2)
    assert torch.isfinite(o.float()).all()
