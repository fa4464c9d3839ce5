"""Shared set-up for the GPU parity tests: seeded inputs on the device and
oracle references on the host for a token sample.  Inputs come only from the
`workloads` generator; expected values only from `oracle`."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O

_WEIGHT_CACHE = {}


def bf16_to_torch(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def device_weights(w: W.Workload, device="cuda"):
    import mxfp8_mxfp4_moe_gb300 as K
    key = (w.E, w.H, w.I, w.sf_lo, w.sf_hi)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        torch.cuda.empty_cache()
        wts = W.gen_expert_weights_torch(w, device)
        p = params(w)
        w13_k, w2_k = K.kmoe_prepare_weights(p, wts["w13"], wts["w13_sf"], wts["w2"], wts["w2_sf"])
        del wts
        torch.cuda.empty_cache()
        _WEIGHT_CACHE[key] = {"w13_k": w13_k, "w2_k": w2_k}
    return _WEIGHT_CACHE[key]


def params(w: W.Workload, **kw):
    import mxfp8_mxfp4_moe_gb300 as K
    d = dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, situ_beta=w.situ_beta, situ_linear_beta=w.situ_linear_beta,
             routed_scaling_factor=w.routed_scaling_factor, activation=w.activation,
             swiglu_alpha=w.swiglu_alpha, swiglu_beta=w.swiglu_beta, swiglu_limit=w.swiglu_limit)
    d.update(kw)
    return K.make_params(**d)


def device_inputs(w: W.Workload, small=None, device="cuda"):
    s = small if small is not None else W.gen_small_inputs(w)
    return {
        "x": bf16_to_torch(s["x"], device),
        "logits": torch.from_numpy(s["logits"]).to(device),
        "bias": torch.from_numpy(s["bias"]).to(device),
    }, s


def run_forward(w, small=None, topk_ids=None, topk_w=None, device="cuda"):
    import mxfp8_mxfp4_moe_gb300 as K
    wt = device_weights(w, device)
    inp, s = device_inputs(w, small, device)
    p = params(w)
    out, ws = K.kmoe_forward(p, inp["x"], inp["logits"], inp["bias"], wt["w13_k"], wt["w2_k"], topk_ids=topk_ids,
                             topk_w=topk_w)
    torch.cuda.synchronize()
    st, word = K.kmoe_device_error(ws)
    assert st == 0, f"device error word {word:#x}"
    return out, ws, p, s, inp


def oracle_forward(w, s, tokens, ids=None, topk_w=None):
    """Oracle output for `tokens`, with the weights of exactly the experts they use."""
    if ids is None:
        ids, topk_w, _ = O.route(s["logits"], s["bias"], w.k)
    used = sorted(set(int(e) for e in ids[tokens].ravel() if e >= 0))
    wts = W.gen_expert_weights_np(w, used)
    return O.forward(w, s["x"], s["logits"], s["bias"], wts, experts_host=used, tokens=tokens, ids=ids,
                     topk_w=topk_w, want_stages=True)


def _oracle_slots_worker(args):
    """One worker of oracle_forward_pool: the oracle's forward of `tokens`
    with every slot whose expert is not in `experts` masked (-1), so the
    stage tensors of the slots it owns come out exactly as in one whole call."""
    w, x_bits, ids, topk_w, experts = args
    wts = W.gen_expert_weights_np(w, experts)
    own = np.isin(ids, experts)
    masked = np.where(own, ids, -1).astype(np.int32)
    n = len(ids)
    r = O.forward(w.with_(T=n), x_bits, None, None, wts, experts_host=list(experts), tokens=np.arange(n),
                  ids=masked, topk_w=topk_w, want_stages=True)
    return own, r["inter_q"], r["inter_s"], r["y"]


def oracle_forward_pool(w, s, tokens, ids=None, topk_w=None, workers=None):
    """oracle_forward for many tokens of a full-size layer, with the experts
    spread over worker processes (started with spawn, so they hold no CUDA
    state).  Every (token, slot) is computed by one oracle call that owns its
    expert; the per-slot y are then summed by the oracle's own combine."""
    import multiprocessing as mp
    import os
    if ids is None:
        ids, topk_w, _ = O.route(s["logits"], s["bias"], w.k)
    tokens = np.asarray(tokens)
    sub_ids, sub_w = ids[tokens], topk_w[tokens]
    used = sorted(set(int(e) for e in sub_ids.ravel() if e >= 0))
    n_workers = workers or max(1, min(8, (os.cpu_count() or 2) // 2, len(used)))
    chunks = [used[i::n_workers] for i in range(n_workers)]
    x_bits = s["x"][tokens]
    jobs = [(w, x_bits, sub_ids, sub_w, c) for c in chunks if c]
    old = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in old:
        os.environ[v] = "2"
    try:
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            parts = pool.map(_oracle_slots_worker, jobs)
    finally:
        for v, val in old.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val
    n, k = sub_ids.shape
    iq = np.zeros((n, k, w.I), np.uint8)
    isf = np.zeros((n, k, w.I // 32), np.uint8)
    y = np.zeros((n, k, w.H), np.float64)
    for own, q, sf, yy in parts:
        iq[own], isf[own], y[own] = q[own], sf[own], yy[own]
    out = O.combine(y, sub_ids, sub_w, w.routed_scaling_factor)
    return {"out": out, "inter_q": iq, "inter_s": isf, "y": y, "ids": ids, "topk_w": topk_w}


def tile_position_tokens(ids: np.ndarray, E: int, BN: int, n: int = 32, seed: int = 0, big_rows: int = 0,
                         BN_big: int = 0):
    """Tokens chosen by where their rows land in the expert-sorted token
    tiles (rows of an expert in slot order, as the permutation lays them
    out; tiles of BN rows, or of BN_big rows for experts with more than
    big_rows rows when BN_big > 0): for the three most- and three
    least-loaded experts and the last expert with rows (whose work items are
    claimed last), the first row, the rows on both sides of the first tile
    boundary, a middle row and the last row (the partial tile); then random
    tokens up to n."""
    T, k = ids.shape
    flat = ids.ravel()
    valid = flat >= 0
    counts = np.bincount(flat[valid], minlength=E)
    order = np.flatnonzero(valid)[np.argsort(flat[valid], kind="stable")]
    starts = np.concatenate([[0], np.cumsum(counts)])
    nz = np.flatnonzero(counts)
    by_load = nz[np.argsort(-counts[nz], kind="stable")]
    chosen = list(dict.fromkeys(list(by_load[:3]) + list(by_load[-3:]) + [nz[-1]]))
    toks = set()
    for e in chosen:
        c = int(counts[e])
        bn = BN_big if (BN_big > 0 and c > big_rows) else BN
        nt = (c + bn - 1) // bn
        mid = (nt // 2) * bn + (min(bn, c - (nt // 2) * bn) // 2)
        rows = {0, mid, c - 1} | ({bn - 1, bn} if nt > 1 else set())
        for r in rows:
            toks.add(int(order[starts[e] + r] // k))
    rng = np.random.default_rng(seed)
    while len(toks) < min(n, T):
        toks.add(int(rng.integers(T)))
    return np.array(sorted(toks)), [int(e) for e in chosen]


def output_errors(gpu_bf16: torch.Tensor, ref: np.ndarray):
    g = gpu_bf16.float().cpu().numpy().astype(np.float64)
    diff = g - ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(diff).max() / max(np.abs(ref).max(), 1e-300)
    return rel, mx


def assert_output_parity(gpu_bf16, ref, tag=""):
    rel, mx = output_errors(gpu_bf16, ref)
    floor = np.linalg.norm(O.bf16_round(ref) - ref) / max(np.linalg.norm(ref), 1e-300)
    print(f"{tag} rel_fro={rel:.3e} (bf16 floor {floor:.3e}) max_abs/max|ref|={mx:.3e}")
    assert np.all(np.isfinite(gpu_bf16.float().cpu().numpy()))
    assert rel <= 2e-3, f"{tag} relative Frobenius error {rel:.3e} > 2e-3"
    assert mx <= 1e-2, f"{tag} max abs error {mx:.3e} x max|ref| > 1e-2"


def tile_sf_offsets(tile, local, g, BN, KB):
    """Byte offsets in a token-tile scale array (layout plumbing; kmoe_tile_sf_offset)."""
    nch = (BN + 127) // 128
    kb = g // 4
    chunk = local // 128
    r = local % 128
    return ((tile * KB + kb) * nch + chunk) * 512 + (r % 32) * 16 + (r // 32) * 4 + (g % 4)


def gather_row_scales(views_np, which: str, rows: np.ndarray, K: int):
    """Scales [len(rows), K/32] of expert-sorted rows from the token-tile
    scale arrays of stage `which` ("x": xsf / xsf_big, "i": isf / isf_big).
    An expert with more than big_rows rows has its rows in the big tiles
    (tile_start_big), the others in the small tiles (tile_start)."""
    L = views_np["layout"]
    seg = views_np["seg_start"]
    counts = views_np["counts"]
    # searchsorted(side=right) - 1 gives the last expert starting <= row: the
    # non-empty one containing it when empty experts share its start
    e = np.searchsorted(seg, rows, side="right") - 1
    local = rows - seg[e]
    big = (counts[e] > L.big_rows) if L.tile_rows_big > 0 else np.zeros(len(rows), bool)
    g = np.arange(K // 32)
    out = np.zeros((len(rows), K // 32), np.uint8)
    for is_big, bn, ts, sf in ((False, L.tile_rows, views_np["tile_start"], views_np[which + "sf"]),
                               (True, L.tile_rows_big, views_np["tile_start_big"], views_np[which + "sf_big"])):
        m = big == is_big
        if not m.any():
            continue
        tile = ts[e[m]] + local[m] // bn
        lr = local[m] % bn
        off = tile_sf_offsets(tile[:, None], lr[:, None], g[None, :], bn, K // 128)
        out[m] = sf[off]
    return out


def stage_numpy(p, ws):
    import mxfp8_mxfp4_moe_gb300 as K
    v = K.stage_views(p, ws)
    out = {k: (t.cpu().numpy() if isinstance(t, torch.Tensor) else t) for k, t in v.items()}
    return out
