"""Kimi-K3 routed-expert MoE forward, written out step by step (float64).

TEST INFRASTRUCTURE ONLY: imported by tests, by the smoke check and by the
CPU-baseline leg of the benchmark; the product path never uses it.

Steps and the passages they follow
0. router     Kimi-K3 SM120 FlashInfer MXFP4 page, "Phase 1: serving call
              chain": the TopK step consumes the router's logits, i.e. the
              gate's dense product of the bf16 hidden state with the bf16
              gate weight [E, H]; read as the exact dot products rounded
              once to fp32.
1. route      Kimi-K3 SM120 FlashInfer MXFP4 page, "Phase 1: serving call
              chain" and its source table (topk.py row): sigmoid scores, the
              e_score_correction_bias takes part only in choosing experts,
              the final weights are gathered from the un-biased sigmoid
              scores and renormalised.  MoE path analysis page (SM100): the
              routed output is scaled by routed_scaling_factor.
2. quantise   MoE path analysis page, SM100 "mega_moe_pre_dispatch": bf16 ->
              per-32 absmax -> UE8M0 scale -> FP8 E4M3 codes.
3. FC1        SM120 page, "real checkpoint contract": w13 is [E, 2I, H/2]
              packed E2M1 with [E, 2I, H/32] E8M0 scales, gate rows first
              then up rows ([gate; up] halves).  Block-scaled GEMM =
              dequantise both operands, then a dense product.
4. SiTU       SM120 page, "SiTU reference formula":
              gate' = beta*tanh(gate/beta)*sigmoid(gate),
              up'   = beta_lin*tanh(up/beta_lin), out = gate'*up'
              with beta = situ_beta = 4, beta_lin = situ_linear_beta = 25.
   control    the SwiGLU control activation the SM120 page's kernel runs
              (alpha 1.702, beta 1, limit 7), in its clamped form (below).
5. requant    the FC2 input is MXFP8 like the FC1 input (both GEMMs are
              MXFP8 activation x MXFP4 weight, SM120 page, "Goal").
6. FC2        w2 is [E, H, I/2] packed E2M1 with [E, H, I/32] scales.
7. combine    SM120 page, "Phase 2 symmetry constraints": the non-fused
              finalize (a fixed-order weighted sum per token) is the
              deterministic reference; masked slots (expert id -1) add 0.

Readings where the pages leave a step open
- routing key = fp32(sigmoid(logit)) + fp32(bias) as one IEEE fp32 add;
  sigmoid evaluated in double and rounded to fp32; ties between equal keys
  go to the lower expert index; plain top-k over all experts (the pages name
  DeepSeek-V3-style grouped top-k but give no group counts).
- the gated-width rule: FC1 must be exactly twice as wide as FC2's K
  ("256 vs 128" at H = I = 128 is the pages' rejected shape).
- SwiGLU control: the pages give only its parameters; read as the clamped
  form out = g' * sigmoid(alpha*g') * (u' + beta), g' = min(g, limit),
  u' = clamp(u, -limit, limit).
"""
from __future__ import annotations

import numpy as np

from . import formats as F


class ShapeError(ValueError):
    pass


def sigmoid_fp32(logits: np.ndarray) -> np.ndarray:
    """fp32(1 / (1 + exp(-x))) evaluated in double."""
    x = np.asarray(logits, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-x))
    return s.astype(np.float32)


def router_logits(x_bits: np.ndarray, wg_bits: np.ndarray) -> np.ndarray:
    """Router GEMM: logits fp32 [T, E] = fp32(x @ W_g^T) with x bf16 [T, H] and
    W_g bf16 [E, H] given as bit patterns; the dot products are taken in
    double (every bf16 product is exact there) and rounded once to fp32."""
    x = F.bf16_decode(x_bits)
    g = F.bf16_decode(wg_bits)
    if x.shape[-1] != g.shape[-1]:
        raise ShapeError(f"hidden size {x.shape[-1]} != gate weight width {g.shape[-1]}")
    return (x @ g.T).astype(np.float32)


def route(logits: np.ndarray, bias: np.ndarray, k: int):
    """Top-k expert choice per token.

    Returns (ids int32 [T,k] in descending key order, weights float64 [T,k]
    summing to 1 per token, scores fp32 [T,E])."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ShapeError(f"top-k {k} out of range for {E} experts")
    s = sigmoid_fp32(logits)
    key = s + np.asarray(bias, dtype=np.float32)[None, :]      # fp32 add
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.argsort(-key[t], kind="stable")              # equal keys: lower index first
        ids[t] = order[:k]
    sel = np.take_along_axis(s, ids.astype(np.int64), axis=1).astype(np.float64)
    w = sel / sel.sum(axis=1, keepdims=True)
    return ids, w, s


def situ(gate: np.ndarray, up: np.ndarray, beta: float = 4.0, beta_lin: float = 25.0) -> np.ndarray:
    g = np.asarray(gate, dtype=np.float64)
    u = np.asarray(up, dtype=np.float64)
    sig = 1.0 / (1.0 + np.exp(-np.clip(g, -700.0, 700.0)))
    return beta * np.tanh(g / beta) * sig * (beta_lin * np.tanh(u / beta_lin))


def swiglu(gate: np.ndarray, up: np.ndarray, alpha: float = 1.702, beta: float = 1.0,
           limit: float = 7.0) -> np.ndarray:
    """The clamped SwiGLU control activation (SM120 page, activation table:
    alpha = 1.702, beta = 1, limit = 7): g' = min(g, limit),
    u' = clamp(u, -limit, limit), out = g' * sigmoid(alpha * g') * (u' + beta)."""
    g = np.minimum(np.asarray(gate, dtype=np.float64), limit)
    u = np.clip(np.asarray(up, dtype=np.float64), -limit, limit)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-alpha * g)) * (u + beta)


def activation(w, gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """The FC1 activation the workload names (SiTU unless it says "swiglu")."""
    if getattr(w, "activation", "situ") == "swiglu":
        return swiglu(gate, up, w.swiglu_alpha, w.swiglu_beta, w.swiglu_limit)
    return situ(gate, up, w.situ_beta, w.situ_linear_beta)


def check_shapes(H: int, I: int, w13: np.ndarray, w2: np.ndarray):
    """The gated-activation width rule: FC1 rows = 2 * FC2 K."""
    fc1_rows = w13.shape[-2]
    fc2_k = w2.shape[-1] * 2
    if fc1_rows != 2 * fc2_k or fc2_k != I:
        raise ShapeError(
            f"gated FC1 needs {2 * fc2_k} weight rows ([gate; up] halves of FC2's K={fc2_k}), "
            f"got {fc1_rows}")
    if w13.shape[-1] * 2 != H or w2.shape[-2] != H:
        raise ShapeError(f"hidden size mismatch: w13 K={w13.shape[-1] * 2}, w2 rows={w2.shape[-2]}, H={H}")


def expert_fc1(xq_rows: np.ndarray, xs_rows: np.ndarray, w13: np.ndarray, w13_sf: np.ndarray, I: int):
    """gate, up [n, I] float64 for the rows routed to one expert."""
    a = F.dequant_mxfp8(xq_rows, xs_rows)            # [n, H]
    b = F.dequant_mxfp4(w13, w13_sf)                 # [2I, H]
    acc = a @ b.T                                    # [n, 2I]
    return acc[:, :I], acc[:, I:]


def expert_fc2(iq_rows: np.ndarray, is_rows: np.ndarray, w2: np.ndarray, w2_sf: np.ndarray):
    a = F.dequant_mxfp8(iq_rows, is_rows)            # [n, I]
    b = F.dequant_mxfp4(w2, w2_sf)                   # [H, I]
    return a @ b.T                                   # [n, H]


def combine(y: np.ndarray, ids: np.ndarray, w: np.ndarray, rsf: float) -> np.ndarray:
    """out[t] = rsf * sum_j w[t,j] * y[t,j], slots in order, id < 0 skipped."""
    T, k = ids.shape
    out = np.zeros((T, y.shape[-1]), dtype=np.float64)
    for j in range(k):
        m = ids[:, j] >= 0
        out[m] += w[m, j, None] * y[m, j]
    return rsf * out


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), kept as float64."""
    f = np.asarray(a, dtype=np.float64)
    # keep 8 significant bits of the double (bf16 precision), ties to even
    m, e = np.frexp(f)                     # f = m * 2^e, |m| in [0.5, 1)
    r = np.round(np.ldexp(m, 8))           # |r| in [128, 256]; numpy rounds half to even
    return np.ldexp(r, e - 8)


def forward(w, x_bits, logits, bias, wts, experts_host=None, tokens=None,
            ids=None, topk_w=None, want_stages=False):
    """The whole layer for the tokens in `tokens` (all tokens by default).

    w         workload (T, H, I, E, k, situ params, routed_scaling_factor)
    x_bits    bf16 bit patterns [T, H]
    wts       dict of packed weights for the experts in `experts_host`
              (the expert id of row i of each array), or for all experts
    ids/topk_w  optional precomputed routing (ids < 0 are masked slots)
    Returns dict with out (float64 [n,H]), out_bf16, and stage tensors."""
    H, I, k = w.H, w.I, w.k
    check_shapes(H, I, wts["w13"], wts["w2"])
    if ids is None:
        ids, topk_w, _ = route(logits, bias, k)
    tokens = np.arange(w.T) if tokens is None else np.asarray(tokens)
    xq, xs = F.quantize_mx(F.bf16_decode(x_bits[tokens]), "e4m3")
    sub_ids = ids[tokens]
    sub_w = topk_w[tokens]
    n = len(tokens)
    pos = {int(e): i for i, e in enumerate(experts_host)} if experts_host is not None else None
    y = np.zeros((n, k, H), dtype=np.float64)
    iq = np.zeros((n, k, I), dtype=np.uint8)
    isf = np.zeros((n, k, I // 32), dtype=np.uint8)
    for e in np.unique(sub_ids[sub_ids >= 0]):
        ti, tj = np.nonzero(sub_ids == e)
        we = pos[int(e)] if pos is not None else int(e)
        gate, up = expert_fc1(xq[ti], xs[ti], wts["w13"][we], wts["w13_sf"][we], I)
        act = activation(w, gate, up)
        q, s = F.quantize_mx(act, "e4m3")
        iq[ti, tj] = q
        isf[ti, tj] = s
        y[ti, tj] = expert_fc2(q, s, wts["w2"][we], wts["w2_sf"][we])
    out = combine(y, sub_ids, sub_w, w.routed_scaling_factor)
    res = {"out": out, "out_bf16": bf16_round(out), "ids": ids, "topk_w": topk_w}
    if want_stages:
        res.update({"xq": xq, "xs": xs, "inter_q": iq, "inter_s": isf, "y": y})
    return res
