"""Pins of the oracle's routing: brute force over all expert subsets, the
renormalisation invariant, bias-only-for-selection, ties and special cases."""
import itertools

import numpy as np

from oracle import moe


def _keys(logits, bias):
    s = moe.sigmoid_fp32(logits)
    return s, s + bias.astype(np.float32)


def test_brute_force_all_subsets_e8_k2():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((64, 8)).astype(np.float32)
    bias = (rng.standard_normal(8) * 0.1).astype(np.float32)
    ids, w, s = moe.route(logits, bias, 2)
    _, key = _keys(logits, bias)
    for t in range(64):
        winners = []
        for sub in itertools.combinations(range(8), 2):
            inside = [key[t, e] for e in sub]
            outside = [key[t, e] for e in range(8) if e not in sub]
            if min(inside) > max(outside):
                winners.append(set(sub))
        assert len(winners) == 1
        assert set(ids[t].tolist()) == winners[0]
        # slots in descending key order
        assert key[t, ids[t, 0]] >= key[t, ids[t, 1]]
        # weights from the UNBIASED scores, renormalised
        sel = s[t, ids[t]].astype(np.float64)
        assert np.allclose(w[t], sel / sel.sum(), rtol=0, atol=1e-15)


def test_weights_sum_to_one_and_bias_shift():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((200, 64)).astype(np.float32)
    bias = (rng.standard_normal(64) * 0.1).astype(np.float32)
    ids, w, _ = moe.route(logits, bias, 16)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    ids2, w2, _ = moe.route(logits, bias + np.float32(0.25), 16)
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=0, atol=0)


def test_zero_bias_is_plain_sigmoid_topk():
    rng = np.random.default_rng(2)
    # well separated logits: the sigmoid keeps their order in fp32
    logits = np.stack([rng.permutation(32).astype(np.float32) * 0.05 - 0.8 for _ in range(50)])
    ids, _, _ = moe.route(logits, np.zeros(32, np.float32), 4)
    ref = np.argsort(-logits, axis=1)[:, :4]
    assert np.array_equal(ids, ref)


def test_k_equals_e_and_ties_to_lower_index():
    logits = np.zeros((3, 6), np.float32)
    logits[1, [1, 4]] = 1.0
    bias = np.zeros(6, np.float32)
    ids, w, _ = moe.route(logits, bias, 6)
    assert sorted(ids[0].tolist()) == list(range(6))
    assert ids[0].tolist() == [0, 1, 2, 3, 4, 5]          # all equal: index order
    assert ids[1].tolist()[:2] == [1, 4]
    assert np.allclose(w[0], 1 / 6)
    ids, _, _ = moe.route(logits, bias, 2)
    assert ids[2].tolist() == [0, 1]


# ---------------------------------------------------------------- the sigmoid's value
# The routing key adds fp32(sigmoid(logit)) to the bias, and routing is
# compared bit-exactly, so the oracle's sigmoid must be the exact sigmoid of
# the fp32 logit rounded ONCE to fp32.  These pins fail for sigmoid evaluated
# in fp32, for a rounding step in between (e.g. exp rounded to fp32 first),
# and for a wrong sign inside the exponential.

def _correctly_rounded_fp32(v):
    """The fp32 value nearest to the mpmath number v (ties to the even code)."""
    import mpmath
    c = np.float32(float(v))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    dist = [abs(mpmath.mpf(float(x)) - v) for x in cands]
    best = min(dist)
    tied = [x for x, d in zip(cands, dist) if d == best]
    if len(tied) > 1:
        tied = [x for x in tied if (np.array(x, np.float32).view(np.uint32) & 1) == 0]
    return tied[0]


def test_sigmoid_closed_forms():
    # sigma(0) = 1/2; sigma(+-ln 3) = 3/4, 1/4: fp32(ln 3) moves the exact
    # value by at most 3/16 * 2^-24, less than half an fp32 ulp of either
    x = np.array([0.0, np.log(3.0), -np.log(3.0)], dtype=np.float32)
    assert moe.sigmoid_fp32(x).tolist() == [0.5, 0.75, 0.25]
    # symmetry sigma(-x) = 1 - sigma(x) is exact in fp32 for these: 1 - 3/4, 1 - 1/2
    # the tails: sigma(x) -> 1 above ~17 (fp32), -> e^x below ~-17; sigma(-88)
    # is an fp32 subnormal (~6.05e-39), sigma(-103) ~ 1.86e-45 rounds to the
    # smallest one (2^-149 ~ 1.40e-45), sigma(-120) to zero
    t = moe.sigmoid_fp32(np.array([20.0, 88.0, -20.0, -88.0, -103.0, -120.0], dtype=np.float32))
    assert t[0] == 1.0 and t[1] == 1.0
    assert t[2] == np.float32(np.exp(-20.0) / (1 + np.exp(-20.0)))
    assert 0 < t[3] < np.finfo(np.float32).tiny and abs(float(t[3]) / np.exp(-88.0) - 1) < 2e-3
    assert t[4] == np.float32(2.0 ** -149) and t[5] == 0.0


def test_sigmoid_correctly_rounded_against_mpmath():
    mpmath = __import__("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * 3.0, rng.uniform(-110, 30, 2000),
                        np.array([-17.0, 17.0, 16.635532, -16.635532, 1e-7, -1e-7])]).astype(np.float32)
    got = moe.sigmoid_fp32(x)
    for xi, gi in zip(x, got):
        v = 1 / (1 + mpmath.exp(-mpmath.mpf(float(xi))))
        assert gi == _correctly_rounded_fp32(v), (float(xi), float(gi))


def test_sigmoid_agrees_with_torch_float64_rounded_once():
    torch = __import__("torch")
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(100000) * 2.0, rng.uniform(-100, 100, 20000),
                        np.array([-20, 20, -88, 88], np.float64)]).astype(np.float32)
    ref = torch.sigmoid(torch.from_numpy(x.astype(np.float64))).to(torch.float32).numpy()
    got = moe.sigmoid_fp32(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
