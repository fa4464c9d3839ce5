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
