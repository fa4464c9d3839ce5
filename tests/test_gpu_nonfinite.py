"""Non-finite and extreme tokens through the whole forward (kmoe_forward),
following the SM120 FlashInfer MXFP4 page's NaN/Inf decision record: the
quantised E4M3 payload is finite, no UE8M0 scale is 0xFF, the output is
finite and bitwise identical over three runs; rows whose dequantised values
overflow (Inf, the bf16 maximum) are diagnostics there and are not compared
numerically, every other row is compared with the oracle as usual.

Rows planted in the seeded batch: NaN elements, +Inf, -Inf, +Inf / -Inf /
NaN in different groups, all +0, all -0, one group at the bf16 maximum,
large finite values (1e30, no fp32 overflow in the GEMMs), bf16 subnormals.
Run at a 224-row-tile shape (the CTA-pair GEMMs) and at the decode layer."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import formats as F
from oracle import moe as O
from tests._moe_setup import assert_output_parity, oracle_forward_pool, run_forward, stage_numpy
from tests.test_gpu_forward import PAIR_EVEN, _check_stages

pytestmark = pytest.mark.gpu

NAN, PINF, NINF, BF16_MAX = 0x7FC0, 0x7F80, 0xFF80, 0x7F7F


def _plant(x: np.ndarray, rows):
    """x: bf16 bits [T, H] (uint16), modified in place; returns
    (overflow rows, numerically checked special rows)."""
    H = x.shape[1]
    r = iter(rows)
    rn = next(r); x[rn, 3] = NAN; x[rn, 40] = NAN | 0x8000; x[rn, 64:96] = NAN   # NaN elements, a NaN group
    rp = next(r); x[rp, 5] = PINF
    rm = next(r); x[rm, 70] = NINF
    rx = next(r); x[rx, 1] = PINF; x[rx, 33] = NINF; x[rx, 97] = NAN           # mixed, different groups
    rz = next(r); x[rz, :] = 0
    rnz = next(r); x[rnz, :] = 0x8000
    rmax = next(r); x[rmax, 32:64] = BF16_MAX; x[rmax, 40] = BF16_MAX | 0x8000  # a group at the bf16 maximum
    rbig = next(r)
    big = np.float32(1e30) * (np.arange(H, dtype=np.float32) % 7 - 3)
    x[rbig, :] = W.f32_to_bf16_bits(big)
    rsub = next(r); x[rsub, :] = (np.arange(H) % 127 + 1).astype(np.uint16) | ((np.arange(H) % 2) << 15).astype(np.uint16)
    return [rp, rm, rx, rmax], [rn, rz, rnz, rbig, rsub]


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


@pytest.mark.parametrize("name", ["pair_tiles", "decode"])
def test_forward_nonfinite_and_extreme_tokens(K, name):
    w = PAIR_EVEN if name == "pair_tiles" else W.WORKLOADS[name]
    s = dict(W.gen_small_inputs(w))
    x = s["x"].astype(np.uint16).copy()
    rows = [0, 1, 2, w.T // 2, w.T // 2 + 1, w.T - 5, w.T - 4, w.T - 3, w.T - 1] if w.T >= 32 else list(range(9))
    overflow, special = _plant(x, rows)
    s["x"] = x
    outs = []
    for _ in range(3):
        out, ws, p, _, _ = run_forward(w, small=s)
        outs.append(out)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16)), "not bitwise deterministic"
    assert torch.isfinite(outs[0].float()).all(), "non-finite output"
    if name == "pair_tiles":
        assert K.kmoe_workspace_layout(p).tile_rows_big == 224

    st = stage_numpy(p, ws)
    # every row: payload finite, no 0xFF scale (x and intermediate)
    assert not np.any((st["xq"] & 0x7F) == 0x7F)
    assert not np.any((st["iq"][: w.T * w.k] & 0x7F) == 0x7F)
    R = w.T * w.k
    xq_ref, xs_ref = F.quantize_mx(F.bf16_decode(x), "e4m3")
    assert not np.any(xs_ref == 0xFF)
    # the Inf rows saturate: their scale byte is 0xFE and the Inf element 448
    assert xs_ref[overflow[0], 0] == 0xFE and xq_ref[overflow[0], 5] == 0x7E
    assert xs_ref[overflow[1], 2] == 0xFE and xq_ref[overflow[1], 70] == 0xFE

    # numeric parity on every row whose values stay in fp32 range (the
    # special finite rows included); x codes, scales, routing and the
    # permutation on every row (inside _check_stages)
    ids, tw, _ = O.route(s["logits"], s["bias"], w.k)
    checked = np.array(sorted(set(range(w.T)) - set(overflow)))
    if len(checked) > 64:
        rng = np.random.default_rng(5)
        checked = np.array(sorted(set(special) | set(rng.choice(checked, 48, replace=False).tolist())))
    ref = oracle_forward_pool(w, s, checked, ids, tw)
    _check_stages(w, p, ws, s, ref, checked)
    assert_output_parity(outs[0][torch.from_numpy(checked).cuda()], ref["out"], f"{name} with planted rows")
    # all-zero rows give exactly zero
    zero_rows = torch.tensor(special[1:3], device="cuda")
    assert torch.all(outs[0][zero_rows].float() == 0)
