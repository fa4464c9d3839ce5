"""GPU parity on shapes that reach the less-travelled paths of the forward,
every token against the float64 oracle:

- 224-row token tiles (experts with more than 64 rows) with an odd number
  of 128-wide K blocks (H = 384) or of FC2 weight tiles (H / 128 odd): the
  CTA-pair GEMM does not apply and the one-CTA kernel runs the 224-row tiles;
- a single expert (E = k = 1, every row to it);
- k = 32 (the largest top-k), 64-row tiles;
- E = 37 (no power of two), k = 5;
- a three-token decode batch (32-row tiles);
- the largest expert count and top-k the routing supports (E = 1024,
  k = 32), 32-row tiles.
The stage checks (routing, permutation, codes and scales bit-exact) are those
of test_gpu_forward."""
import numpy as np
import pytest

import workloads as W
from tests._moe_setup import assert_output_parity, oracle_forward, run_forward
from tests.test_gpu_forward import _check_stages

pytestmark = pytest.mark.gpu

BASE = W.WORKLOADS["tiny"]
# name: (workload, small-tile rows, big-tile rows or 0 when no expert can exceed 64 rows)
SHAPES = {
    "odd_kblocks_224": (BASE.with_(name="odd_kblocks_224", T=1024, H=384, I=256, E=8, k=2), 64, 224),
    "one_expert": (BASE.with_(name="one_expert", T=100, H=128, I=128, E=1, k=1), 64, 224),
    "k32": (BASE.with_(name="k32", T=64, H=256, I=128, E=64, k=32), 64, 0),
    "e37_k5": (BASE.with_(name="e37_k5", T=333, H=256, I=256, E=37, k=5), 64, 224),
    "decode3": (BASE.with_(name="decode3", T=3, H=512, I=256, E=64, k=4), 32, 0),
    "max_e_k": (BASE.with_(name="max_e_k", T=64, H=256, I=128, E=1024, k=32), 32, 0),
}


@pytest.fixture(scope="module")
def K():
    import mxfp8_mxfp4_moe_gb300 as K
    assert K.kmoe_check_device(0) == 0
    return K


@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_shape_every_token(K, name):
    w, tile_rows, tile_rows_big = SHAPES[name]
    out, ws, p, s, _ = run_forward(w)
    L = K.kmoe_workspace_layout(p)
    assert (L.tile_rows, L.tile_rows_big) == (tile_rows, tile_rows_big)
    tokens = np.arange(w.T)
    ref = oracle_forward(w, s, tokens)
    _check_stages(w, p, ws, s, ref, tokens)
    assert_output_parity(out, ref["out"], w.name)
