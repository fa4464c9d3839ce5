"""Plain CPU oracle of the Kimi-K3 routed-expert MXFP8 x MXFP4 MoE forward.

TEST INFRASTRUCTURE ONLY.  It is slow and obviously correct by design:
float64 numpy, lookup-table decode of every code, explicit power-of-two
scales, a full sort for routing and library matmuls for the contractions.
Only tests, the smoke check and the benchmark's CPU-baseline leg may import
it; the CUDA library and its Python binding share no code with it.
"""
from . import formats, moe  # noqa: F401
