"""outer_product_associative_chunked_b300: outer-product associative-memory
layers (Tensor Cache, DeltaNet delta rule, BDH-style sparse linear attention)
as hand-written CUDA kernels for sm_103a behind a C-ABI library.
"""
from . import synth  # noqa: F401
