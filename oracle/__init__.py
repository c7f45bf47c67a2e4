"""float64 CPU oracle for the outer-product associative-memory layers.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA library; both are fed by the seeded generators in
``outer_product_associative_chunked_b300.synth``.
"""
from . import oracle  # noqa: F401
