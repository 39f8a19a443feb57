"""CPU oracle of batch-1 Llama-shaped decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its binding) never does.
"""
from .oracle import OracleDecoder, build_oracle, oracle_lib  # noqa: F401
