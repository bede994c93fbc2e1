"""CPU oracle of the verify step (TEST INFRASTRUCTURE ONLY).

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import
this package. The product path (the CUDA library and its binding) never does.
"""
from .oracle import Oracle, build, lib  # noqa: F401
