"""Seeded synthetic inputs (weights, caches, states, tokens) for the verify step.

Shared by the CPU oracle and the CUDA path; holds none of the step's arithmetic.
"""
from .synth import (  # noqa: F401
    lib, make_weights, make_pool, fill_pool, make_seq_states, uniform_tokens,
    permutation, normal_f64, raw_draws, q4_matrix, q4_nbytes,
)
from . import configs  # noqa: F401
