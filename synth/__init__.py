"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package is the only code both sides use.  It turns token sequences into
bf16 Q/K/V values through a prefix hash, draws the token traces of the five
workloads, and plays the part of the language model when a request decodes
(the next token is a hash of the prefix).  It holds none of the radix-tree
rules and none of the attention arithmetic.
"""
from .hashgen import (  # noqa: F401
    GAMMA, KIND_K, KIND_V, KIND_Q, mix64, prefix_hashes, prefix_hashes_from,
    root_hash, gen_values, gen_token, bf16_bits_to_f32,
)
