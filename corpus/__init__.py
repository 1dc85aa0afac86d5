"""Seeded synthetic corpora for the packed-assembly workloads.

This package only draws random inputs (token ids, document lengths, source and
stratum weights).  It holds none of the packing arithmetic, so both the CPU
oracle and the CUDA library can consume what it produces.
"""
from .synthetic import (  # noqa: F401
    Corpus,
    PRESETS,
    make_corpus,
    make_preset,
)
