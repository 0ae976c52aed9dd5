"""Seeded synthetic inputs for paged grouped-query decode attention.

This module only produces inputs: query vectors, K/V block pools, block tables
and sequence lengths.  It computes no attention result and holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it.  See ``gen.synth`` for the workload recipes.
"""
from .synth import CONFIGS, Q8, Workload, config_names, make, to_numpy_bits  # noqa: F401
